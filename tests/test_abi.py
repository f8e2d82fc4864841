"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA = range(6)
A = 0x10000  # a 16-byte aligned fake device address; never dereferenced here


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return gdn.library()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ["gdn_chunk_prefill", "gdn_decode_step", "gdn_chunk_prefill_workspace_size",
              "gdn_status_string", "gdn_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} not exported"


def test_debug_library_exports_the_same_entry_points(lib):
    dbg = gdn.debug_library()
    assert dbg._name != lib._name
    for name in declared_symbols():
        assert hasattr(dbg, name), f"{name} not exported by the debug build"


def test_status_strings(lib):
    for code in range(8):
        s = gdn.gdn_status_string(code)
        assert s.startswith("GDN_")
    assert "UNKNOWN" in gdn.gdn_status_string(99)
    assert gdn.gdn_version() >= 100


def prob(N=1, T=64, Hk=1, Hv=1, dk=128, dv=128, dtype=gdn.GDN_BF16, ws=None, wsb=0):
    return gdn.Problem(N, T, Hk, Hv, dk, dv, dtype, ws, wsb)


def prefill(lib, p, q=A, k=A + 4096, v=A + 8192, g=A + 12288, b=A + 16384, cu=A + 20480,
            h0=None, out=A + 24576, hT=None):
    return lib.gdn_chunk_prefill(ctypes.byref(p) if p is not None else None, q, k, v, g, b, cu,
                                 h0, out, hT, None)


def decode(lib, p, q=A, k=A + 4096, v=A + 8192, g=A + 12288, b=A + 16384, s=A + 20480,
           out=A + 24576):
    return lib.gdn_decode_step(ctypes.byref(p) if p is not None else None, q, k, v, g, b, s,
                               out, None)


def test_prefill_argument_errors(lib):
    assert prefill(lib, None) == INVALID
    assert prefill(lib, prob(N=-1)) == INVALID
    assert prefill(lib, prob(T=-5)) == INVALID
    assert prefill(lib, prob(Hk=0)) == INVALID
    assert prefill(lib, prob(dk=96, dv=96)) == UNSUPPORTED
    assert prefill(lib, prob(dk=128, dv=64)) == UNSUPPORTED
    assert prefill(lib, prob(Hk=2, Hv=3)) == UNSUPPORTED
    assert prefill(lib, prob(dtype=7)) == UNSUPPORTED
    assert prefill(lib, prob(), cu=None) == INVALID
    assert prefill(lib, prob(), q=None) == INVALID
    assert prefill(lib, prob(), out=None) == INVALID
    assert prefill(lib, prob(), q=A + 2) == MISALIGNED
    assert prefill(lib, prob(), h0=A + 8) == MISALIGNED
    assert prefill(lib, prob(), hT=A + 4) == MISALIGNED
    assert prefill(lib, prob(), cu=A + 2) == MISALIGNED
    assert prefill(lib, prob(), out=A) == INVALID          # aliases q
    assert prefill(lib, prob(N=0, T=5)) == INVALID
    assert prefill(lib, prob(N=0, T=0)) == OK              # nothing to do, no launch


def test_prefill_workspace_checks(lib):
    p = prob(N=2, T=5000, Hk=16, Hv=48)
    need = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(p))
    if need == 0:
        pytest.skip("this configuration needs no workspace")
    assert prefill(lib, p) == WORKSPACE
    small = prob(N=2, T=5000, Hk=16, Hv=48, ws=A, wsb=need - 16)
    assert prefill(lib, small) == WORKSPACE
    mis = prob(N=2, T=5000, Hk=16, Hv=48, ws=A + 8, wsb=need)
    assert prefill(lib, mis) == WORKSPACE


def test_workspace_size_of_invalid_problem_is_zero(lib):
    p = prob(dk=96, dv=96)
    assert lib.gdn_chunk_prefill_workspace_size(ctypes.byref(p)) == 0
    assert lib.gdn_chunk_prefill_workspace_size(None) == 0


def test_decode_argument_errors(lib):
    assert decode(lib, None) == INVALID
    assert decode(lib, prob(N=4, T=5)) == INVALID
    assert decode(lib, prob(N=4, T=4), s=None) == INVALID
    assert decode(lib, prob(N=4, T=4), s=A + 4) == MISALIGNED
    assert decode(lib, prob(N=4, T=4), out=A + 4096) == INVALID   # aliases k
    assert decode(lib, prob(N=4, T=4, dk=32, dv=32)) == UNSUPPORTED
    assert decode(lib, prob(N=0, T=0)) == OK


def half_decode(lib, p, sdt, s=A + 20480, out=A + 24576):
    return lib.gdn_decode_step_half_state(ctypes.byref(p) if p is not None else None, A,
                                          A + 4096, A + 8192, A + 12288, A + 16384, s, sdt,
                                          out, None)


def test_half_state_decode_argument_errors(lib):
    assert half_decode(lib, None, gdn.GDN_F16) == INVALID
    assert half_decode(lib, prob(N=4, T=4), gdn.GDN_F32) == UNSUPPORTED
    assert half_decode(lib, prob(N=4, T=4), 7) == UNSUPPORTED
    assert half_decode(lib, prob(N=4, T=5), gdn.GDN_F16) == INVALID
    assert half_decode(lib, prob(N=4, T=4), gdn.GDN_BF16, s=A + 2) == MISALIGNED
    assert half_decode(lib, prob(N=4, T=4, dtype=gdn.GDN_F16), gdn.GDN_F16) == UNSUPPORTED
    assert half_decode(lib, prob(N=0, T=0), gdn.GDN_F16) == OK


def verify(lib, p, K, sdt=gdn.GDN_F32, state=A + 20480, slots=A + 28672, out=A + 24576):
    return lib.gdn_verify_step(ctypes.byref(p) if p is not None else None, K, A, A + 4096,
                               A + 8192, A + 12288, A + 16384, state, sdt, slots, out, None)


def test_verify_argument_errors(lib):
    assert verify(lib, None, 4) == INVALID
    assert verify(lib, prob(N=4, T=16), 0) == INVALID
    assert verify(lib, prob(N=4, T=36), 9) == INVALID
    assert verify(lib, prob(N=4, T=15), 4) == INVALID          # T != N * K
    assert verify(lib, prob(N=4, T=16), 4, sdt=9) == UNSUPPORTED
    assert verify(lib, prob(N=4, T=16), 4, slots=A + 20480) == INVALID   # slots alias state
    assert verify(lib, prob(N=4, T=16), 4, slots=A + 8) == MISALIGNED
    assert verify(lib, prob(N=4, T=16), 4, out=A) == INVALID   # out aliases q
    assert verify(lib, prob(N=0, T=0), 4) == OK


def test_snapshot_entry_points(lib):
    p = prob(N=2, T=130, Hk=1, Hv=3, ws=A, wsb=1 << 40)
    slots = lib.gdn_chunk_prefill_snapshot_slots
    assert slots(ctypes.byref(p), 1) == (3 + 2) + 2
    assert slots(ctypes.byref(p), 2) == 3 + 2
    assert slots(ctypes.byref(p), 0) == 0
    assert slots(ctypes.byref(prob(dtype=gdn.GDN_F32)), 1) == 0
    assert slots(ctypes.byref(prob(dk=64, dv=64)), 1) == 0

    def snap(p, snaps, s=1):
        return lib.gdn_chunk_prefill_snapshots(ctypes.byref(p), A, A + 4096, A + 8192,
                                               A + 12288, A + 16384, A + 20480, None,
                                               A + 24576, None, snaps, s, None)
    assert snap(p, None) == INVALID
    assert snap(p, A + 32768, s=0) == INVALID
    assert snap(p, A + 8) == MISALIGNED
    assert snap(prob(N=1, T=64, dtype=gdn.GDN_F32), A + 32768) == UNSUPPORTED
    assert snap(prob(N=1, T=64, dk=64, dv=64), A + 32768) == UNSUPPORTED


def test_binding_rejects_cpu_tensors(lib):
    x = torch.zeros(4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdn.gdn_decode_step(x, x, x, torch.zeros(4, 1), torch.zeros(4, 1),
                            torch.zeros(4, 1, 128, 128))


def test_timed_prefill_argument_errors(lib):
    """Checks that need no device: the events array and each event must be
    given, and only the tensor-core configuration is timed."""
    timed = lib.gdn_chunk_prefill_timed

    def call(p, events):
        return timed(ctypes.byref(p), A, A + 4096, A + 8192, A + 12288, A + 16384, A + 20480,
                     None, A + 24576, None, events, None, None)
    p = prob(N=1, T=64)
    assert call(p, None) == INVALID
    missing = (ctypes.c_void_p * 4)(A, A, None, A)
    assert call(p, ctypes.cast(missing, ctypes.c_void_p)) == INVALID
    fake = (ctypes.c_void_p * 4)(A, A, A, A)
    assert call(prob(N=1, T=64, dtype=gdn.GDN_F32), ctypes.cast(fake, ctypes.c_void_p)) == \
        UNSUPPORTED
    assert call(prob(N=1, T=64, dk=64, dv=64), ctypes.cast(fake, ctypes.c_void_p)) == \
        UNSUPPORTED


def test_fused_mode_needs_no_device(lib):
    """The mode switch is a plain atomic: set, query, restore."""
    old = lib.gdn_prefill_fused_mode(-1)
    assert old in (0, 1, 2, 3)
    assert lib.gdn_prefill_fused_mode(0) == old
    assert lib.gdn_prefill_fused_mode(3) == 0
    assert lib.gdn_prefill_fused_mode(9) == 3
    assert lib.gdn_prefill_fused_mode(4) == 3
    assert lib.gdn_prefill_fused_mode(old) == 3


def scan(lib, p, L, out=A + 24576):
    return lib.gdn_chunk_prefill_scan(ctypes.byref(p) if p is not None else None, L, A, A + 4096,
                                      A + 8192, A + 12288, A + 16384, A + 20480, None, out,
                                      None, None)


def test_scan_argument_errors(lib):
    """Checks that need no device: sizes, unsupported shapes, bad group
    sizes, missing workspace."""
    p = prob(N=2, T=5000, Hk=16, Hv=48)
    size = lib.gdn_chunk_prefill_scan_workspace_size
    assert size(ctypes.byref(p), 8) > lib.gdn_chunk_prefill_workspace_size(ctypes.byref(p))
    assert size(ctypes.byref(p), 0) > 0
    assert size(ctypes.byref(p), -1) == 0
    assert size(ctypes.byref(prob(dk=64, dv=64)), 4) == 0
    assert size(None, 4) == 0
    assert scan(lib, None, 4) == INVALID
    assert scan(lib, p, -1) == INVALID
    assert scan(lib, prob(dk=64, dv=64), 4) == UNSUPPORTED
    assert scan(lib, p, 4) == WORKSPACE
    assert scan(lib, prob(N=2, T=5000, Hk=16, Hv=48, ws=A, wsb=size(ctypes.byref(p), 4) - 16),
                4) == WORKSPACE
    assert scan(lib, prob(N=0, T=0), 4) == OK


def test_host_pipeline_argument_errors(lib):
    def call(p, pieces):
        # problem, pieces, 6 host tensors, no initial/final state, 6 device
        # staging buffers, cu, state, default stream; every case below is
        # refused before anything is enqueued
        return lib.gdn_chunk_prefill_host(ctypes.byref(p) if p is not None else None, pieces,
                                          *([A] * 6), None, None, *([A] * 8), None)
    assert call(None, 4) == INVALID
    assert call(prob(N=2, T=128), 4) == INVALID     # one sequence only
    assert call(prob(N=1, T=128), 0) == INVALID
    assert call(prob(N=1, T=128), 65) == INVALID
    assert call(prob(N=1, T=128, dtype=gdn.GDN_F16), 2) == UNSUPPORTED
    # the whole sequence's workspace is checked before anything is enqueued
    need = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob(N=1, T=128)))
    assert need > 0
    assert call(prob(N=1, T=128), 2) == WORKSPACE
    assert call(prob(N=1, T=128, ws=A, wsb=need - 1), 2) == WORKSPACE


def test_binding_rejects_tensors_on_another_device():
    """Every tensor of a call must be on q's device: the check runs before
    any pointer reaches the library (shown here with meta and CPU tensors,
    which need no GPU)."""
    q = torch.empty(2, 1, 128, device="meta")
    with pytest.raises(ValueError, match="one device"):
        gdn._same_device(torch.device("cuda", 0), k=q)
    with pytest.raises(ValueError, match="one device"):
        gdn._same_device(torch.device("cuda", 1), v=torch.empty(1))
    gdn._same_device(torch.device("cpu"), k=torch.empty(1), out=None)
