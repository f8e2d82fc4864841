"""gdn_chunk_prefill_noalloc, the prefill entry point for callers that cannot
allocate device memory at call time (engines that reserve nearly all device
memory for their own pools, plug-ins inside a framework that owns the
allocator, latency-critical paths that cannot afford cudaMalloc's device-wide
synchronisation).  It takes its scratch from a 64 MiB array built into the
library.  These tests call it through the C ABI and compare it with
gdn_chunk_prefill on two calls in a row (the second finds the first call's
leftovers in the shared array).  The two entry points run the same kernels
on the same problem, so the results must be equal bit for bit.  The tests
also check the size limit on both sides of it, and a malformed cu_seqlens
through the Python wrapper.

This file is collected last so that a stop-at-first-failure run has already
run every other test before it."""
import ctypes

import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

GDN_ERR_INVALID_ARG = 1
GDN_ERR_WORKSPACE = 4


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return gdn.library()


def _call_noalloc(lib, p, dev, out, fin):
    T, Hk, dk = p.q.shape
    Hv, dv = p.v.shape[1:]
    N = p.cu_seqlens.shape[0] - 1
    dt = gdn.GDN_BF16 if p.q.dtype == torch.bfloat16 else gdn.GDN_F32
    # The descriptor's workspace fields are deliberately left empty.
    prob = gdn.Problem(N, T, Hk, Hv, dk, dv, dt, None, 0)
    args = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    h0 = None if p.initial_state is None else p.initial_state.to(dev)
    rc = lib.gdn_chunk_prefill_noalloc(
        ctypes.byref(prob), *[a.data_ptr() for a in args],
        None if h0 is None else h0.data_ptr(), out.data_ptr(),
        None if fin is None else fin.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc


def _check_equal(lib, p, dev):
    ref_out, ref_fin = gdn.gdn_chunk_prefill(
        p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev),
        p.cu_seqlens.to(dev), None if p.initial_state is None else p.initial_state.to(dev),
        output_final_state=True)
    out = torch.full_like(ref_out, float("nan"))
    fin = torch.full_like(ref_fin, float("nan"))
    assert _call_noalloc(lib, p, dev, out, fin) == 0
    assert torch.equal(out, ref_out), "output differs from gdn_chunk_prefill"
    assert torch.equal(fin, ref_fin), "final state differs from gdn_chunk_prefill"


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_noalloc_matches_prefill_twice(lib, dtype, d):
    dev = torch.device("cuda")
    runs = [inputs.prefill_inputs([300, 0, 65, 1000], 2, 6, d, d, dtype=dtype, seed=31,
                                  initial_state_std=0.02),
            inputs.prefill_inputs([129, 700], 2, 6, d, d, dtype=dtype, seed=32,
                                  initial_state_std=0.02)]
    for p in runs:  # two calls in a row, different problems
        _check_equal(lib, p, dev)


def _largest_fitting_tokens(lib, Hk, Hv):
    """Largest T of one bf16, d = 128 sequence whose workspace fits the
    built-in scratch (the size query decides, so this follows the layout)."""
    def need(T):
        prob = gdn.Problem(1, T, Hk, Hv, 128, 128, gdn.GDN_BF16, None, 0)
        return lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob))
    lo, hi = 1, 1 << 22
    assert need(lo) <= gdn.NOALLOC_SCRATCH_BYTES < need(hi)
    while lo + 1 < hi:
        mid = (lo + hi) // 2
        if need(mid) <= gdn.NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_at_its_size_limit(lib):
    """16 key / 48 value heads: the largest one-sequence problem that fits
    matches gdn_chunk_prefill, one token more is refused before any launch."""
    dev = torch.device("cuda")
    T = _largest_fitting_tokens(lib, 16, 48)
    p = inputs.prefill_inputs([T], 16, 48, 128, 128, dtype=torch.bfloat16, seed=33,
                              initial_state_std=0.02)
    _check_equal(lib, p, dev)
    prob = gdn.Problem(1, T + 1, 16, 48, 128, 128, gdn.GDN_BF16, None, 0)
    fake = 0x10000  # never dereferenced: the call must fail on the host
    rc = lib.gdn_chunk_prefill_noalloc(ctypes.byref(prob), fake, fake + 4096, fake + 8192,
                                       fake + 12288, fake + 16384, fake + 20480, None,
                                       fake + 24576, None, None)
    assert rc == GDN_ERR_WORKSPACE


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    T = 200_000
    prob = gdn.Problem(1, T, 16, 48, 128, 128, gdn.GDN_BF16, None, 0)
    assert lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob)) > gdn.NOALLOC_SCRATCH_BYTES
    fake = 0x10000
    rc = lib.gdn_chunk_prefill_noalloc(ctypes.byref(prob), fake, fake + 4096, fake + 8192,
                                       fake + 12288, fake + 16384, fake + 20480, None,
                                       fake + 24576, None, None)
    assert rc == GDN_ERR_WORKSPACE


def test_noalloc_wrapper_reports_malformed_cu_seqlens(lib):
    """Through the Python wrapper: a decreasing cu_seqlens is caught on the
    device, the call writes nothing, and the built-in scratch's status word
    says so; the next good call clears it."""
    dev = torch.device("cuda")
    p = inputs.prefill_inputs([100, 28], 2, 6, 128, 128, dtype=torch.bfloat16, seed=34)
    args = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta)]
    out = torch.full((128, 6, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    bad = torch.tensor([0, 100, 50], dtype=torch.int32, device=dev)
    gdn.gdn_chunk_prefill_noalloc(*args, bad, out=out)
    assert gdn.gdn_chunk_prefill_device_status(noalloc=True) == GDN_ERR_INVALID_ARG
    assert torch.isnan(out.float()).all(), "a rejected call wrote output"
    good = p.cu_seqlens.to(dev)
    gdn.gdn_chunk_prefill_noalloc(*args, good, out=out)
    assert gdn.gdn_chunk_prefill_device_status(noalloc=True) == 0
    ref, _ = gdn.gdn_chunk_prefill(*args, good)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
