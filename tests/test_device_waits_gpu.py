"""Failure detection on the device without a GPU fault.

The library's kernels bound every wait: after a time limit a wait gives up,
raises the kernel's abort flag (so that every role of the CTA leaves) and the
kernel records a time-out in its error word.  A probe kernel runs the same wait
helpers on an mbarrier that nothing ever arrives at, with a short limit, and
the host checks what they report and that the context stays usable.  The
prefill's device-side status query is checked on malformed cu_seqlens (which
the kernels detect and turn into a no-op)."""
import ctypes
import os
import subprocess

import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, check_prefill

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.join(os.path.dirname(HERE), "gated_deltanet_linear_chunk_gb300")
LIMIT = 2_000_000  # cycles (about 1 ms)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("wprobe") / "libwait_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(PKG, "csrc"),
                    "-I", os.path.join(os.path.dirname(HERE), "include"),
                    os.path.join(HERE, "csrc", "wait_probe.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.wait_probe_run.restype = ctypes.c_int
    lib.wait_probe_run.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p]
    return lib


def run(probe, mode, limit=LIMIT):
    out = torch.full((9,), -1, dtype=torch.int32, device="cuda")  # (out[8]: the ready flag)
    assert probe.wait_probe_run(mode, limit, out.data_ptr()) == 0
    o = out.cpu().tolist()
    return [dict(ok=o[4 * w], abort=o[4 * w + 1], kcycles=o[4 * w + 2]) for w in range(2)]


@pytest.mark.parametrize("mode", [1, 3])
def test_bounded_wait_gives_up_and_raises_abort(probe, mode):
    """The ready-flag wait (1) and the all-lane mbarrier wait (3)."""
    for w in run(probe, mode):
        assert w["ok"] == 0 and w["abort"] == 1
        assert w["kcycles"] * 1024 >= LIMIT - 1024


def test_polling_wait_gives_up(probe):
    """The prep units' polling wait reports the time-out to its caller (which
    raises the error itself) and leaves the abort flag alone."""
    for w in run(probe, 0):
        assert w["ok"] == 0 and w["abort"] == 0
        assert w["kcycles"] * 1024 >= LIMIT - 1024


@pytest.mark.parametrize("mode", [2, 4])
def test_abort_releases_the_other_waiters(probe, mode):
    """Warp 0 times out; warp 1, whose own limit is 100 times longer, leaves
    on the abort flag well before its limit."""
    w0, w1 = run(probe, mode)
    assert w0["ok"] == 0 and w1["ok"] == 0 and w1["abort"] == 1
    assert w1["kcycles"] * 1024 < 10 * LIMIT


def test_context_usable_after_time_outs(probe):
    run(probe, 3)
    p = inputs.prefill_inputs([100], 1, 3, 128, 128, dtype=torch.bfloat16, seed=11)
    check_prefill(p, TOL_BF16)
    assert gdn.gdn_chunk_prefill_device_status() == gdn.GDN_OK


@pytest.mark.parametrize("bad", [[0, 100, 149], [1, 100, 150], [0, 120, 100, 150]])
def test_prefill_device_status_reports_malformed_cu_seqlens(bad):
    """cu_seqlens not ending at T, not starting at 0, or decreasing: the call
    writes nothing and the status query reports GDN_ERR_INVALID_ARG; the next
    good call reports GDN_OK."""
    N = len(bad) - 1
    p = inputs.prefill_inputs([150 // N] * (N - 1) + [150 - (150 // N) * (N - 1)], 1, 3, 128,
                              128, dtype=torch.bfloat16, seed=12, initial_state_std=0.02)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta)]
    h0 = p.initial_state.to(dev)
    out = torch.full((150, 3, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    fin = torch.full_like(h0, 7.0)
    cu = torch.tensor(bad, dtype=torch.int32, device=dev)
    gdn.gdn_chunk_prefill(*a, cu, h0, out=out, final_state=fin)
    assert gdn.gdn_chunk_prefill_device_status() == gdn.GDN_ERR_INVALID_ARG
    assert torch.isnan(out.float()).all()
    assert (fin == 7.0).all()
    gdn.gdn_chunk_prefill(*a, p.cu_seqlens.to(dev), h0, out=out, final_state=fin)
    assert gdn.gdn_chunk_prefill_device_status() == gdn.GDN_OK
    assert not torch.isnan(out.float()).any()


def test_noalloc_device_status():
    p = inputs.prefill_inputs([80, 40], 1, 3, 128, 128, dtype=torch.bfloat16, seed=13)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta)]
    out = torch.empty((120, 3, 128), dtype=torch.bfloat16, device=dev)
    gdn.gdn_chunk_prefill_noalloc(*a, torch.tensor([0, 80, 119], dtype=torch.int32, device=dev),
                                  out=out)
    assert gdn.gdn_chunk_prefill_device_status(noalloc=True) == gdn.GDN_ERR_INVALID_ARG
    gdn.gdn_chunk_prefill_noalloc(*a, p.cu_seqlens.to(dev), out=out)
    assert gdn.gdn_chunk_prefill_device_status(noalloc=True) == gdn.GDN_OK
