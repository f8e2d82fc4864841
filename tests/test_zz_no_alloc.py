"""gdn_chunk_prefill_noalloc, the prefill entry point for callers that cannot
allocate device memory at call time (engines that reserve nearly all device
memory for their own pools, plug-ins inside a framework that owns the
allocator, latency-critical paths that cannot afford cudaMalloc's device-wide
synchronisation).  It takes its scratch from a 64 MiB array built into the
library; this checks it through the C ABI against gdn_chunk_prefill, on two
calls in a row (the second finds the first call's leftovers in the shared
array), and that oversized problems are refused.

This file is collected last so that a stop-at-first-failure run has already
run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, TOL_F32, f64, rel

pytestmark = pytest.mark.gpu

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
        None if h0 is None else h0.data_ptr(), out.data_ptr(), fin.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc


@pytest.mark.parametrize("dtype,d,tol", [(torch.bfloat16, 128, TOL_BF16),
                                         (torch.float32, 64, TOL_F32)])
def test_noalloc_matches_prefill_twice(lib, dtype, d, tol):
    dev = torch.device("cuda")
    runs = [inputs.prefill_inputs([300, 0, 65, 1000], 2, 6, d, d, dtype=dtype, seed=31,
                                  initial_state_std=0.02),
            inputs.prefill_inputs([129, 700], 2, 6, d, d, dtype=dtype, seed=32,
                                  initial_state_std=0.02)]
    for p in runs:  # two calls in a row, different problems
        ref_out, ref_fin = gdn.gdn_chunk_prefill(
            p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev),
            p.cu_seqlens.to(dev), p.initial_state.to(dev), output_final_state=True)
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        assert _call_noalloc(lib, p, dev, out, fin) == 0
        assert rel(f64(out), f64(ref_out)) <= tol
        assert rel(f64(fin), f64(ref_fin)) <= tol


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    # bf16, d=128, 48 value heads needs ~48 KiB of workspace per chunk and
    # value head: 200k tokens need far more than 64 MiB.
    T = 200_000
    prob = gdn.Problem(1, T, 16, 48, 128, 128, gdn.GDN_BF16, None, 0)
    need = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob))
    assert need > gdn.NOALLOC_SCRATCH_BYTES
    fake = 0x10000
    rc = lib.gdn_chunk_prefill_noalloc(ctypes.byref(prob), fake, fake + 4096, fake + 8192,
                                       fake + 12288, fake + 16384, fake + 20480, None,
                                       fake + 24576, None, None)
    assert rc == GDN_ERR_WORKSPACE
