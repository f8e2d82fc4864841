"""Decode parity: consecutive recurrent steps through the C ABI against the
fp64 oracle, checked at every step."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
import oracle
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, TOL_F32, f64, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def run_steps(N, Hk, Hv, d, steps, dtype, tol, state_sample=None, full_state_at=()):
    dev = torch.device("cuda")
    S0 = inputs.decode_state(N, Hv, d, d)
    S_dev = S0.to(dev)
    S_ref = f64(S0)
    worst = 0.0
    for s in range(steps):
        x = inputs.decode_step_inputs(s, N, Hk, Hv, d, d, dtype=dtype)
        o = gdn.gdn_decode_step(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.g.to(dev),
                                x.beta.to(dev), S_dev)
        o_ref, _ = oracle.decode(f64(x.q), f64(x.k), f64(x.v), f64(x.g), f64(x.beta), S_ref,
                                 inplace=True)
        torch.cuda.synchronize()
        e = rel(f64(o), o_ref)
        assert e <= tol, f"step {s}: out rel err {e:.3e}"
        if state_sample is not None:
            e2 = rel(f64(S_dev[state_sample]), S_ref[state_sample])
            assert e2 <= tol, f"step {s}: sampled state rel err {e2:.3e}"
        if s in full_state_at or s == steps - 1:
            e3 = rel(f64(S_dev), S_ref)
            assert e3 <= tol, f"step {s}: state rel err {e3:.3e}"
        worst = max(worst, e)
    return worst


@pytest.mark.parametrize("d", [64, 128])
def test_decode_small_fp32(d):
    run_steps(5, 2, 6, d, 12, torch.float32, TOL_F32, state_sample=slice(None))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_small_bf16(d):
    run_steps(3, 1, 3, d, 20, torch.bfloat16, TOL_BF16, state_sample=slice(None))


def test_decode_batch64_48_heads_256_steps():
    """64 sequences x 1 token, 16 key / 48 value heads, d=128, fp32 state
    ~N(0, 0.02^2), bf16 q/k/v, 256 consecutive steps, every step checked
    (all outputs; the state of sequences 0, 17, 63 every step; the whole state
    at steps 0, 127, 255)."""
    run_steps(64, 16, 48, 128, 256, torch.bfloat16, TOL_BF16,
              state_sample=[0, 17, 63], full_state_at=(0, 127))


def test_decode_steps_equal_prefill():
    """T decode steps from S0 match a T-token prefill from S0 (fp32 path)."""
    dev = torch.device("cuda")
    T, Hk, Hv, d = 40, 1, 3, 64
    p = inputs.prefill_inputs([T], Hk, Hv, d, d, dtype=torch.float32, seed=9,
                              initial_state_std=0.02)
    out, fin = gdn.gdn_chunk_prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev),
                                     p.beta.to(dev), p.cu_seqlens.to(dev),
                                     p.initial_state.to(dev), output_final_state=True)
    S = p.initial_state.to(dev).clone()
    outs = []
    for t in range(T):
        sl = slice(t, t + 1)
        outs.append(gdn.gdn_decode_step(p.q[sl].to(dev), p.k[sl].to(dev), p.v[sl].to(dev),
                                        p.g[sl].to(dev), p.beta[sl].to(dev), S))
    torch.cuda.synchronize()
    assert rel(f64(torch.cat(outs)), f64(out)) <= TOL_F32
    assert rel(f64(S), f64(fin)) <= TOL_F32
