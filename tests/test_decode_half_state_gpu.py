"""Decode with the state stored in 16 bits (fp16, the pages' choice, or bf16):
each step against the fp64 oracle fed the same stored state (the GPU step
computes in fp32 and rounds the new state to nearest even; the oracle's new
state is rounded the same way), plus the drift of a 16-bit trajectory from
the fp64 one, reported."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
import oracle
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, f64, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def step_parity(N, Hk, Hv, d, steps, sdt, heads=None):
    dev = torch.device("cuda")
    S = inputs.decode_state(N, Hv, d, d).to(sdt).to(dev)
    hs = list(range(Hv)) if heads is None else heads
    worst_o = worst_s = 0.0
    worst_flip = 0.0
    for s in range(steps):
        x = inputs.decode_step_inputs(s, N, Hk, Hv, d, d, dtype=torch.bfloat16)
        s_in = f64(S)
        o = gdn.gdn_decode_step_half_state(x.q.to(dev), x.k.to(dev), x.v.to(dev),
                                           x.g.to(dev), x.beta.to(dev), S)
        torch.cuda.synchronize()
        o_ref, s_ref = oracle.decode(f64(x.q), f64(x.k), f64(x.v), f64(x.g), f64(x.beta), s_in,
                                     heads=hs)
        o_gpu = f64(o)[:, hs]
        e_o = rel(o_gpu, o_ref[:, hs])
        # The oracle's new state, rounded to the storage type like the kernel's.
        s_ref_r = torch.from_numpy(s_ref[:, hs]).to(sdt)
        s_gpu = S[:, hs].cpu()
        e_s = rel(f64(s_gpu), f64(s_ref_r))
        flip = float((s_gpu != s_ref_r).float().mean())
        assert e_o <= TOL_BF16, f"step {s}: out rel err {e_o:.3e}"
        assert e_s <= TOL_BF16, f"step {s}: state rel err {e_s:.3e}"
        assert flip <= 0.01, f"step {s}: {flip:.2%} of state elements round differently"
        worst_o, worst_s, worst_flip = max(worst_o, e_o), max(worst_s, e_s), max(worst_flip, flip)
    print(f"[parity] half-state decode {sdt} N={N} Hv={Hv} d={d} steps={steps}: out {worst_o:.3e} "
          f"state {worst_s:.3e} rounding flips {worst_flip:.2e}")


@pytest.mark.parametrize("sdt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
def test_half_state_steps_small(sdt, d):
    step_parity(3, 2, 6, d, 6, sdt)


@pytest.mark.parametrize("sdt", [torch.float16, torch.bfloat16])
def test_half_state_decode_workload_sampled(sdt):
    """64 sequences x 16/48 heads, d = 128: every step of 4 checked on 6 heads."""
    step_parity(64, 16, 48, 128, 4, sdt, heads=[0, 1, 2, 23, 40, 47])


@pytest.mark.parametrize("sdt", [torch.float16, torch.bfloat16])
def test_half_state_trajectory_drift(sdt):
    """64 steps kept in 16 bits against the fp64 trajectory (reported; the
    per-step parity above is the bar)."""
    dev = torch.device("cuda")
    N, Hk, Hv, d = 4, 2, 6, 128
    S0 = inputs.decode_state(N, Hv, d, d)
    S = S0.to(sdt).to(dev)
    S_ref = f64(S0.to(sdt))
    errs = []
    for s in range(64):
        x = inputs.decode_step_inputs(s, N, Hk, Hv, d, d, dtype=torch.bfloat16)
        o = gdn.gdn_decode_step_half_state(x.q.to(dev), x.k.to(dev), x.v.to(dev),
                                           x.g.to(dev), x.beta.to(dev), S)
        o_ref, _ = oracle.decode(f64(x.q), f64(x.k), f64(x.v), f64(x.g), f64(x.beta), S_ref,
                                 inplace=True)
        torch.cuda.synchronize()
        errs.append(rel(f64(o), o_ref))
    e_state = rel(f64(S), S_ref)
    print(f"[drift] {sdt} 64 steps: out max {max(errs):.3e} last {errs[-1]:.3e}, "
          f"state {e_state:.3e}")
    assert np.isfinite(errs).all() and np.isfinite(e_state)


def test_half_state_rejects_other_dtypes():
    dev = torch.device("cuda")
    x = inputs.decode_step_inputs(0, 2, 1, 3, 64, 64, dtype=torch.bfloat16)
    S = torch.zeros((2, 3, 64, 64), dtype=torch.float32, device=dev)
    with pytest.raises(TypeError):
        gdn.gdn_decode_step_half_state(x.q.to(dev), x.k.to(dev), x.v.to(dev), x.g.to(dev),
                                       x.beta.to(dev), S)
