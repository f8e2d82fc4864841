"""Verify step of speculative decoding (K tokens per sequence from one stored
state, every position's output, the state after every position in its own
slot) against the fp64 oracle applied token by token, and against K
successive decode steps."""
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


def verify_inputs(N, K, Hk, Hv, d, seed_step=0):
    """K consecutive decode-step inputs stacked per sequence: [N, K, ...]."""
    xs = [inputs.decode_step_inputs(seed_step + j, N, Hk, Hv, d, d, dtype=torch.bfloat16)
          for j in range(K)]
    return [torch.stack([getattr(x, f) for x in xs], dim=1).contiguous()
            for f in ("q", "k", "v", "g", "beta")]


def oracle_chain(q, k, v, g, b, S0):
    """fp64 outputs and states after each of the K tokens."""
    K = q.shape[1]
    S = f64(S0).copy()
    outs, states = [], []
    for j in range(K):
        o, S = oracle.decode(f64(q[:, j]), f64(k[:, j]), f64(v[:, j]), f64(g[:, j]),
                             f64(b[:, j]), S)
        outs.append(o)
        states.append(S.copy())
    return np.stack(outs, axis=1), np.stack(states, axis=1)


@pytest.mark.parametrize("K", [1, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_verify_fp32_state_against_oracle(K, d):
    N, Hk, Hv = 5, 2, 6
    dev = torch.device("cuda")
    q, k, v, g, b = verify_inputs(N, K, Hk, Hv, d)
    S0 = inputs.decode_state(N, Hv, d, d)
    out, slots = gdn.gdn_verify_step(*[x.to(dev) for x in (q, k, v, g, b)], S0.to(dev))
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_chain(q, k, v, g, b, S0)
    e_o, e_s = rel(f64(out), o_ref), rel(f64(slots), s_ref)
    print(f"[parity] verify fp32 state K={K} d={d}: out {e_o:.3e} slots {e_s:.3e}")
    assert e_o <= TOL_BF16 and e_s <= TOL_BF16


def test_verify_equals_successive_decode_steps():
    """With an fp32 state, slot t and output t are bit for bit what t + 1
    successive decode steps give."""
    N, K, Hk, Hv, d = 64, 8, 16, 48, 128
    dev = torch.device("cuda")
    q, k, v, g, b = [x.to(dev) for x in verify_inputs(N, K, Hk, Hv, d)]
    S0 = inputs.decode_state(N, Hv, d, d).to(dev)
    out, slots = gdn.gdn_verify_step(q, k, v, g, b, S0)
    S = S0.clone()
    for j in range(K):
        o = gdn.gdn_decode_step(q[:, j].contiguous(), k[:, j].contiguous(), v[:, j].contiguous(),
                                g[:, j].contiguous(), b[:, j].contiguous(), S)
        torch.cuda.synchronize()
        assert torch.equal(o, out[:, j]), f"output of token {j}"
        assert torch.equal(S, slots[:, j]), f"slot {j}"
    assert torch.equal(S0, inputs.decode_state(N, Hv, d, d).to(dev)), "state must be read only"


@pytest.mark.parametrize("sdt", [torch.float16, torch.bfloat16])
def test_verify_half_state_against_oracle(sdt):
    """16-bit state and slots: the tokens chain in fp32; each slot is the
    oracle's state after that token (from the same stored start state),
    rounded like the kernel's."""
    N, K, Hk, Hv, d = 8, 8, 2, 6, 128
    dev = torch.device("cuda")
    q, k, v, g, b = verify_inputs(N, K, Hk, Hv, d, seed_step=3)
    S0 = inputs.decode_state(N, Hv, d, d).to(sdt)
    out, slots = gdn.gdn_verify_step(*[x.to(dev) for x in (q, k, v, g, b)], S0.to(dev))
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_chain(q, k, v, g, b, S0)
    s_ref_r = torch.from_numpy(s_ref).to(sdt)
    e_o = rel(f64(out), o_ref)
    e_s = rel(f64(slots.cpu()), f64(s_ref_r))
    flips = float((slots.cpu() != s_ref_r).float().mean())
    print(f"[parity] verify {sdt} K={K}: out {e_o:.3e} slots {e_s:.3e} rounding flips {flips:.2e}")
    assert e_o <= TOL_BF16 and e_s <= TOL_BF16 and flips <= 0.01


def test_verify_rejects_bad_shapes():
    dev = torch.device("cuda")
    q, k, v, g, b = [x.to(dev) for x in verify_inputs(2, 9, 1, 3, 64)]
    S0 = inputs.decode_state(2, 3, 64, 64).to(dev)
    with pytest.raises(gdn.GDNError):
        gdn.gdn_verify_step(q, k, v, g, b, S0)  # K = 9 > 8
