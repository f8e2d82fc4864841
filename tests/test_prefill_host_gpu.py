"""gdn_chunk_prefill_host: one sequence from pinned host memory in pieces,
transfers overlapped with the computation.  Against the fp64 oracle, and
against the device-resident prefill: bit for bit with one piece; with more,
the pieces restart the state's running scale at their boundaries, which
changes the bf16 rounding of the state operand, so the two agree to the bf16
tolerance."""
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, f64, oracle_prefill, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("pieces", [1, 3, 4, 64])
@pytest.mark.parametrize("T,Hk,Hv,h0", [(1000, 2, 6, True), (4000, 16, 48, False), (97, 1, 3, True)])
def test_host_pipeline(pieces, T, Hk, Hv, h0):
    p = inputs.prefill_inputs([T], Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=31,
                              initial_state_std=0.02 if h0 else None)
    hq, hk, hv, hg, hb = (x.pin_memory() for x in (p.q, p.k, p.v, p.g, p.beta))
    hout = torch.full((T, Hv, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    dev = torch.device("cuda")
    h0_d = p.initial_state.to(dev) if h0 else None
    fin = torch.empty((1, Hv, 128, 128), device=dev)
    gdn.gdn_chunk_prefill_host(hq, hk, hv, hg, hb, hout, h0_d, fin, pieces=pieces)
    torch.cuda.synchronize()
    o_dev, f_dev = gdn.gdn_chunk_prefill(*[x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta,
                                                                  p.cu_seqlens)],
                                         h0_d, output_final_state=True)
    torch.cuda.synchronize()
    key_heads = None if Hk <= 2 else [0, Hk - 1]
    o_ref, f_ref, vh = oracle_prefill(p, key_heads)
    e_o, e_f = rel(f64(hout[:, vh]), o_ref), rel(f64(fin[:, vh]), f_ref)
    d_o, d_f = rel(f64(hout), f64(o_dev)), rel(f64(fin), f64(f_dev))
    print(f"[parity] host pieces={pieces} T={T}: out {e_o:.3e} final {e_f:.3e}; "
          f"vs device out {d_o:.1e} final {d_f:.1e}")
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16
    if pieces == 1:
        # One piece is the device call itself.
        assert torch.equal(hout, o_dev.cpu()) and torch.equal(fin, f_dev)
    else:
        # A piece starts its state's running scale at 1, so the bf16 operand of
        # the state products rounds S instead of S / sigma from there on: two
        # equally valid roundings, a few 2^-9 apart.
        assert d_o <= TOL_BF16 and d_f <= TOL_BF16


@pytest.mark.parametrize("h0", [True, False])
def test_host_pipeline_empty_sequence(h0):
    """T = 0: nothing is copied or computed; the final state is the initial
    state (or zero) and out stays empty."""
    p = inputs.prefill_inputs([0], 2, 6, 128, 128, dtype=torch.bfloat16, seed=33,
                              initial_state_std=0.02 if h0 else None)
    dev = torch.device("cuda")
    out = torch.empty((0, 6, 128), dtype=torch.bfloat16)
    h0_d = p.initial_state.to(dev) if h0 else None
    fin = torch.full((1, 6, 128, 128), 7.0, device=dev)
    gdn.gdn_chunk_prefill_host(p.q, p.k, p.v, p.g, p.beta, out, h0_d, fin, pieces=4)
    torch.cuda.synchronize()
    if h0:
        assert torch.equal(fin, h0_d)
    else:
        assert torch.count_nonzero(fin) == 0


def test_device_prefill_all_sequences_empty_bf16():
    """The tensor-core path with every sequence empty (T = 0, N = 2): the
    final states are the initial states, bit for bit."""
    p = inputs.prefill_inputs([0, 0], 2, 6, 128, 128, dtype=torch.bfloat16, seed=34,
                              initial_state_std=0.02)
    dev = torch.device("cuda")
    out, fin = gdn.gdn_chunk_prefill(*[x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta,
                                                            p.cu_seqlens, p.initial_state)],
                                     output_final_state=True)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(fin.cpu(), p.initial_state)
