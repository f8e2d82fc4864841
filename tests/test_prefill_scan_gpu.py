"""Chunk-parallel scan of the prefill recurrence (gdn_chunk_prefill_scan)
against the fp64 oracle, and against the sequential recurrence of
gdn_chunk_prefill on the same inputs."""
import numpy as np
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


def run_scan(p, L, final=True):
    dev = torch.device("cuda")
    out, fin = gdn.gdn_chunk_prefill_scan(
        p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev),
        p.cu_seqlens.to(dev), None if p.initial_state is None else p.initial_state.to(dev),
        output_final_state=final, chunks_per_group=L)
    torch.cuda.synchronize()
    return out, fin


def check_scan(p, L, key_heads=None, tol=TOL_BF16):
    out, fin = run_scan(p, L)
    o_ref, f_ref, vh = oracle_prefill(p, key_heads)
    e_out = rel(f64(out[:, vh]), o_ref)
    e_fin = rel(f64(fin[:, vh]), f_ref)
    assert np.isfinite(f64(out)).all() and np.isfinite(f64(fin)).all()
    print(f"[parity] scan L={L} T={p.q.shape[0]} N={p.cu_seqlens.shape[0] - 1}: "
          f"out {e_out:.3e} final {e_fin:.3e}")
    assert e_out <= tol and e_fin <= tol
    return out, fin


@pytest.mark.parametrize("L", [1, 2, 3, 0])
def test_scan_small_varlen_ragged(L):
    """Ragged tails, an empty and a one-token sequence, a sequence of exactly
    one chunk, GQA 1:3, nonzero initial states; groups of 1, 2, 3 chunks and
    the automatic choice."""
    p = inputs.prefill_inputs([130, 1, 64, 0, 77, 400], 2, 6, 128, 128, dtype=torch.bfloat16,
                              seed=1, initial_state_std=0.02)
    check_scan(p, L)


def test_scan_zero_start_one_sequence():
    """No initial state, T=1000 (16 chunks) in groups of 5, one key head."""
    p = inputs.prefill_inputs([1000], 1, 3, 128, 128, dtype=torch.bfloat16, seed=2)
    check_scan(p, 5)


def test_scan_matches_sequential_recurrence():
    """Same inputs through both paths: the scan reorders the rounding of the
    state chain only, so the two agree far inside the oracle tolerance."""
    p = inputs.prefill_inputs([700, 300, 2100], 2, 6, 128, 128, dtype=torch.bfloat16, seed=3,
                              initial_state_std=0.02)
    dev = torch.device("cuda")
    args = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    h0 = p.initial_state.to(dev)
    o1, f1 = gdn.gdn_chunk_prefill(*args, h0, output_final_state=True)
    o2, f2 = gdn.gdn_chunk_prefill_scan(*args, h0, output_final_state=True, chunks_per_group=4)
    torch.cuda.synchronize()
    e_o, e_f = rel(f64(o2), f64(o1)), rel(f64(f2), f64(f1))
    print(f"[scan vs sequential] out {e_o:.3e} final {e_f:.3e}")
    assert e_o <= 5e-3 and e_f <= 5e-3


def test_scan_t20480_few_heads():
    """The case the scan is for: one long sequence (320 chunks), 4 key / 12
    value heads, nonzero initial state; all heads checked."""
    p = inputs.prefill_inputs([20480], 4, 12, 128, 128, dtype=torch.bfloat16, seed=4,
                              initial_state_std=0.02)
    check_scan(p, 0)


def test_scan_t4000_48_heads_sampled():
    """The 4000-token, 16/48-head workload in groups of 21 chunks: three
    key-head groups checked against the oracle."""
    p = inputs.prefill_inputs([4000], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    check_scan(p, 21, key_heads=[0, 7, 15])


def test_scan_malformed_cu_seqlens_is_a_no_op():
    p = inputs.prefill_inputs([100, 50], 1, 3, 128, 128, dtype=torch.bfloat16, seed=5,
                              initial_state_std=0.02)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta)]
    out = torch.full((150, 3, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    fin = torch.full((2, 3, 128, 128), 7.0, device=dev)
    bad = torch.tensor([0, 120, 100], dtype=torch.int32, device=dev)
    gdn.gdn_chunk_prefill_scan(*a, bad, p.initial_state.to(dev), out=out, final_state=fin,
                               chunks_per_group=1)
    torch.cuda.synchronize()
    assert (fin == 7.0).all()
    assert torch.isnan(out.float()).all()


def test_scan_rejects_bad_arguments():
    p = inputs.prefill_inputs([100], 1, 3, 64, 64, dtype=torch.bfloat16, seed=6)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    with pytest.raises(gdn.GDNError):
        gdn.gdn_chunk_prefill_scan(*a, chunks_per_group=2)   # d = 64: unsupported
    p = inputs.prefill_inputs([100], 1, 3, 128, 128, dtype=torch.bfloat16, seed=6)
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    with pytest.raises(gdn.GDNError):
        gdn.gdn_chunk_prefill_scan(*a, chunks_per_group=-1)
