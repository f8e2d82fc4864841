"""Chunk-boundary state snapshots from the prefill (for prefix caching):
every slot against the fp64 oracle run on the prefix that ends at that
chunk boundary, plus the invariants (last slot of a sequence = its final
state, unwritten slots untouched, outputs identical to the plain call)."""
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


def slot_table(lens, stride=1):
    """(sequence, snapshot index, tokens covered) of every snapshot slot, in
    order: a snapshot every `stride` chunks and after the last chunk."""
    rows = []
    for n, L in enumerate(lens):
        chunks = (L + 63) // 64
        for i in range((chunks + stride - 1) // stride):
            rows.append((n, i, min(64 * stride * (i + 1), L)))
    return rows


def oracle_prefix_state(p, n, upto, heads):
    """fp64 state of sequence n after its first `upto` tokens (value heads
    `heads`, all of whose key heads are taken)."""
    cu = p.cu_seqlens.tolist()
    s = cu[n]
    Hk, Hv = p.q.shape[1], p.v.shape[1]
    G = Hv // Hk
    kh = sorted({h // G for h in heads})
    vh = [hk * G + j for hk in kh for j in range(G)]
    sl = slice(s, s + upto)
    h0 = None if p.initial_state is None else f64(p.initial_state[n:n + 1, vh])
    _, fin = oracle.prefill(f64(p.q[sl, kh]), f64(p.k[sl, kh]), f64(p.v[sl, vh]),
                            f64(p.g[sl, vh]), f64(p.beta[sl, vh]),
                            np.array([0, upto], dtype=np.int32), h0)
    return fin[0], vh


@pytest.mark.parametrize("stride", [1, 2])
def test_snapshots_small_varlen(stride):
    lens = [130, 0, 64, 77, 1, 300]
    p = inputs.prefill_inputs(lens, 2, 6, 128, 128, dtype=torch.bfloat16, seed=21,
                              initial_state_std=0.02)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    h0 = p.initial_state.to(dev)
    T, N = sum(lens), len(lens)
    slots = gdn.gdn_chunk_prefill_snapshot_slots(N, T, 2, 6, 128, 128, stride)
    snaps = torch.full((slots, 6, 128, 128), float("nan"), device=dev)
    out, fin, snaps = gdn.gdn_chunk_prefill_snapshots(*a, h0, output_final_state=True,
                                                      snapshots=snaps, snapshot_chunks=stride)
    ref_out, ref_fin = gdn.gdn_chunk_prefill(*a, h0, output_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    table = slot_table(lens, stride)
    worst = 0.0
    for sidx, (n, i, upto) in enumerate(table):
        ref, vh = oracle_prefix_state(p, n, upto, list(range(6)))
        e = rel(f64(snaps[sidx]), ref)
        worst = max(worst, e)
        assert e <= TOL_BF16, f"slot {sidx} (sequence {n}, snapshot {i}): {e:.3e}"
        if upto == lens[n]:
            assert torch.equal(snaps[sidx], fin[n]), "last slot of a sequence = final state"
    assert torch.isnan(snaps[len(table):]).all(), "slots past the batch's count are written"
    print(f"[parity] snapshots every {stride} chunks, varlen {lens}: {len(table)} slots, "
          f"worst {worst:.3e}")


def test_snapshots_t4000_sampled():
    """The 4000-token workload with a snapshot every 8 chunks (512 tokens):
    slots 0, 3 and 7 (the last) against the oracle on the prefix, two key-head
    groups."""
    p = inputs.prefill_inputs([4000], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    dev = torch.device("cuda")
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    out, fin, snaps = gdn.gdn_chunk_prefill_snapshots(*a, output_final_state=True,
                                                      snapshot_chunks=8)
    torch.cuda.synchronize()
    heads = [0, 1, 2, 30, 31, 32]
    for sidx in (0, 3, 7):  # tokens 512, 2048, 4000 (the last, partial group)
        upto = min(512 * (sidx + 1), 4000)
        ref, vh = oracle_prefix_state(p, 0, upto, heads)
        e = rel(f64(snaps[sidx][vh]), ref)
        assert e <= TOL_BF16, f"slot {sidx}: {e:.3e}"
    assert torch.equal(snaps[7], fin[0])


def test_snapshots_unsupported_configs():
    dev = torch.device("cuda")
    p = inputs.prefill_inputs([70], 1, 1, 64, 64, dtype=torch.float32, seed=22)
    a = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    with pytest.raises(gdn.GDNError):
        gdn.gdn_chunk_prefill_snapshots(*a)
