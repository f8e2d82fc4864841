"""The fused prep + recurrence kernel against the separate kernels and the
fp64 oracle.  Both paths run the same arithmetic per chunk, so their outputs
and final states are equal bit for bit; the fused path is forced on for
batches the cost model would send to the separate kernels.  Batches whose
(sequence, value head) recurrences do not fit beside prep take the fused
variant with one recurrence per value head over all sequences in turn
(reported as 2 by the timed call)."""
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
    yield
    gdn.gdn_prefill_fused_mode(2)


def run(p, mode):
    """The timed entry point reports which path ran; its events bracket the
    kernels in order."""
    gdn.gdn_prefill_fused_mode(mode)
    dev = torch.device("cuda")
    out, fin, fused, ev = gdn.gdn_chunk_prefill_timed(
        p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev),
        p.cu_seqlens.to(dev), None if p.initial_state is None else p.initial_state.to(dev),
        output_final_state=True)
    torch.cuda.synchronize()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(t >= 0.0 for t in ms)
    if fused:
        assert ms[1] < 0.01, "no prep launch between events 1 and 2 on the fused path"
    return out, fin, fused


@pytest.mark.parametrize("lens,Hk,Hv", [
    ([130, 1, 64, 0, 77, 400], 2, 6),   # ragged, empty and one-token sequences
    ([1000], 1, 3),
    ([2000, 2000], 4, 12),
    ([300, 2500, 900], 8, 24),
])
def test_fused_equals_separate_and_oracle(lens, Hk, Hv):
    p = inputs.prefill_inputs(lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=21,
                              initial_state_std=0.02)
    o1, f1, fused1 = run(p, 1)
    o0, f0, fused0 = run(p, 0)
    assert fused1 and not fused0
    assert torch.equal(o1, o0), "outputs differ between the fused and separate kernels"
    assert torch.equal(f1, f0), "final states differ"
    o_ref, f_ref, vh = oracle_prefill(p)
    e_o, e_f = rel(f64(o1[:, vh]), o_ref), rel(f64(f1[:, vh]), f_ref)
    print(f"[parity] fused lens={lens} {Hk}/{Hv}: out {e_o:.3e} final {e_f:.3e}")
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16


@pytest.mark.parametrize("lens,Hk,Hv,h0", [
    # 8 x 48 recurrences: one per value head; empty, one-token and ragged
    # sequences, the first ones shorter than the four chunks each recurrence
    # preps itself (so its own prep spans sequences)
    ([64, 1, 0, 100, 130, 2000, 0, 77, 1000, 0], 16, 48, True),
    ([0, 0, 700, 64, 1500], 16, 48, False),
    # 40 sequences x 6 value heads (240 recurrences)
    ([37 * (i % 7) + 64 * (i % 3) for i in range(40)], 2, 6, True),
])
def test_multi_fused_equals_separate_and_oracle(lens, Hk, Hv, h0):
    p = inputs.prefill_inputs(lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=23,
                              initial_state_std=0.02 if h0 else None)
    o1, f1, fused1 = run(p, 1)
    o0, f0, fused0 = run(p, 0)
    assert fused1 == 2 and fused0 == 0
    assert torch.equal(o1, o0), "outputs differ between the fused and separate kernels"
    assert torch.equal(f1, f0), "final states differ"
    o_ref, f_ref, vh = oracle_prefill(p)
    e_o, e_f = rel(f64(o1[:, vh]), o_ref), rel(f64(f1[:, vh]), f_ref)
    print(f"[parity] fused per head N={len(lens)} {Hk}/{Hv}: out {e_o:.3e} final {e_f:.3e}")
    assert e_o <= TOL_BF16 and e_f <= TOL_BF16


def test_default_choice_of_the_per_head_variant():
    """The default (mode 2) takes the per-head fused variant where its cost
    model expects it to be faster than the separate kernels: several waves of
    (sequence, value head) recurrences; not for three equal sequences, whose
    144 recurrences run in one wave; never with more value heads than it
    leaves room for (Hv + 16 > 152 SMs).  Mode 3 takes it whenever it can
    run."""
    for lens, want in (([1500, 900, 2600, 1200], 2), ([1024] * 8, 2), ([1000] * 3, 0)):
        p = inputs.prefill_inputs(lens, 16, 48, 128, 128, dtype=torch.bfloat16, seed=24)
        _, _, fused = run(p, 2)
        assert fused == want, lens
    p = inputs.prefill_inputs([1000] * 3, 16, 48, 128, 128, dtype=torch.bfloat16, seed=24)
    assert run(p, 3)[2] == 2
    p = inputs.prefill_inputs([300, 200], 16, 144, 128, 128, dtype=torch.bfloat16, seed=24)
    assert run(p, 2)[2] == 0 and run(p, 3)[2] == 0
    gdn.gdn_prefill_fused_mode(2)


def test_fused_mode_query_and_default():
    old = gdn.gdn_prefill_fused_mode(-1)
    assert old in (0, 1, 2, 3)
    assert gdn.gdn_prefill_fused_mode(2) == old
    assert gdn.gdn_prefill_fused_mode(7) == 2   # out of range: query only
    p = inputs.prefill_inputs([4000], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    _, _, fused = run(p, 2)
    assert fused, "the cost model picks the fused kernel for one 4000-token sequence"
    p = inputs.prefill_inputs([352], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    _, _, fused = run(p, 2)
    assert not fused, "a short sequence does not repay the fused kernel's first prep round"
    p = inputs.prefill_inputs([2000, 2000], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    _, _, fused = run(p, 2)
    assert not fused, "two sequences x 48 heads leave too few SMs for prep"


def test_timed_call_equals_plain_call():
    """Timing changes only the launch attributes, never the results."""
    p = inputs.prefill_inputs([700, 64], 2, 6, 128, 128, dtype=torch.bfloat16, seed=22,
                              initial_state_std=0.02)
    dev = torch.device("cuda")
    args = [x.to(dev) for x in (p.q, p.k, p.v, p.g, p.beta, p.cu_seqlens)]
    h0 = p.initial_state.to(dev)
    o1, f1 = gdn.gdn_chunk_prefill(*args, h0, output_final_state=True)
    o2, f2, _, _ = gdn.gdn_chunk_prefill_timed(*args, h0, output_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


@pytest.mark.parametrize("lens,Hk,Hv", [
    ([4000], 16, 48), ([300], 16, 48), ([2000, 2000], 16, 48), ([1024] * 8, 16, 48),
    ([700, 64], 2, 6),
])
def test_path_diagnostic_matches_the_call(lens, Hk, Hv):
    """gdn_prefill_path (sizes only, no device) names the kernels a real call
    runs on this GPU, in the default mode and with the per-head variant forced."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = inputs.prefill_inputs(lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, seed=25)
    for mode in (2, 3):
        _, _, ran = run(p, mode)
        assert gdn.gdn_prefill_path(len(lens), sum(lens), Hk, Hv, sms=sms, mode=mode) == ran
    gdn.gdn_prefill_fused_mode(2)
