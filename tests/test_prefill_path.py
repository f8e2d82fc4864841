"""Which kernels a prefill runs (gdn_prefill_path, no device needed).  Each
case is a batch whose paths were timed on a GB300 (152 SMs, 16 key / 48 value
heads, d = 128, bf16, L2 flushed); the comment gives the measured call times.
The cost models see only the token and sequence counts, so the one case they
get wrong by design is marked: unequal lengths they cannot see."""
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn

SEP, FUSED, PER_HEAD = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("lens,want", [
    ([4000], FUSED),        # fused 111 us, separate 141
    ([20480], FUSED),       # 431 against 632
    ([2000], FUSED),        # 71.3 against 81.6
    ([1000], SEP),          # 50.8 against 51.9
    ([352], SEP),           # 30.3 against 38.5
    ([256], SEP),           # 27.3 against 32.4
    ([2000] * 2, SEP),      # 114.3; fused 164.5, per head 121.5
    ([4000] * 2, SEP),      # 200.4; per head 206.5
    ([1000] * 3, SEP),      # 89.7; per head 98.9
    ([2048] * 3, SEP),      # 163.0; per head 167.6
    ([512, 1000, 2048, 4000, 6000, 8192, 16384, 32768], PER_HEAD),  # 1510 against 1861
    ([2000] * 4, PER_HEAD),  # 208.5 against 233.1
    ([1024] * 8, PER_HEAD),  # 210.6 against 218.8
    ([512] * 16, PER_HEAD),  # 210.6 against 219.3
    ([128] * 64, PER_HEAD),  # 212.7 against 243.4
    ([4] * 2000, PER_HEAD),  # 2962 against 4276
    ([8000, 1000], SEP),     # by design: per head measured 226.9 against 277.2
])
def test_default_path_follows_the_measurements(lens, want):
    assert gdn.gdn_prefill_path(len(lens), sum(lens), 16, 48, mode=2) == want


def test_modes_and_limits():
    path = gdn.gdn_prefill_path
    assert path(1, 4000, 16, 48, mode=0) == SEP
    assert path(2, 4000, 16, 48, mode=1) == FUSED          # 96 + 16 <= 152 SMs
    assert path(4, 8000, 16, 48, mode=1) == PER_HEAD       # 192 recurrences do not fit
    assert path(1, 4000, 16, 48, mode=3) == PER_HEAD
    assert path(2, 500, 16, 144, mode=2) == SEP            # 144 + 16 > 152: no fused variant
    assert path(2, 500, 16, 144, mode=3) == SEP
    assert path(1, 4000, 16, 48, sms=0, mode=2) == SEP     # fused kernels unavailable
    assert path(1, 0, 16, 48, mode=1) == SEP               # nothing to do
    assert path(1, 100, 1, 1, 64, 64, dtype=torch.float32) == -1   # no tensor-core path
    assert path(1, 100, 16, 48, sms=-1) == -1
