"""The bench's accounting, recounted on the CPU: the algorithmic flops per
token per value head from the list of products the chunked algorithm does,
the compulsory bytes from the sizes of the tensors a call actually moves,
and the traffic record's source check."""
import hashlib
import json
import os
from fractions import Fraction

import torch

import bench
from gated_deltanet_linear_chunk_gb300 import inputs

C, D, G = 64, 128, 3


def test_flops_per_token_head_from_the_products():
    # (flops per chunk per value head): 2 m n k per product; lower-triangular
    # operands count half; key-head products are shared by the G value heads;
    # the triangular inverse costs C^3 / 3.
    per_chunk = {
        "W S0^T": 2 * C * D * D,
        "Q~ S0^T": 2 * C * D * D,
        "Delta^T K~ (state update)": 2 * D * C * D,
        "U = T diag(b) V (T triangular)": Fraction(2 * C * C * D, 2),
        "W = T diag(b e^g) K (T triangular)": Fraction(2 * C * C * D, 2),
        "(M o Q K^T) Delta (M triangular)": Fraction(2 * C * C * D, 2),
        "K K^T, strictly lower, per key head": Fraction(2 * C * C * D, 2 * G),
        "Q K^T, lower, per key head": Fraction(2 * C * C * D, 2 * G),
        "(I + A)^-1": Fraction(C ** 3, 3),
    }
    per_token = sum(per_chunk.values()) / C
    # the bench rounds the two thirds down separately
    assert abs(per_token - bench.FLOPS_PER_TOKEN_HEAD) < 1
    recurrence = (per_chunk["W S0^T"] + per_chunk["Q~ S0^T"] +
                  per_chunk["Delta^T K~ (state update)"] +
                  per_chunk["U = T diag(b) V (T triangular)"] +
                  per_chunk["(M o Q K^T) Delta (M triangular)"]) / C
    assert recurrence == bench.FLOPS_RECURRENCE
    assert bench.FLOPS_PREP + bench.FLOPS_RECURRENCE == bench.FLOPS_PER_TOKEN_HEAD
    assert bench.flops_of(4000, 48) == 4000 * 48 * bench.FLOPS_PER_TOKEN_HEAD


def test_prefill_bytes_are_the_tensors_a_call_moves():
    p = inputs.prefill_inputs([300, 200], 16, 48, D, D, dtype=torch.bfloat16, seed=0)
    moved = sum(t.numel() * t.element_size() for t in (p.q, p.k, p.v, p.g, p.beta))
    moved += p.v.numel() * p.v.element_size()  # out has v's shape and dtype
    assert bench.prefill_bytes(500, 16, 48, D) == moved


def test_verify_bytes_are_the_tensors_a_call_moves():
    N, K, Hk, Hv = 4, 8, 16, 48
    q, k, v, g, beta = bench.verify_inputs(N, K, Hk, Hv, D)
    for state_bytes in (4, 2):
        moved = sum(t.numel() * t.element_size() for t in (q, k, v, g, beta))
        moved += v.numel() * v.element_size()                 # out
        moved += N * Hv * D * D * state_bytes * (1 + K)      # state read, K slots written
        assert bench.verify_bytes(N, K, Hk, Hv, D, state_bytes) == moved


def test_traffic_record_is_dropped_when_the_code_changes(tmp_path, monkeypatch):
    src = tmp_path / "gated_deltanet_linear_chunk_gb300" / "csrc" / "prefill_tc.cu"
    src.parent.mkdir(parents=True)
    src.write_text("// kernel source\nint x = 1;  // one\n")
    (tmp_path / "profiles").mkdir()
    rec = {"code_sha256": bench.code_digest(str(src)), "bytes_per_launch": {"fused": 123}}
    (tmp_path / "profiles" / "prefill_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("fused") == 123
    assert bench.recorded_traffic("prep") is None       # not captured
    src.write_text("// the same kernel, comments reworded\n\nint x = 1;  // still one\n")
    assert bench.recorded_traffic("fused") == 123       # comments do not count
    src.write_text("// kernel source\nint x = 2;  // one\n")
    assert bench.recorded_traffic("fused") is None      # stale record


def test_committed_traffic_record_is_well_formed():
    with open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "profiles",
                           "prefill_traffic.json")) as f:
        rec = json.load(f)
    assert len(rec["code_sha256"]) == 64
    for kernel, total in rec["bytes_per_launch"].items():
        assert total == sum(rec["read_write"][kernel])
        # at least the compulsory bytes of the 4000-token workload it was taken on
        assert total >= bench.prefill_bytes(4000, 16, 48, D)
