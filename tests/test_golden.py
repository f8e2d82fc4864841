"""Figures the pages print, pinned against the workload the library is built
and benchmarked for (tests/golden/state_sizes.json cites the passage): the
fp32 state of one request over the 48 GDN layers is about 150 MB, which the
workload's 48 value heads of 128 x 128 give (151.0 MB); and the 16-bit state the decode and verify
steps can keep halves it, enough for every configured slot where the fp32
state allowed 37."""
import json
import os

import torch

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "state_sizes.json")


def facts():
    with open(GOLDEN) as f:
        return json.load(f)["facts"]


def state_bytes_per_layer(element_bytes):
    Hv, d = bench.DECODE["Hv"], bench.DECODE["d"]
    assert (bench.PREFILL["Hv"], bench.PREFILL["d"]) == (Hv, d)
    return Hv * d * d * element_bytes


def test_layer_split():
    f = facts()
    assert f["attention_layers"] + f["gdn_layers"] == f["total_layers"]


def test_fp32_state_per_request_matches_the_page():
    f = facts()
    fp32 = torch.empty((), dtype=torch.float32).element_size()
    per_request = f["gdn_layers"] * state_bytes_per_layer(fp32)
    # "about 150 MB": the workload's 48 x 128 x 128 fp32 state is 151.0 MB
    assert abs(per_request / 1e6 - f["fp32_state_mb_per_request"]) <= 0.02 * f[
        "fp32_state_mb_per_request"]
    # "about" cannot tell 47 or 49 heads from 48, but it rules out the other
    # usual shapes: 32 or 64 value heads, head dimension 64 or 256
    for Hv, d in ((32, 128), (64, 128), (48, 64), (48, 256)):
        other = f["gdn_layers"] * Hv * d * d * fp32 / 1e6
        assert abs(other - f["fp32_state_mb_per_request"]) > 0.02 * f["fp32_state_mb_per_request"]


def test_fp16_state_fits_every_configured_slot():
    f = facts()
    fp32 = torch.empty((), dtype=torch.float32).element_size()
    fp16 = torch.empty((), dtype=torch.float16).element_size()
    s32 = f["gdn_layers"] * state_bytes_per_layer(fp32)
    s16 = f["gdn_layers"] * state_bytes_per_layer(fp16)
    # the smallest state pool that holds 37 fp32 states but not 38 ...
    pool = f["fp32_max_concurrent_requests"] * s32
    assert pool // s32 == f["fp32_max_concurrent_requests"]
    assert pool < (f["fp32_max_concurrent_requests"] + 1) * s32
    # ... holds every configured slot once the state is stored in 16 bits
    assert pool // s16 >= f["configured_request_slots"]
    assert f["fp16_state_makes_all_slots_usable"]
