"""The tcgen05 operand layouts (K-major and MN-major 128-byte-swizzled bf16
tiles, negated A, accumulate) that the prefill kernels use, each checked
against a plain matmul on one 128-row tile."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.join(os.path.dirname(HERE), "gated_deltanet_linear_chunk_gb300")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("probe") / "libtc_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", os.path.join(PKG, "csrc"),
                    "-I", os.path.join(os.path.dirname(HERE), "include"),
                    os.path.join(HERE, "csrc", "tc_probe.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.tc_probe_run.restype = ctypes.c_int
    lib.tc_probe_run.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_void_p]
    return lib


def bf(x):
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 6])
def test_layout(probe, mode):
    rng = np.random.default_rng(mode)
    K = 64 if mode in (1, 2) else 128
    N = 128 if mode == 2 else 64
    a = rng.standard_normal((K, 128) if mode == 1 else (128, K)).astype(np.float32)
    b = rng.standard_normal((K, N) if mode in (2, 4) else (N, K)).astype(np.float32)
    A = bf(a).T if mode == 1 else bf(a)
    B = bf(b) if mode in (2, 4) else bf(b).T
    ref = A @ B
    if mode == 3:
        ref = ref - ref
    da = torch.from_numpy(a).cuda()
    db = torch.from_numpy(b).cuda()
    dd = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_run(da.data_ptr(), db.data_ptr(), dd.data_ptr(), mode, st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    got = dd.cpu().double().numpy()
    assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.abs(A @ B).max())


def test_m64_lane_layout(probe):
    """M = 64: find which TMEM lane holds each row of D, and check the values.
    The mapping found is printed; rows must land on distinct lanes."""
    rng = np.random.default_rng(5)
    a = rng.standard_normal((64, 64)).astype(np.float32)
    b = rng.standard_normal((64, 64)).astype(np.float32)
    ref = bf(a) @ bf(b)
    da = torch.from_numpy(a).cuda()
    db = torch.from_numpy(b).cuda()
    dd = torch.full((128, 64), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_run(da.data_ptr(), db.data_ptr(), dd.data_ptr(), 5, st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    got = dd.cpu().double().numpy()
    lanes = []
    for r in range(64):
        err = np.abs(got - ref[r][None, :]).max(axis=1)
        lane = int(np.argmin(err))
        assert err[lane] <= 1e-4 * max(1.0, np.abs(ref).max()), f"row {r} not found"
        lanes.append(lane)
    print("M=64 row->lane:", lanes)
    assert len(set(lanes)) == 64


@pytest.mark.parametrize("mode", [7, 8])
def test_mma_issue_and_latency(probe, mode):
    """Cycles to issue 64 tcgen05.mma (M=128, K=16) from one thread, and to
    complete them, for operand placements and majors the kernels use
    (printed; sanity-checked only)."""
    rng = np.random.default_rng(7)
    a = rng.standard_normal((128, 128)).astype(np.float32)
    b = rng.standard_normal((64, 128)).astype(np.float32)
    dd = torch.zeros((128, 64), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_run(torch.from_numpy(a).cuda().data_ptr(),
                            torch.from_numpy(b).cuda().data_ptr(), dd.data_ptr(), mode, st.data_ptr())
    assert rc == 0
    t = dd.flatten()[:12].cpu().numpy()
    names = ["A smem, B K-major, N=64", "A smem, B K-major, N=128", "A TMEM, B K-major, N=64",
             "A TMEM, B MN-major, N=64", "A smem, B MN-major, N=64", "A TMEM, B MN-major, N=128"]
    for v, nm in enumerate(names):
        print(f"[{'warp' if mode == 8 else 'thread'} issue] 64 MMAs {nm}: issue {t[2 * v]:.0f} cyc, done {t[2 * v + 1]:.0f} cyc")
    assert (t[1::2] > 0).all()


def test_mma_accumulator_chains(probe):
    """64 MMAs into one accumulator vs interleaved over several (printed)."""
    rng = np.random.default_rng(9)
    a = rng.standard_normal((128, 128)).astype(np.float32)
    b = rng.standard_normal((64, 128)).astype(np.float32)
    dd = torch.zeros((128, 64), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_run(torch.from_numpy(a).cuda().data_ptr(),
                            torch.from_numpy(b).cuda().data_ptr(), dd.data_ptr(), 9, st.data_ptr())
    assert rc == 0
    t = dd.flatten()[:12].cpu().numpy()
    names = ["N=64 x1 chain", "N=64 x4 chains", "N=128 x1", "N=128 x2", "N=256 x1", "N=64 x2"]
    for v, nm in enumerate(names):
        print(f"[chains] 64 MMAs {nm}: issue {t[2 * v]:.0f} cyc, done {t[2 * v + 1]:.0f} cyc")
    assert (t[1::2] > 0).all()


def test_mma_group_latency(probe):
    """Issue -> commit -> wait latency of small MMA groups (printed)."""
    rng = np.random.default_rng(10)
    a = rng.standard_normal((128, 128)).astype(np.float32)
    b = rng.standard_normal((64, 128)).astype(np.float32)
    dd = torch.zeros((128, 64), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.tc_probe_run(torch.from_numpy(a).cuda().data_ptr(),
                            torch.from_numpy(b).cuda().data_ptr(), dd.data_ptr(), 10, st.data_ptr())
    assert rc == 0
    t = dd.flatten()[:6].cpu().numpy()
    names = ["8 x N=64, A TMEM, B K-major", "8 x N=64, A TMEM, B MN-major",
             "8 x N=64, A smem K-major, B K-major", "8 x N=64, A smem MN-major, B K-major",
             "4 x N=128, A TMEM, B K-major", "4 x N=128, A TMEM, B MN-major"]
    for v, nm in enumerate(names):
        print(f"[group] {nm}: {t[v]:.0f} cyc")
    assert (t > 0).all()
