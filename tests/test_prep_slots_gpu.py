"""Kernel parity of the intra-chunk prep on its own: every chunk's products
(W^T, T diag(b), P, diag(e^gamma) Q, e^gamma, e^{gamma_L - gamma}) as the
prep kernel leaves them in the workspace, against the fp64 chunk model
(oracle/chunk_model.py, itself pinned to the token oracle).  The page this
layer comes from checks each of its kernels against a reference separately
(page "cf-1.com", section "精度"); an error confined to prep would otherwise
only show diluted through the layer's output."""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs
from gpu_util import TOL_BF16, rel
from oracle import chunk_model

pytestmark = pytest.mark.gpu

C = 64


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return gdn.library()


def image(raw: np.ndarray, rows: int) -> np.ndarray:
    """A bf16 image of `rows` rows of 64 elements (the layout the header
    documents: element (r, c) at byte 128 r + 16 ((c / 8) xor (r mod 8)) +
    2 (c mod 8)) as fp64 [rows, 64]."""
    chunks = raw[:rows * 128].reshape(rows, 8, 16)
    r = np.arange(rows)[:, None]
    logical = chunks[r, np.arange(8)[None, :] ^ (r % 8)]
    u16 = np.ascontiguousarray(logical).view(np.uint16).reshape(rows, 64)
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_prep(lib, p):
    """The chunk table and prep kernels only; returns (workspace bytes, layout)."""
    T, Hk, dk = p.q.shape
    Hv, dv = p.v.shape[1:]
    N = p.cu_seqlens.shape[0] - 1
    dev = torch.device("cuda")
    prob = gdn.make_problem(N, T, Hk, Hv, dk, dv, torch.bfloat16)
    need = lib.gdn_chunk_prefill_workspace_size(ctypes.byref(prob))
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)  # reads as NaN
    prob = gdn.make_problem(N, T, Hk, Hv, dk, dv, torch.bfloat16, ws)
    layout = (ctypes.c_int64 * 8)()
    assert lib.gdn_chunk_prefill_prep_layout(ctypes.byref(prob),
                                             ctypes.cast(layout, ctypes.c_void_p)) == 0
    args = [x.to(dev) for x in (p.q, p.k, p.g, p.beta, p.cu_seqlens)]
    rc = lib.gdn_chunk_prefill_prep_only(ctypes.byref(prob), *[a.data_ptr() for a in args],
                                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    return ws.cpu().numpy(), list(layout)


def check_slots(lib, p, heads=None):
    ws, lay = run_prep(lib, p)
    base, sbytes, o_wt, o_tb, o_p, o_q, o_eg, o_dec = lay
    Hk, Hv = p.q.shape[1], p.v.shape[1]
    G = Hv // Hk
    cu = p.cu_seqlens.tolist()
    q, k = (x.double().numpy() for x in (p.q, p.k))
    g, b = (x.double().numpy() for x in (p.g, p.beta))
    worst = {}
    tol_worst = 0.0
    chunk = 0
    for n in range(len(cu) - 1):
        for s in range(cu[n], cu[n + 1], C):
            e = min(s + C, cu[n + 1])
            L = e - s
            for h in (range(Hv) if heads is None else heads):
                hk = h // G
                slot = ws[base + (chunk * Hv + h) * sbytes:][:sbytes]
                gam, T, W, _ = chunk_model.chunk_prep(k[s:e, hk], np.zeros((L, 1)), g[s:e, h],
                                                       b[s:e, h])
                Qtil, P, dec = chunk_model.chunk_output_factors(q[s:e, hk], k[s:e, hk], gam)
                wt = image(slot[o_wt:], 128)
                tb = image(slot[o_tb:], 64)
                pp = image(slot[o_p:], 64)
                qt = np.concatenate([image(slot[o_q:], 64), image(slot[o_q + 8192:], 64)], 1)
                eg = slot[o_eg:o_eg + 256].view(np.float32).astype(np.float64)
                dc = slot[o_dec:o_dec + 256].view(np.float32).astype(np.float64)
                # The decay factors come from an fp32 prefix sum of g: a few
                # roundings of partial sums as large as sum |g| (scan depth
                # 6), i.e. an error of about 2^-24 * 8 * sum |g| in the exponent.
                tol_exp = max(1e-5, 8 * 2.0 ** -24 * float(np.sum(np.abs(g[s:e, h]))))
                tol_worst = max(tol_worst, tol_exp)
                errs = {
                    "W^T": rel(wt[:, :L], W.T),
                    "T diag(b)": rel(tb[:L, :L], T * b[s:e, h][None, :]),
                    "P": rel(pp[:L, :L], P),
                    "diag(e^gamma) Q": rel(qt[:L], Qtil),
                    "e^gamma": rel(eg[:L], np.exp(gam)),
                    "e^{gamma_L - gamma}": rel(dc[:L], dec),
                }
                # Tokens past the end: no contribution to W or U, decay held.
                where = f"sequence {n}, chunk at token {s} (L = {L}), head {h}"
                assert np.all(wt[:, L:] == 0), f"W^T past the end, {where}"
                assert np.all(tb[L:] == 0) and np.all(tb[:, L:] == 0), f"T diag(b), {where}"
                # (the prefix sum over the chunk adds in a different order for
                # each pair of tokens, so these agree to fp32 rounding)
                assert np.allclose(eg[L:], eg[L - 1], rtol=tol_exp, atol=0), \
                    f"e^gamma past the end {eg[L - 1:]}, {where}"
                assert np.allclose(dc[L:], 1.0, rtol=tol_exp, atol=0), \
                    f"decay past the end {dc[L:]}, {where}"
                for name, err in errs.items():
                    worst[name] = max(worst.get(name, 0.0), err)
            chunk += 1
    print("[prep parity] " + ", ".join(f"{k} {v:.2e}" for k, v in worst.items()))
    for name in ("e^gamma", "e^{gamma_L - gamma}"):
        assert worst[name] <= tol_worst, f"{name}: {worst[name]:.2e} > {tol_worst:.1e}"
    for name, err in worst.items():
        assert err <= TOL_BF16, f"{name}: rel err {err:.2e} > {TOL_BF16:.0e}"
    return worst


def test_prep_slots_small_ragged(lib):
    """Ragged chunks, a one-token and a five-token sequence, GQA 2 / 6."""
    p = inputs.prefill_inputs([130, 64, 5, 1, 200], 2, 6, 128, 128, dtype=torch.bfloat16,
                              seed=41)
    check_slots(lib, p)


def test_prep_slots_strong_decay_and_saturated_gates(lib):
    p = inputs.prefill_inputs([150], 1, 3, 128, 128, dtype=torch.bfloat16, seed=42)
    p.g[::7] = -30.0
    p.g[3::11] = -1e4
    p.beta[::5] = 0.0
    p.beta[2::5] = 1.0
    check_slots(lib, p)


def test_prep_slots_t4000_48_heads(lib):
    """The 4000-token workload: every chunk of every value head."""
    p = inputs.prefill_inputs([4000], 16, 48, 128, 128, dtype=torch.bfloat16, seed=0)
    check_slots(lib, p)
