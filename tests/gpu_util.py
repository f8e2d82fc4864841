"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI binding and the fp64 oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import gated_deltanet_linear_chunk_gb300 as gdn
from gated_deltanet_linear_chunk_gb300 import inputs

# max |gpu - ref| / max |ref| per tensor, from the layer's specification:
# bf16 inputs with fp32 accumulation, and the fp32 check path.
TOL_BF16 = 1e-2
TOL_F32 = 1e-4


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if b.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)) / max(float(np.max(np.abs(b))), 1e-30))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def poison_workspace(p: inputs.PrefillInputs, dev) -> None:
    """Fills the binding's cached prefill workspace for this problem (created
    if needed) with 0xFF bytes, which read as NaN in every float field: a
    kernel that reads scratch it did not write this call shows up as NaN."""
    T, Hk, dk = p.q.shape
    Hv, dv = p.v.shape[1:]
    need = gdn.gdn_chunk_prefill_workspace_size(p.cu_seqlens.shape[0] - 1, T, Hk, Hv, dk, dv,
                                                p.q.dtype)
    ws = gdn._workspace(dev, need)
    if ws is not None:
        ws.fill_(0xFF)


def run_prefill(p: inputs.PrefillInputs, final=True, device="cuda", poison=True):
    """The prefill through the binding; with `poison`, out, the final state
    and the workspace start as NaN, so any element the call fails to write
    (or any stale scratch it reads) fails the comparison."""
    dev = torch.device(device)
    T, Hv, dv = p.v.shape
    N, dk = p.cu_seqlens.shape[0] - 1, p.q.shape[2]
    out = fin = None
    if poison:
        out = torch.full((T, Hv, dv), float("nan"), dtype=p.q.dtype, device=dev)
        if final:
            fin = torch.full((N, Hv, dv, dk), float("nan"), dtype=torch.float32, device=dev)
        poison_workspace(p, dev)
    out, fin = gdn.gdn_chunk_prefill(
        p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev),
        p.cu_seqlens.to(dev), None if p.initial_state is None else p.initial_state.to(dev),
        out=out, final_state=fin, output_final_state=final)
    torch.cuda.synchronize()
    return out, fin


def oracle_prefill(p: inputs.PrefillInputs, key_heads=None):
    """Oracle on all heads, or on whole key-head groups (value heads
    hk*G .. hk*G+G-1 for hk in key_heads).  Returns (out, final, value_heads)."""
    Hk, Hv = p.q.shape[1], p.v.shape[1]
    G = Hv // Hk
    if key_heads is None:
        key_heads = list(range(Hk))
    vh = [hk * G + j for hk in key_heads for j in range(G)]
    q = f64(p.q[:, key_heads])
    k = f64(p.k[:, key_heads])
    v = f64(p.v[:, vh])
    g = f64(p.g[:, vh])
    b = f64(p.beta[:, vh])
    h0 = None if p.initial_state is None else f64(p.initial_state[:, vh])
    out, fin = oracle.prefill(q, k, v, g, b, p.cu_seqlens.numpy(), h0)
    return out, fin, vh


def check_prefill(p: inputs.PrefillInputs, tol: float, key_heads=None):
    out, fin = run_prefill(p)
    o_ref, f_ref, vh = oracle_prefill(p, key_heads)
    e_out = rel(f64(out[:, vh]), o_ref)
    e_fin = rel(f64(fin[:, vh]), f_ref)
    assert np.isfinite(f64(out)).all(), "non-finite output"
    assert np.isfinite(f64(fin)).all(), "non-finite final state"
    assert e_out <= tol, f"out rel err {e_out:.3e} > {tol:.0e}"
    assert e_fin <= tol, f"final state rel err {e_fin:.3e} > {tol:.0e}"
    print(f"[parity] T={p.q.shape[0]} N={p.cu_seqlens.shape[0] - 1} dtype={p.q.dtype} "
          f"d={p.q.shape[2]} out {e_out:.3e} final {e_fin:.3e} (tol {tol:.0e})")
    return e_out, e_fin
