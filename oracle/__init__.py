"""fp64 CPU oracle of the Gated DeltaNet recurrence (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product path (the
CUDA library and its binding) never imports this package, and this package
imports nothing from it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, OpenMP over
(sequence, value head)); this module compiles it with gcc and wraps it with
ctypes.  ``chunk_model`` holds an fp64 numpy restatement of the chunked
(WY/UT) form, used only to check the chunk algebra against this oracle.

Method: per token, ``S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T``,
``o_t = S_t q_t``, ``a_t = exp(g_t)`` -- the Gated DeltaNet layer of the hybrid
Qwen3.8-27B model (page "cf-1.com", section "三个优化", item 2; page
"reactapp.top", section "Exploiter l'architecture hybride").
"""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lib = None


def library_path(source: str = _SRC, tag: str = "") -> str:
    return os.path.join(_BUILD, f"libgdn_oracle{tag}_{platform.machine()}.so")


def build(source: str = _SRC, out: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when the compiler supports it)."""
    out = out or library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", source, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.gdn_oracle_prefill.restype = ctypes.c_int
    lib.gdn_oracle_prefill.argtypes = [I64, P, I64, I64, I64, I64, P, P, P, P, P, P,
                                       P, I64, P, P, ctypes.c_int]
    lib.gdn_oracle_decode.restype = ctypes.c_int
    lib.gdn_oracle_decode.argtypes = [I64, I64, I64, I64, I64, P, P, P, P, P,
                                      P, I64, P, P, ctypes.c_int]
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(load().gdn_oracle_max_threads())


def prefill(q, k, v, g, beta, cu_seqlens, initial_state=None,
            heads: Optional[Sequence[int]] = None, num_threads: int = 0,
            lib=None):
    """Token-by-token fp64 GDN prefill.

    q, k: [T, Hk, dk]; v: [T, Hv, dv]; g, beta: [T, Hv]; cu_seqlens: [N+1];
    initial_state: [N, Hv, dv, dk] or None (zeros).  ``heads`` restricts the
    work to a subset of value heads (their rows of ``out`` are the only ones
    filled; others are NaN).  Returns (out [T, Hv, dv], final [N, Hv, dv, dk]).
    """
    lib = lib or load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == q.shape and v.shape[0] == T and g.shape == (T, Hv)
    assert beta.shape == (T, Hv) and int(cu[-1]) == T
    h0 = None if initial_state is None else _f64(initial_state)
    if h0 is not None:
        assert h0.shape == (N, Hv, dv, dk)
    hl = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    out = np.full((T, Hv, dv), np.nan)
    final = np.full((N, Hv, dv, dk), np.nan)
    rc = lib.gdn_oracle_prefill(N, _ptr(cu), Hk, Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(g), _ptr(beta), _ptr(h0), _ptr(hl),
                                0 if hl is None else hl.shape[0],
                                _ptr(out), _ptr(final), int(num_threads))
    if rc != 0:
        raise ValueError("gdn_oracle_prefill rejected its arguments")
    return out, final


def decode(q, k, v, g, beta, state, heads: Optional[Sequence[int]] = None,
           num_threads: int = 0, lib=None, inplace: bool = False):
    """One fp64 recurrent step for N sequences.

    q, k: [N, Hk, dk]; v: [N, Hv, dv]; g, beta: [N, Hv]; state [N, Hv, dv, dk]
    (updated in place when ``inplace`` and it is a C-contiguous float64 array,
    else copied).  Returns (out [N, Hv, dv], new_state).
    """
    lib = lib or load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    if inplace:
        S = state
        assert isinstance(S, np.ndarray) and S.dtype == np.float64 and S.flags.c_contiguous
    else:
        S = _f64(state).copy()
    N, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    assert S.shape == (N, Hv, dv, dk) and g.shape == (N, Hv) and beta.shape == (N, Hv)
    hl = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    out = np.full((N, Hv, dv), np.nan)
    rc = lib.gdn_oracle_decode(N, Hk, Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(hl), 0 if hl is None else hl.shape[0],
                               _ptr(S), _ptr(out), int(num_threads))
    if rc != 0:
        raise ValueError("gdn_oracle_decode rejected its arguments")
    return out, S
