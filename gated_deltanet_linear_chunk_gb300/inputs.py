"""Seeded synthetic inputs for the GDN layer (shared by the tests, the bench
and the oracle's callers).

This module holds none of the layer's arithmetic.  It draws random numbers
and shapes them into the distributions of the workloads:

* q, k ~ N(0, 1), L2-normalised over the head dimension in fp64 (the layer
  expects unit q and k; the normalisation is the caller's job), then rounded
  to the storage dtype;
* v ~ N(0, 1);
* beta = sigmoid(z), g = -0.1 * softplus(z) with z ~ N(0, 1), computed in
  fp64, stored as fp32;
* states ~ N(0, 0.02**2) (standard deviation 0.02), fp32.

Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014; the 64-bit finaliser constants
as published by Vigna).  Element i of stream s under seed x is the finaliser
applied to ``key(x, s) + (i + 1) * 0x9E3779B97F4A7C15``, where key(x, s) is
itself the finaliser of ``x * 0x9E3779B97F4A7C15 + s``.  Uniforms take the top
53 bits; normals come from Box-Muller on consecutive pairs of uniforms.  The
integer part is identical on every platform; the float transforms use numpy's
libm, so cross-machine bit equality of the normals is not promised.

Stream numbers fix the order of draws: q=0, k=1, v=2, beta=3, g=4, initial
state=5; decode step s uses streams 16 + 8 s + {0: q, 1: k, 2: v, 3: beta, 4: g}.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22

STREAM_Q, STREAM_K, STREAM_V, STREAM_BETA, STREAM_G, STREAM_H0 = 0, 1, 2, 3, 4, 5


def _mix_(z: np.ndarray, tmp: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place (tmp is scratch of the same shape)."""
    np.right_shift(z, np.uint64(30), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=tmp)
    np.bitwise_xor(z, tmp, out=z)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        x = np.array([np.uint64(seed) * _GOLDEN + np.uint64(stream)], dtype=np.uint64)
        return _mix_(x, np.empty_like(x))[0]


class _Work:
    """Reusable block buffers (fresh allocations are slow to first touch)."""

    def __init__(self, n: int):
        self.ctr = np.empty(n, dtype=np.uint64)
        self.tmp = np.empty(n, dtype=np.uint64)
        self.u = np.empty(n, dtype=np.float64)
        self.r = np.empty(n // 2, dtype=np.float64)
        self.th = np.empty(n // 2, dtype=np.float64)
        self.c = np.empty(n // 2, dtype=np.float64)


def _uniform_block(key, start: int, n: int, w: _Work) -> np.ndarray:
    z = w.ctr[:n]
    np.copyto(z, np.arange(start + 1, start + n + 1, dtype=np.uint64))
    with np.errstate(over="ignore"):
        np.multiply(z, _GOLDEN, out=z)
        np.add(z, key, out=z)
        _mix_(z, w.tmp[:n])
    np.right_shift(z, np.uint64(11), out=z)
    u = w.u[:n]
    np.multiply(z, 1.0 / 9007199254740992.0, out=u, casting="unsafe")
    return u


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniforms in [0, 1) (fp64) for elements offset .. offset+n-1."""
    key = _key(seed, stream)
    out = np.empty(n, dtype=np.float64)
    w = _Work(min(n, _BLOCK))
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        out[s:e] = _uniform_block(key, offset + s, e - s, w)
    return out


def _normal_range(key, out: np.ndarray, s: int, e: int) -> None:
    """Normals for pair indices s..e-1 of the stream, written into out."""
    half = _BLOCK // 2
    w = _Work(2 * min(e - s, half))
    for b in range(s, e, half):
        be = min(e, b + half)
        k = be - b
        u = _uniform_block(key, 2 * b, 2 * k, w)
        r, th, c = w.r[:k], w.th[:k], w.c[:k]
        np.negative(u[0::2], out=r)
        np.log1p(r, out=r)
        np.multiply(r, -2.0, out=r)
        np.sqrt(r, out=r)
        np.multiply(u[1::2], 2.0 * np.pi, out=th)
        np.cos(th, out=c)
        np.multiply(r, c, out=out[2 * b:2 * be:2])
        np.sin(th, out=c)
        np.multiply(r, c, out=out[2 * b + 1:2 * be:2])


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (fp64) by Box-Muller over pairs of uniforms.

    Work is split over threads by counter range; the values do not depend on
    the number of threads.
    """
    key = _key(seed, stream)
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    per = _BLOCK // 2
    ranges = [(s, min(m, s + per)) for s in range(0, m, per)]
    if len(ranges) <= 1:
        for s, e in ranges:
            _normal_range(key, out, s, e)
    else:
        workers = min(len(ranges), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(max_workers=workers) as pool:
            list(pool.map(lambda r: _normal_range(key, out, r[0], r[1]), ranges))
    return out[:n]


def _unit_rows(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _to(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


@dataclass
class PrefillInputs:
    q: torch.Tensor          # [T, Hk, dk]
    k: torch.Tensor          # [T, Hk, dk]
    v: torch.Tensor          # [T, Hv, dv]
    g: torch.Tensor          # [T, Hv] fp32
    beta: torch.Tensor       # [T, Hv] fp32
    cu_seqlens: torch.Tensor  # [N+1] int32
    initial_state: Optional[torch.Tensor]  # [N, Hv, dv, dk] fp32 or None


def gates(seed: int, stream_beta: int, stream_g: int, shape):
    n = int(np.prod(shape))
    beta = 1.0 / (1.0 + np.exp(-normal(seed, stream_beta, n)))
    g = -0.1 * np.logaddexp(0.0, normal(seed, stream_g, n))
    return (torch.from_numpy(beta.astype(np.float32).reshape(shape)),
            torch.from_numpy(g.astype(np.float32).reshape(shape)))


def unit_heads(seed: int, stream: int, shape, dtype: torch.dtype) -> torch.Tensor:
    n = int(np.prod(shape))
    return _to(_unit_rows(normal(seed, stream, n).reshape(shape)), dtype)


def state(seed: int, stream: int, shape, std: float = 0.02) -> torch.Tensor:
    n = int(np.prod(shape))
    return torch.from_numpy((std * normal(seed, stream, n)).astype(np.float32).reshape(shape))


def prefill_inputs(seqlens, Hk: int, Hv: int, dk: int, dv: int,
                   dtype: torch.dtype = torch.bfloat16, seed: int = 0,
                   initial_state_std: Optional[float] = None) -> PrefillInputs:
    """Packed varlen prefill inputs on the host (CPU tensors)."""
    seqlens = [int(s) for s in seqlens]
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    q = unit_heads(seed, STREAM_Q, (T, Hk, dk), dtype)
    k = unit_heads(seed, STREAM_K, (T, Hk, dk), dtype)
    v = _to(normal(seed, STREAM_V, T * Hv * dv).reshape(T, Hv, dv), dtype)
    beta, g = gates(seed, STREAM_BETA, STREAM_G, (T, Hv))
    h0 = None
    if initial_state_std is not None:
        h0 = state(seed, STREAM_H0, (len(seqlens), Hv, dv, dk), initial_state_std)
    return PrefillInputs(q, k, v, g, beta, torch.from_numpy(cu), h0)


def prefill_inputs_on_device(seqlens, Hk: int, Hv: int, dk: int, dv: int, device,
                             dtype: torch.dtype = torch.bfloat16, seed: int = 0,
                             initial_state_std: Optional[float] = None) -> PrefillInputs:
    """The same recipe as prefill_inputs, drawn with torch's seeded generator
    on `device` (fp32 arithmetic): for timing large workloads, where the
    host generator would take tens of seconds.  The values differ from
    prefill_inputs'; the parity tests use prefill_inputs."""
    seqlens = [int(s) for s in seqlens]
    T = sum(seqlens)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def normal_(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32)

    def unit(x):
        return (x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)).to(dtype)

    q = unit(normal_(T, Hk, dk))
    k = unit(normal_(T, Hk, dk))
    v = normal_(T, Hv, dv).to(dtype)
    beta = torch.sigmoid(normal_(T, Hv))
    g = -0.1 * torch.nn.functional.softplus(normal_(T, Hv))
    h0 = None
    if initial_state_std is not None:
        h0 = initial_state_std * normal_(len(seqlens), Hv, dv, dk)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(seqlens)]), dtype=torch.int32, device=dev)
    return PrefillInputs(q, k, v, g.contiguous(), beta.contiguous(), cu, h0)


@dataclass
class DecodeStepInputs:
    q: torch.Tensor     # [N, Hk, dk]
    k: torch.Tensor     # [N, Hk, dk]
    v: torch.Tensor     # [N, Hv, dv]
    g: torch.Tensor     # [N, Hv] fp32
    beta: torch.Tensor  # [N, Hv] fp32


def decode_step_inputs(step: int, N: int, Hk: int, Hv: int, dk: int, dv: int,
                       dtype: torch.dtype = torch.bfloat16, seed: int = 0) -> DecodeStepInputs:
    base = 16 + 8 * step
    q = unit_heads(seed, base + 0, (N, Hk, dk), dtype)
    k = unit_heads(seed, base + 1, (N, Hk, dk), dtype)
    v = _to(normal(seed, base + 2, N * Hv * dv).reshape(N, Hv, dv), dtype)
    beta, g = gates(seed, base + 3, base + 4, (N, Hv))
    return DecodeStepInputs(q, k, v, g, beta)


def decode_state(N: int, Hv: int, dv: int, dk: int, seed: int = 0, std: float = 0.02) -> torch.Tensor:
    return state(seed, STREAM_H0, (N, Hv, dv, dk), std)
