"""Checks that pin the fp64 oracle to facts other than its own code.

Each check takes an oracle library handle (so the same checks can be run
against deliberately broken builds of the oracle) and returns the largest
relative error it saw; the tests compare that against a bound.  None of the
checks re-types the oracle's update rule: each uses a closed form, an
invariant, an explicit dense-matrix expansion or exact rational arithmetic.

The recurrence being pinned: S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
o_t = S_t q_t, a_t = exp(g_t) (Gated DeltaNet; pages "cf-1.com" section
"三个优化" item 2 and "reactapp.top" section "Exploiter l'architecture hybride").
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def check_beta_zero_decay(lib, seed=1) -> float:
    """b = 0: S_t = e^{g_1+..+g_t} S_0 and o_t = e^{gamma_t} S_0 q_t."""
    rng = np.random.default_rng(seed)
    lens = [7, 0, 12]
    T, Hk, Hv, d = sum(lens), 2, 4, 5
    cu = np.concatenate([[0], np.cumsum(lens)])
    q = unit(rng.standard_normal((T, Hk, d)))
    k = unit(rng.standard_normal((T, Hk, d)))
    v = rng.standard_normal((T, Hv, d))
    g = -rng.uniform(0.0, 0.5, (T, Hv))
    b = np.zeros((T, Hv))
    S0 = rng.standard_normal((len(lens), Hv, d, d))
    out, fin = oracle.prefill(q, k, v, g, b, cu, S0, lib=lib)
    err = 0.0
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        for h in range(Hv):
            hk = h // (Hv // Hk)
            gam = np.cumsum(g[s:e, h])
            for i, t in enumerate(range(s, e)):
                err = max(err, rel(out[t, h], np.exp(gam[i]) * S0[n, h] @ q[t, hk]))
            tot = np.exp(gam[-1]) if e > s else 1.0
            err = max(err, rel(fin[n, h], tot * S0[n, h]))
    return err


def check_orthonormal_retrieval(lib, seed=2) -> float:
    """a = 1, b = 1, orthonormal keys k_1..k_T (T < d):
    S_T k_j = v_j, S_T x = S_0 x for x orthogonal to every key, and from
    S_0 = 0, querying q_t = k_j (j <= t) returns exactly v_j."""
    rng = np.random.default_rng(seed)
    d, T = 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Qm.T[:T]
    perp = Qm.T[T:]
    v = rng.standard_normal((T, 1, d))
    g = np.zeros((T, 1))
    b = np.ones((T, 1))
    k = keys[:, None, :]
    err = 0.0
    S0 = rng.standard_normal((1, 1, d, d))
    _, fin = oracle.prefill(k, k, v, g, b, [0, T], S0, lib=lib)
    ST = fin[0, 0]
    for j in range(T):
        err = max(err, rel(ST @ keys[j], v[j, 0]))
    for x in perp:
        err = max(err, rel(ST @ x, S0[0, 0] @ x))
    # Zero start: query earlier keys.
    qsel = rng.integers(0, T, size=T)
    qsel = np.minimum(qsel, np.arange(T))
    q = keys[qsel][:, None, :]
    out, _ = oracle.prefill(q, k, v, g, b, [0, T], None, lib=lib)
    for t in range(T):
        err = max(err, rel(out[t, 0], v[qsel[t], 0]))
    return err


def check_overwrite(lib, seed=3) -> float:
    """b = 1, a = 1, any unit key: the new state maps k_t to v_t exactly
    (queried with q_t = k_t, o_t = S_t k_t = v_t)."""
    rng = np.random.default_rng(seed)
    T, d = 20, 6
    k = unit(rng.standard_normal((T, 1, d)))
    v = rng.standard_normal((T, 1, d))
    S0 = rng.standard_normal((1, 1, d, d))
    out, _ = oracle.prefill(k, k, v, np.zeros((T, 1)), np.ones((T, 1)), [0, T], S0, lib=lib)
    return max(rel(out[t, 0], v[t, 0]) for t in range(T))


def check_scalar_closed_form(lib, seed=4) -> float:
    """d = 1: s_T = s_0 prod_t m_t + sum_i b_i v_i k_i prod_{j>i} m_j with
    m_t = a_t (1 - b_t k_t^2), a first-order linear recurrence; o_t = s_t q_t."""
    rng = np.random.default_rng(seed)
    T = 30
    k = rng.uniform(-1, 1, (T, 1, 1))
    q = rng.standard_normal((T, 1, 1))
    v = rng.standard_normal((T, 1, 1))
    g = -rng.uniform(0, 0.3, (T, 1))
    b = rng.uniform(0, 1, (T, 1))
    s0 = rng.standard_normal()
    out, fin = oracle.prefill(q, k, v, g, b, [0, T], np.full((1, 1, 1, 1), s0), lib=lib)
    m = np.exp(g[:, 0]) * (1 - b[:, 0] * k[:, 0, 0] ** 2)
    c = b[:, 0] * v[:, 0, 0] * k[:, 0, 0]
    err = 0.0
    for t in range(T):
        st = s0 * np.prod(m[:t + 1]) + sum(c[i] * np.prod(m[i + 1:t + 1]) for i in range(t + 1))
        err = max(err, rel(out[t, 0, 0], st * q[t, 0, 0]))
        if t == T - 1:
            err = max(err, rel(fin[0, 0, 0, 0], st))
    return err


def dense_expansion(S0, q, k, v, a, b):
    """S_T = S_0 M_1..M_T + sum_i b_i v_i k_i^T M_{i+1}..M_T with explicit dense
    M_t = a_t (I - b_t k_t k_t^T); returns (outputs, S_T).  Works for numpy
    floats and for Fractions (object arrays)."""
    T, d = k.shape
    I = np.eye(d, dtype=object if isinstance(a[0], Fraction) else np.float64)
    if isinstance(a[0], Fraction):
        I = np.array([[Fraction(int(i == j)) for j in range(d)] for i in range(d)], dtype=object)
    M = [a[t] * (I - b[t] * np.outer(k[t], k[t])) for t in range(T)]
    outs = []
    for t in range(T):
        P = I.copy()
        for j in range(t + 1):
            P = P @ M[j]
        St = S0 @ P
        for i in range(t + 1):
            R = I.copy()
            for j in range(i + 1, t + 1):
                R = R @ M[j]
            St = St + b[i] * np.outer(v[i], k[i]) @ R
        outs.append(St @ q[t])
    return np.array(outs), St


def check_dense_products(lib, seed=5) -> float:
    """fp64 against the explicit product expansion on tiny inputs."""
    rng = np.random.default_rng(seed)
    err = 0.0
    for (T, dk, dv) in [(1, 3, 3), (6, 4, 4), (9, 3, 5), (5, 5, 2)]:
        q = rng.standard_normal((T, 1, dk))
        k = unit(rng.standard_normal((T, 1, dk)))
        v = rng.standard_normal((T, 1, dv))
        g = -rng.uniform(0, 0.7, (T, 1))
        b = rng.uniform(0, 1, (T, 1))
        S0 = rng.standard_normal((1, 1, dv, dk))
        out, fin = oracle.prefill(q, k, v, g, b, [0, T], S0, lib=lib)
        ref_o, ref_S = dense_expansion(S0[0, 0], q[:, 0], k[:, 0], v[:, 0], np.exp(g[:, 0]), b[:, 0])
        err = max(err, rel(out[:, 0], ref_o), rel(fin[0, 0], ref_S))
    return err


def check_exact_rational(lib, seed=6) -> float:
    """d <= 3, T <= 6 in exact rational arithmetic: the inputs are the fp64
    values handed to the oracle (converted exactly), a_t = exp(g_t) rounded to
    fp64 as the C library returns it, so the only error left is the oracle's
    own fp64 rounding."""
    rng = np.random.default_rng(seed)
    err = 0.0
    for (T, dk, dv) in [(4, 2, 3), (6, 3, 3), (3, 3, 1)]:
        q = rng.standard_normal((T, 1, dk))
        k = unit(rng.standard_normal((T, 1, dk)))
        v = rng.standard_normal((T, 1, dv))
        g = -rng.uniform(0, 1, (T, 1))
        b = rng.uniform(0, 1, (T, 1))
        S0 = rng.standard_normal((1, 1, dv, dk))
        out, fin = oracle.prefill(q, k, v, g, b, [0, T], S0, lib=lib)
        F = np.vectorize(Fraction, otypes=[object])
        a = [Fraction(math.exp(float(x))) for x in g[:, 0]]
        bb = [Fraction(float(x)) for x in b[:, 0]]
        ref_o, ref_S = dense_expansion(F(S0[0, 0]), F(q[:, 0]), F(k[:, 0]), F(v[:, 0]), a, bb)
        err = max(err, rel(out[:, 0], ref_o.astype(np.float64)),
                  rel(fin[0, 0], ref_S.astype(np.float64)))
    return err


def check_gqa_grouping(lib, seed=7) -> float:
    """Value head h reads key head h // (Hv/Hk) (contiguous groups): each value
    head of a 2-key/6-value problem equals a 1-key/1-value run on its key head."""
    rng = np.random.default_rng(seed)
    T, Hk, Hv, d = 9, 2, 6, 4
    q = unit(rng.standard_normal((T, Hk, d)))
    k = unit(rng.standard_normal((T, Hk, d)))
    v = rng.standard_normal((T, Hv, d))
    g = -rng.uniform(0, 0.5, (T, Hv))
    b = rng.uniform(0, 1, (T, Hv))
    out, fin = oracle.prefill(q, k, v, g, b, [0, T], None, lib=lib)
    err = 0.0
    for h in range(Hv):
        hk = h // 3
        o1, f1 = oracle.prefill(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1],
                                g[:, h:h + 1], b[:, h:h + 1], [0, T], None, lib=lib)
        err = max(err, rel(out[:, h], o1[:, 0]), rel(fin[0, h], f1[0, 0]))
    return err


def check_decode_equals_prefill(lib, seed=8) -> float:
    """T decode steps from S_0 reproduce a T-token prefill from S_0."""
    rng = np.random.default_rng(seed)
    T, Hk, Hv, d = 11, 1, 2, 4
    q = unit(rng.standard_normal((T, Hk, d)))
    k = unit(rng.standard_normal((T, Hk, d)))
    v = rng.standard_normal((T, Hv, d))
    g = -rng.uniform(0, 0.5, (T, Hv))
    b = rng.uniform(0, 1, (T, Hv))
    S0 = rng.standard_normal((1, Hv, d, d))
    out, fin = oracle.prefill(q, k, v, g, b, [0, T], S0, lib=lib)
    S = S0.copy()
    err = 0.0
    for t in range(T):
        o, S = oracle.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], S, lib=lib)
        err = max(err, rel(o[0], out[t]))
    return max(err, rel(S, fin))


def check_decode_gqa_grouping(lib, seed=9) -> float:
    """Decode with 2 key / 6 value heads: value head h reads key head
    h // (Hv/Hk), so each value head of one batched step equals a 1-key /
    1-value step on its own key head (contiguous groups; the same reading as
    the prefill's).  Three steps, each from the batched call's state."""
    rng = np.random.default_rng(seed)
    N, Hk, Hv, d = 3, 2, 6, 4
    S = rng.standard_normal((N, Hv, d, d))
    err = 0.0
    for _ in range(3):
        q = unit(rng.standard_normal((N, Hk, d)))
        k = unit(rng.standard_normal((N, Hk, d)))
        v = rng.standard_normal((N, Hv, d))
        g = -rng.uniform(0, 0.5, (N, Hv))
        b = rng.uniform(0, 1, (N, Hv))
        out, S_new = oracle.decode(q, k, v, g, b, S, lib=lib)
        for h in range(Hv):
            hk = h // (Hv // Hk)
            o1, s1 = oracle.decode(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1],
                                   g[:, h:h + 1], b[:, h:h + 1], S[:, h:h + 1].copy(), lib=lib)
            err = max(err, rel(out[:, h], o1[:, 0]), rel(S_new[:, h], s1[:, 0]))
        S = S_new
    return err


ALL_CHECKS = {
    "beta_zero_decay": (check_beta_zero_decay, 1e-13),
    "orthonormal_retrieval": (check_orthonormal_retrieval, 1e-13),
    "overwrite": (check_overwrite, 1e-12),
    "scalar_closed_form": (check_scalar_closed_form, 1e-12),
    "dense_products": (check_dense_products, 1e-12),
    "exact_rational": (check_exact_rational, 1e-13),
    "gqa_grouping": (check_gqa_grouping, 0.0),
    "decode_equals_prefill": (check_decode_equals_prefill, 0.0),
    "decode_gqa_grouping": (check_decode_gqa_grouping, 0.0),
}
