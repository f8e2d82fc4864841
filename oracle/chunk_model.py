"""fp64 numpy model of the chunked (WY/UT) form of the GDN recurrence.

TEST INFRASTRUCTURE ONLY.  This is not the oracle: it is a second, blocked
evaluation of the same recurrence, checked against the token-by-token oracle
in ``gdn_oracle.c`` to 1e-12, and used to confirm the chunk algebra that the
CUDA kernels implement.  It shares no code with them.

Derivation (chunk of L <= C tokens, start state S0, gamma_r = g_1 + ... + g_r):
write delta_t = b_t (v_t - a_t S_{t-1} k_t), so S_t = a_t S_{t-1} + delta_t k_t^T
and, unrolled inside the chunk,
    S_r = e^{gamma_r} S0 + sum_{i<=r} e^{gamma_r - gamma_i} delta_i k_i^T.
Substituting into delta_t gives the unit lower-triangular system
    (I + A) Delta = diag(b) V - diag(b e^gamma) K S0^T,
    A_ti = b_t e^{gamma_t - gamma_i} (k_t . k_i)  for i < t,
so with T = (I + A)^-1, W = T diag(b e^gamma) K, U = T diag(b) V:
    Delta = U - W S0^T
    O     = diag(e^gamma) Q S0^T + (M o Q K^T) Delta,  M_ri = e^{gamma_r - gamma_i}, i <= r
    S_end = e^{gamma_L} S0 + Delta^T Ktil,  Ktil_i = e^{gamma_L - gamma_i} k_i.
The pages fix the chunk length (64) and the three-stage split (intra-chunk
prep, inter-chunk recurrence, output): page "cf-1.com", section "三个优化",
item 2 "GDN prefill".
"""
from __future__ import annotations

import numpy as np


def chunk_prep(Kc, Vc, gc, bc):
    """Intra-chunk prep: returns (gamma, T, W, U) for one chunk of one head."""
    L = Kc.shape[0]
    gam = np.cumsum(gc)
    decay = np.exp(gam[:, None] - gam[None, :])
    A = np.tril(bc[:, None] * decay * (Kc @ Kc.T), -1)
    T = np.linalg.inv(np.eye(L) + A)
    W = T @ ((bc * np.exp(gam))[:, None] * Kc)
    U = T @ (bc[:, None] * Vc)
    return gam, T, W, U


def chunk_output_factors(Qc, Kc, gam):
    """The state-independent factors of the chunk's output and state update:
    (Qtil = diag(e^gamma) Q, P = M o Q K^T, dec = e^{gamma_L - gamma})."""
    M = np.tril(np.exp(gam[:, None] - gam[None, :]))
    return np.exp(gam)[:, None] * Qc, M * (Qc @ Kc.T), np.exp(gam[-1] - gam)


def chunk_step(S, Qc, Kc, Vc, gc, bc):
    """One chunk: returns (O [L, dv], S_end) from the start state S [dv, dk]."""
    gam, T, W, U = chunk_prep(Kc, Vc, gc, bc)
    Delta = U - W @ S.T
    Qtil, P, dec = chunk_output_factors(Qc, Kc, gam)
    O = Qtil @ S.T + P @ Delta
    Ktil = dec[:, None] * Kc
    S_end = np.exp(gam[-1]) * S + Delta.T @ Ktil
    return O, S_end


def prefill(q, k, v, g, beta, cu_seqlens, initial_state=None, chunk=64):
    """Chunked fp64 prefill with the same interface as ``oracle.prefill``."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, Hk, dk = q.shape
    Hv, dv = v.shape[1:]
    group = Hv // Hk
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    out = np.zeros((T, Hv, dv))
    final = np.zeros((N, Hv, dv, dk))
    for n in range(N):
        for h in range(Hv):
            hk = h // group
            S = (np.zeros((dv, dk)) if initial_state is None
                 else np.array(initial_state[n, h], dtype=np.float64))
            for s in range(cu[n], cu[n + 1], chunk):
                e = min(s + chunk, cu[n + 1])
                O, S = chunk_step(S, q[s:e, hk], k[s:e, hk], v[s:e, h], g[s:e, h], beta[s:e, h])
                out[s:e, h] = O
            final[n, h] = S
    return out, final
