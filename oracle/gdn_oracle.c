/*
 * gdn_oracle.c -- fp64 CPU oracle for the Gated DeltaNet (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the plain token-by-token definition, no chunking):
 *
 *   For every sequence n and value head h, with key head hk = h / (Hv/Hk)
 *   (contiguous GQA groups: value heads 3j, 3j+1, 3j+2 read key head j when
 *   Hv = 3 Hk), start from S = initial_state[n, h] (or zero), a dv x dk
 *   matrix whose row i is value dimension i.  For each token t of the
 *   sequence, in order:
 *
 *       a_t = exp(g_t)
 *       S_t = a_t * S_{t-1} * (I - b_t k_t k_t^T) + b_t v_t k_t^T
 *       o_t = S_t q_t            (updated state; no 1/sqrt(d) scale)
 *
 *   Expanding the product once, a S (I - b k k^T) = a S - a b (S k) k^T, so
 *   the update is the rank-1 correction
 *       S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) k_t^T,
 *   which is what the loops below evaluate, row by row, in fp64.
 *
 * Source of the method: the recurrence of the Gated DeltaNet layer used in
 * the hybrid Qwen3.8-27B model; the serving pages describe it as linear
 * attention with a fixed-size state per conversation ("reactapp.top",
 * section "Exploiter l'architecture hybride": 48 of 64 layers, fp32 state of
 * about 150 MB per request) and its prefill as chunked with chunk length 64
 * ("cf-1.com", section "三个优化", item 2 "GDN prefill").  The chunking does
 * not change the exact result, so the oracle does not chunk.
 *
 * Inputs are the exact values the GPU sees (bf16 or fp32 upcast to fp64).
 * Layouts (token-major, packed over sequences):
 *   q, k          [T, Hk, dk]
 *   v, out        [T, Hv, dv]
 *   g, beta       [T, Hv]
 *   cu_seqlens    [N + 1], cu[0] = 0, nondecreasing, cu[N] = T
 *   state         [N, Hv, dv, dk]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of the recurrence for one (sequence, value head): updates the
 * dv x dk state S in place and writes o = S_t q. */
static void gdn_token_step(double *S, int64_t dk, int64_t dv,
                           const double *q, const double *k, const double *v,
                           double g, double beta, double *o)
{
    const double a = exp(g);
    for (int64_t i = 0; i < dv; ++i) {
        double *row = S + i * dk;
        /* x_i = (S_{t-1} k)_i */
        double x = 0.0;
        for (int64_t j = 0; j < dk; ++j) x += row[j] * k[j];
        /* S_t[i, :] = a S_{t-1}[i, :] + b (v_i - a x_i) k^T */
        const double u = beta * (v[i] - a * x);
        for (int64_t j = 0; j < dk; ++j) row[j] = a * row[j] + u * k[j];
        /* o_i = (S_t q)_i */
        double y = 0.0;
        for (int64_t j = 0; j < dk; ++j) y += row[j] * q[j];
        o[i] = y;
    }
}

/*
 * Prefill: runs the recurrence over every sequence for the value heads in
 * `heads` (all Hv heads when heads == NULL).  out rows of heads not listed are
 * left untouched.  final_state (nullable) receives S after each sequence's
 * last token; for a zero-length sequence it is the initial state.
 * Returns 0, or -1 on an argument error.
 */
int gdn_oracle_prefill(int64_t num_seqs, const int32_t *cu_seqlens,
                       int64_t Hk, int64_t Hv, int64_t dk, int64_t dv,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta,
                       const double *initial_state,
                       const int32_t *heads, int64_t num_heads,
                       double *out, double *final_state, int num_threads)
{
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0) return -1;
    if (Hv % Hk != 0) return -1;
    const int64_t group = Hv / Hk;
    const int64_t nh = heads ? num_heads : Hv;
    const int64_t units = num_seqs * nh;
    int rc = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int64_t n = unit / nh;
        const int64_t h = heads ? heads[unit % nh] : unit % nh;
        if (h < 0 || h >= Hv) { rc = -1; continue; }
        const int64_t hk = h / group;
        double *S = (double *)calloc((size_t)(dv * dk), sizeof(double));
        if (!S) { rc = -1; continue; }
        if (initial_state)
            memcpy(S, initial_state + (n * Hv + h) * dv * dk,
                   (size_t)(dv * dk) * sizeof(double));
        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            gdn_token_step(S, dk, dv,
                           q + (t * Hk + hk) * dk,
                           k + (t * Hk + hk) * dk,
                           v + (t * Hv + h) * dv,
                           g[t * Hv + h], beta[t * Hv + h],
                           out + (t * Hv + h) * dv);
        }
        if (final_state)
            memcpy(final_state + (n * Hv + h) * dv * dk, S,
                   (size_t)(dv * dk) * sizeof(double));
        free(S);
    }
    return rc;
}

/*
 * Decode: one token for each of num_seqs sequences, updating state in place.
 * q, k [N, Hk, dk]; v, out [N, Hv, dv]; g, beta [N, Hv]; state [N, Hv, dv, dk].
 * heads (nullable) restricts the work to the listed value heads.
 */
int gdn_oracle_decode(int64_t num_seqs, int64_t Hk, int64_t Hv,
                      int64_t dk, int64_t dv,
                      const double *q, const double *k, const double *v,
                      const double *g, const double *beta,
                      const int32_t *heads, int64_t num_heads,
                      double *state, double *out, int num_threads)
{
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0) return -1;
    if (Hv % Hk != 0) return -1;
    const int64_t group = Hv / Hk;
    const int64_t nh = heads ? num_heads : Hv;
    const int64_t units = num_seqs * nh;
    int rc = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(static)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int64_t n = unit / nh;
        const int64_t h = heads ? heads[unit % nh] : unit % nh;
        if (h < 0 || h >= Hv) { rc = -1; continue; }
        const int64_t hk = h / group;
        gdn_token_step(state + (n * Hv + h) * dv * dk, dk, dv,
                       q + (n * Hk + hk) * dk, k + (n * Hk + hk) * dk,
                       v + (n * Hv + h) * dv, g[n * Hv + h], beta[n * Hv + h],
                       out + (n * Hv + h) * dv);
    }
    return rc;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
