/*
 * sse_oracle.c -- plain fp64 CPU oracle of the Sparse State Expansion (SSE)
 * layer.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's
 * CPU-baseline leg call it; the CUDA library never does, and the two share no
 * code, header, table or helper.
 *
 * What it computes ("Scaling Linear Attention with Sparse State Expansion",
 * close-reading notes, section 2.3, equations 9-14; shared partition from
 * section 2.5), per sequence b and head h, in time order, in float64:
 *
 *   e_t   = softmax over the N router logits of token t            (eq. 9)
 *   T_t   = the k partitions with the largest logits; equal logits
 *           are ordered by ascending partition index               (eq. 10)
 *   a_t   = exp(g_t)  -- the diagonal of the gate Lambda_t, one entry
 *           per key row (GLA-style diagonal decay, section 2.1 eq. 6)
 *   for i in T_t:  S_i <- diag(a_t) S_i + e_t[i] * k_t^T v_t          (eq. 13)
 *   for i not in T_t: S_i unchanged (neither decays nor is written)
 *   shared slot N (always active, weight 1, same gate; section 2.5):
 *                  S_N <- diag(a_t) S_N + ks_t^T v_t
 *   o_t   = sum_{i in T_t} e_t[i] * (scale q_t) S_i + (scale qs_t) S_N  (eq. 14)
 *
 * The read uses the states after the update of step t.  The weights e_t are
 * the full-N softmax values (not renormalised over the selected k), so their
 * sum over T_t is at most 1 (section 2.3, the classification-strength
 * identity).  The key k_t is taken as given: the caller applies the key
 * softmax of eq. 12.
 *
 * A decode step is one iteration of the loop body on a resident state
 * (section 2.6: decoding recurs only on the selected states).
 *
 * Layouts (row-major, contiguous):
 *   q, k, g, qs, ks : [T, H, c]      v, out : [T, H, d]   logits : [T, H, N]
 *   states          : [S, H, P, c, d] with P = N + use_shared, slot N = shared
 *   topk_idx/topk_w : [T, H, k]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_N 256

typedef struct {
    int32_t H, c, d, N, k, use_shared;
    double scale;
} oracle_dims;

/* eq. 9-10: softmax over the N logits and the k largest logits (ties to the
 * lower index), returned in descending-logit order. */
static void route_token(const double *logit, int N, int k, double *e, int32_t *idx)
{
    double m = logit[0];
    for (int i = 1; i < N; ++i)
        if (logit[i] > m) m = logit[i];
    double s = 0.0;
    for (int i = 0; i < N; ++i) {
        e[i] = exp(logit[i] - m);
        s += e[i];
    }
    for (int i = 0; i < N; ++i) e[i] /= s;

    unsigned char taken[ORACLE_MAX_N];
    memset(taken, 0, (size_t)N);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int i = 0; i < N; ++i) {
            if (taken[i]) continue;
            if (best < 0 || logit[i] > logit[best]) best = i; /* strict: keeps lower index */
        }
        taken[best] = 1;
        idx[j] = best;
    }
}

/* One token of one (sequence, head): route, update the selected states and
 * the shared state, read out.  S points at the P = N + use_shared states of
 * this (sequence, head), each c x d. */
static void step_token(const oracle_dims *D, double *S,
                       const double *q, const double *kk, const double *v,
                       const double *g, const double *logit,
                       const double *qs, const double *ks,
                       double *out, int32_t *idx_out, double *w_out,
                       double *e, double *a)
{
    const int c = D->c, d = D->d, N = D->N, k = D->k;
    int32_t idx[ORACLE_MAX_N];
    route_token(logit, N, k, e, idx);
    for (int r = 0; r < c; ++r) a[r] = exp(g[r]);

    /* eq. 13: selected partitions decay then receive the e-weighted write */
    for (int j = 0; j < k; ++j) {
        const int i = idx[j];
        double *Si = S + (size_t)i * c * d;
        for (int r = 0; r < c; ++r)
            for (int col = 0; col < d; ++col)
                Si[(size_t)r * d + col] = a[r] * Si[(size_t)r * d + col] + e[i] * kk[r] * v[col];
    }
    /* shared partition: every step, weight 1 */
    if (D->use_shared) {
        double *Sn = S + (size_t)N * c * d;
        for (int r = 0; r < c; ++r)
            for (int col = 0; col < d; ++col)
                Sn[(size_t)r * d + col] = a[r] * Sn[(size_t)r * d + col] + ks[r] * v[col];
    }
    /* eq. 14 (+ shared read): gated sum of q S over the selected states */
    for (int col = 0; col < d; ++col) out[col] = 0.0;
    for (int j = 0; j < k; ++j) {
        const int i = idx[j];
        const double *Si = S + (size_t)i * c * d;
        for (int r = 0; r < c; ++r) {
            const double w = e[i] * D->scale * q[r];
            for (int col = 0; col < d; ++col) out[col] += w * Si[(size_t)r * d + col];
        }
    }
    if (D->use_shared) {
        const double *Sn = S + (size_t)N * c * d;
        for (int r = 0; r < c; ++r) {
            const double w = D->scale * qs[r];
            for (int col = 0; col < d; ++col) out[col] += w * Sn[(size_t)r * d + col];
        }
    }
    if (idx_out)
        for (int j = 0; j < k; ++j) idx_out[j] = idx[j];
    if (w_out)
        for (int j = 0; j < k; ++j) w_out[j] = e[idx[j]];
}

int sse_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over packed varlen sequences.  pair_list (optional) restricts the
 * work to the listed (b * H + h) pairs; outputs of other pairs are left
 * untouched.  Returns the number of threads used, or -1 on bad arguments. */
int sse_oracle_forward(int64_t total_tokens, int32_t H, int32_t c, int32_t d,
                       int32_t N, int32_t k, int32_t use_shared, double scale,
                       const double *q, const double *kk, const double *v,
                       const double *g, const double *logits,
                       const double *q_shared, const double *k_shared,
                       const int64_t *cu_seqlens, int32_t num_seqs,
                       const double *initial_state, double *final_state,
                       double *out, int32_t *topk_idx, double *topk_w,
                       const int64_t *pair_list, int64_t num_pairs)
{
    if (N < 1 || N > ORACLE_MAX_N || k < 1 || k > N || c < 1 || d < 1 || H < 1)
        return -1;
    if (cu_seqlens[num_seqs] != total_tokens) return -1;
    const oracle_dims D = {H, c, d, N, k, use_shared, scale};
    const int P = N + (use_shared ? 1 : 0);
    const size_t state_sz = (size_t)P * c * d;
    const double *qs_base = q_shared ? q_shared : q;
    const double *ks_base = k_shared ? k_shared : kk;
    const int64_t npairs = pair_list ? num_pairs : (int64_t)num_seqs * H;
    int nthreads = 1;

#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        nthreads = omp_get_num_threads();
#endif
        double *S = (double *)malloc(state_sz * sizeof(double));
        double e[ORACLE_MAX_N];
        double *a = (double *)malloc((size_t)c * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < npairs; ++p) {
            const int64_t bh = pair_list ? pair_list[p] : p;
            const int b = (int)(bh / H), h = (int)(bh % H);
            if (initial_state)
                memcpy(S, initial_state + (size_t)bh * state_sz, state_sz * sizeof(double));
            else
                memset(S, 0, state_sz * sizeof(double));
            for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
                const size_t th = (size_t)t * H + h;
                step_token(&D, S, q + th * c, kk + th * c, v + th * d, g + th * c,
                           logits + th * N, qs_base + th * c, ks_base + th * c,
                           out + th * d, topk_idx ? topk_idx + th * k : NULL,
                           topk_w ? topk_w + th * k : NULL, e, a);
            }
            if (final_state)
                memcpy(final_state + (size_t)bh * state_sz, S, state_sz * sizeof(double));
        }
        free(a);
        free(S);
    }
    return nthreads;
}

/* One decode step on resident states [B, H, P, c, d] (updated in place);
 * token inputs are [B, H, .].  Returns threads used, -1 on bad arguments. */
int sse_oracle_decode_step(int32_t B, int32_t H, int32_t c, int32_t d, int32_t N,
                           int32_t k, int32_t use_shared, double scale,
                           const double *q, const double *kk, const double *v,
                           const double *g, const double *logits,
                           const double *q_shared, const double *k_shared,
                           double *state, double *out, int32_t *topk_idx, double *topk_w,
                           const int64_t *pair_list, int64_t num_pairs)
{
    if (N < 1 || N > ORACLE_MAX_N || k < 1 || k > N || c < 1 || d < 1 || H < 1)
        return -1;
    const oracle_dims D = {H, c, d, N, k, use_shared, scale};
    const int P = N + (use_shared ? 1 : 0);
    const size_t state_sz = (size_t)P * c * d;
    const double *qs_base = q_shared ? q_shared : q;
    const double *ks_base = k_shared ? k_shared : kk;
    const int64_t npairs = pair_list ? num_pairs : (int64_t)B * H;
    int nthreads = 1;
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        nthreads = omp_get_num_threads();
#endif
        double e[ORACLE_MAX_N];
        double *a = (double *)malloc((size_t)c * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t p = 0; p < npairs; ++p) {
            const int64_t bh = pair_list ? pair_list[p] : p;
            step_token(&D, state + (size_t)bh * state_sz, q + bh * c, kk + bh * c,
                       v + bh * d, g + bh * c, logits + bh * N, qs_base + bh * c,
                       ks_base + bh * c, out + bh * d,
                       topk_idx ? topk_idx + bh * k : NULL,
                       topk_w ? topk_w + bh * k : NULL, e, a);
        }
        free(a);
    }
    return nthreads;
}

/* Token -> partition grouping (section 2.6, varlen schedule): segment
 * s = (b * H + h) * N + i lists, in ascending time, the tokens t of sequence b
 * whose selected set for head h contains i.  seg_off[s] is the start of
 * segment s in perm (exclusive prefix over s), seg_off[S*H*N] the total. */
int sse_oracle_group(int64_t total_tokens, int32_t H, int32_t N, int32_t k,
                     const int32_t *topk_idx, const int64_t *cu_seqlens, int32_t num_seqs,
                     int64_t *seg_off, int64_t *perm)
{
    (void)total_tokens;
    int64_t pos = 0;
    for (int b = 0; b < num_seqs; ++b)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < N; ++i) {
                seg_off[((int64_t)b * H + h) * N + i] = pos;
                for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
                    const int32_t *sel = topk_idx + ((size_t)t * H + h) * k;
                    for (int j = 0; j < k; ++j)
                        if (sel[j] == i) {
                            perm[pos++] = t;
                            break;
                        }
                }
            }
    seg_off[(int64_t)num_seqs * H * N] = pos;
    return 0;
}
