/*
 * sdpa_oracle.c -- plain fp64 CPU reference for scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the five-step definition of attention printed on the
 * pages, taken one query row at a time so that no L x L matrix is ever held:
 *
 *   1. scores = q . k^T              ("Profiling attention in PyTorch: kernels,
 *   2. scores = scores * scale         backends and where the time goes"
 *   3. scores.masked_fill(mask, -inf)  (news.bpdata.com), section "Naiv causal
 *   4. attn = softmax(scores, -1)      attention", the NaiveCausalAttention
 *   5. out = attn . v                  module; the same module and the same
 *                                      five numbered steps appear in "PyTorch
 *                                      attention profiling: Flash, cuDNN and
 *                                      Math backends compared"
 *                                      (dev.smart-guide.co.kr), section 1)
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes):
 *   - scale defaults to 1/sqrt(head_dim) (the module's __init__ on both pages);
 *     the caller passes the value explicitly here.
 *   - mask polarity follows masked_fill: a nonzero mask byte means the key is
 *     removed (its score becomes -inf).
 *   - causal: query i sees keys j <= i (the "[seq, seq] triangular matrix" the
 *     math backend rebuilds each call, same two pages, math-backend sections).
 *     Query and key lengths are equal, so no alignment question arises.
 *   - safe softmax: a row whose scores are all -inf yields zeros, not NaN (the
 *     _safe_softmax step of the math backend, same sections).  This is the one
 *     place where the oracle deliberately departs from the naive module, which
 *     would produce NaN.
 *   - everything is fp64; inputs arrive already rounded to the 16-bit input
 *     type and widened exactly to double.
 *
 * Layout: q, k, v, out are dense row-major [B, H, L, D] doubles; mask, when
 * not NULL, is a dense row-major [L, L] byte matrix shared by every (b, h).
 * lse, when not NULL, receives per row the log-sum-exp of the scaled,
 * masked scores (the log of the softmax denominator; -inf for a row with no
 * admissible key) -- the second output of the fused forward that the
 * FlashInfer pull-request page shows as `out, lse = fwd(...)`.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row i of one (b, h): the five steps, in order.
 * s is caller-provided scratch of length L. */
static void attend_one_row(const double *qi, const double *K, const double *V,
                           int64_t L, int64_t D, int64_t i,
                           const uint8_t *mask_row, int is_causal, double scale,
                           double *s, double *out_row, double *lse)
{
    int64_t j, d;

    /* step 1: scores[j] = q_i . k_j */
    for (j = 0; j < L; ++j) {
        const double *kj = K + j * D;
        double acc = 0.0;
        for (d = 0; d < D; ++d)
            acc += qi[d] * kj[d];
        s[j] = acc;
    }

    /* step 2: scores *= scale */
    for (j = 0; j < L; ++j)
        s[j] = s[j] * scale;

    /* step 3: masked_fill(mask, -inf); the causal triangle removes j > i */
    for (j = 0; j < L; ++j) {
        int removed = 0;
        if (is_causal && j > i)
            removed = 1;
        if (mask_row != NULL && mask_row[j] != 0)
            removed = 1;
        if (removed)
            s[j] = -INFINITY;
    }

    /* step 4: softmax over the key axis, NaN-safe for an all -inf row */
    double m = -INFINITY;
    for (j = 0; j < L; ++j)
        if (s[j] > m)
            m = s[j];
    if (m == -INFINITY) {
        /* every key removed: the safe softmax gives a zero row */
        for (j = 0; j < L; ++j)
            s[j] = 0.0;
        if (lse)
            *lse = -INFINITY; /* log of an empty sum */
    } else {
        double total = 0.0;
        for (j = 0; j < L; ++j) {
            s[j] = exp(s[j] - m);
            total += s[j];
        }
        for (j = 0; j < L; ++j)
            s[j] = s[j] / total;
        /* log-sum-exp of the scaled, masked scores: the softmax denominator
         * in log form, log(sum_j exp(s_j)) = m + log(sum_j exp(s_j - m)) */
        if (lse)
            *lse = m + log(total);
    }

    /* step 5: out_i = attn_i . V */
    for (d = 0; d < D; ++d)
        out_row[d] = 0.0;
    for (j = 0; j < L; ++j) {
        const double p = s[j];
        const double *vj = V + j * D;
        for (d = 0; d < D; ++d)
            out_row[d] += p * vj[d];
    }
}

/* Whole tensor: out[b, h, i, :] for every b, h, i.  Returns 0, or -1 on a bad
 * argument or an allocation failure. */
int oracle_sdpa_fp64(const double *q, const double *k, const double *v,
                     double *out, int64_t B, int64_t H, int64_t L, int64_t D,
                     const uint8_t *mask, int is_causal, double scale,
                     double *lse)
{
    if (!q || !k || !v || !out || B < 0 || H < 0 || L < 0 || D < 1)
        return -1;
    const int64_t rows = B * H * L;
    int failed = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (s == NULL) {
#pragma omp atomic write
            failed = 1;
        } else {
            int64_t r;
#pragma omp for schedule(dynamic, 16)
            for (r = 0; r < rows; ++r) {
                const int64_t bh = r / L, i = r % L;
                const double *Q = q + bh * L * D, *K = k + bh * L * D,
                             *V = v + bh * L * D;
                attend_one_row(Q + i * D, K, V, L, D, i,
                               mask ? mask + i * L : NULL, is_causal, scale, s,
                               out + r * D, lse ? lse + r : NULL);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/* Selected rows only: idx holds n triples (b, h, i); row t of out_rows (n x D)
 * receives out[b, h, i, :].  Lets full-size workloads be checked on a sample. */
int oracle_sdpa_rows_fp64(const double *q, const double *k, const double *v,
                          int64_t B, int64_t H, int64_t L, int64_t D,
                          const uint8_t *mask, int is_causal, double scale,
                          const int64_t *idx, int64_t n, double *out_rows,
                          double *lse_rows)
{
    if (!q || !k || !v || !idx || !out_rows || L < 1 || D < 1)
        return -1;
    int failed = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        if (s == NULL) {
#pragma omp atomic write
            failed = 1;
        } else {
            int64_t t;
#pragma omp for schedule(dynamic, 1)
            for (t = 0; t < n; ++t) {
                const int64_t b = idx[3 * t], h = idx[3 * t + 1],
                              i = idx[3 * t + 2];
                if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= L) {
#pragma omp atomic write
                    failed = 1;
                    continue;
                }
                const int64_t bh = b * H + h;
                attend_one_row(q + (bh * L + i) * D, k + bh * L * D,
                               v + bh * L * D, L, D, i,
                               mask ? mask + i * L : NULL, is_causal, scale, s,
                               out_rows + t * D, lse_rows ? lse_rows + t : NULL);
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/* Threads the parallel regions above will use (reported beside CPU timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
