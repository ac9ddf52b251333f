/*
 * Attention forward oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. The CUDA path never calls it
 * and shares no code with it.
 *
 * Definition followed ("Android Transformer Optimization: Attention and Mobile
 * GPU Bottlenecks", section "The Self-Attention Bottleneck Is Memory Traffic,
 * Not Compute": S = QK^T, P = softmax(S), O = PV, with the score row written
 * out and read three times; the scale 1/sqrt(headDim) multiplies the scores,
 * as in the SGEMM alpha of "Flash Attention on Android: tiled SGEMM with
 * RenderScript", section "Architecture: tiled attention with RenderScript
 * BLAS"):
 *
 *   s_ij  = scale * sum_d q_id k_jd            for j in J(i)
 *   J(i)  = {0..N-1}, or {0..i} when causal (top-left aligned, N_q = N_k)
 *   M_i   = max_j s_ij                         (pass 1)
 *   L_i   = sum_j exp(s_ij - M_i)              (pass 2)
 *   O_id  = sum_j exp(s_ij - M_i) v_jd / L_i   (pass 3)
 *   lse_i = M_i + ln L_i                       (natural log)
 *
 * The score row of each requested query row is materialised in full before
 * the three passes. Inputs are fp64 copies of the fp16/bf16 tensors (the
 * widening is exact). Layout: q, k, v, o are dense row-major [B*H, N, D];
 * lse is [B*H, N].
 *
 * Partial results over a key range. The same definition restricted to the
 * keys j in J(i) with lo <= j < hi gives the partial result (O_i, lse_i) of
 * that range; splitting the keys into ranges and combining the partials with
 * the online-softmax update of "Android Transformer Optimization: Attention and
 * Mobile GPU Bottlenecks", section "The Essence of FlashAttention: Reordering
 * the Computation" (merge.py) gives back the full result. A range holding no
 * key of J(i) has an empty sum: lse_i = ln 0 = -inf, and O_i is set to 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * One query row (bh, i) over the keys j in J(i) with lo <= j < hi: three passes
 * over its materialised score row (entries lo..nj-1 of s_row are used).
 */
static void oracle_row(const double *q, const double *k, const double *v,
                       int64_t N, int64_t D, double scale, int causal,
                       int64_t bh, int64_t i, int64_t lo, int64_t hi,
                       double *s_row, double *o_row, double *lse_out)
{
    const double *qi = q + (bh * N + i) * D;
    const double *kh = k + bh * N * D;
    const double *vh = v + bh * N * D;
    int64_t nj = causal ? (i + 1) : N; /* J(i) = {0..nj-1} */
    if (nj > hi)
        nj = hi;
    if (lo >= nj) { /* no key: empty sum */
        for (int64_t d = 0; d < D; ++d)
            o_row[d] = 0.0;
        *lse_out = -INFINITY;
        return;
    }

    /* s_ij = scale * <q_i, k_j> */
    for (int64_t j = lo; j < nj; ++j) {
        double acc = 0.0;
        const double *kj = kh + j * D;
        for (int64_t d = 0; d < D; ++d)
            acc += qi[d] * kj[d];
        s_row[j] = scale * acc;
    }

    /* pass 1: row max */
    double m = -INFINITY;
    for (int64_t j = lo; j < nj; ++j)
        if (s_row[j] > m)
            m = s_row[j];

    /* pass 2: denominator */
    double l = 0.0;
    for (int64_t j = lo; j < nj; ++j)
        l += exp(s_row[j] - m);

    /* pass 3: weighted sum of V rows, divided by the denominator */
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = 0.0;
    for (int64_t j = lo; j < nj; ++j) {
        const double p = exp(s_row[j] - m);
        const double *vj = vh + j * D;
        for (int64_t d = 0; d < D; ++d)
            o_row[d] += p * vj[d];
    }
    for (int64_t d = 0; d < D; ++d)
        o_row[d] /= l;

    *lse_out = m + log(l);
}

/*
 * Computes the requested rows. rows[2r] = bh, rows[2r+1] = i. key_ranges is
 * NULL (all keys) or holds [lo, hi) of request r at key_ranges[2r], [2r+1].
 * Output row r of o ([nrows, D]) and lse ([nrows]) belongs to request r.
 * Returns 0 on success, -1 on a bad argument, -2 when scratch memory cannot be
 * allocated.
 */
int oracle_attention_rows_keyrange_f64(const double *q, const double *k, const double *v,
                                       int64_t BH, int64_t N, int64_t D, double scale,
                                       int causal, const int64_t *rows, int64_t nrows,
                                       const int64_t *key_ranges,
                                       double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || !rows || BH <= 0 || N <= 0 || D <= 0 || nrows < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        if (rows[2 * r] < 0 || rows[2 * r] >= BH || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= N)
            return -1;
        if (key_ranges && (key_ranges[2 * r] < 0 || key_ranges[2 * r + 1] > N ||
                           key_ranges[2 * r] > key_ranges[2 * r + 1]))
            return -1;
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
    const int nt = omp_get_max_threads();
#else
    const int nt = 1;
#endif
    /* one materialised score row per thread */
    double *scratch = (double *)malloc((size_t)nt * (size_t)N * sizeof(double));
    if (!scratch)
        return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
#ifdef _OPENMP
        double *s_row = scratch + (size_t)omp_get_thread_num() * (size_t)N;
#else
        double *s_row = scratch;
#endif
        const int64_t lo = key_ranges ? key_ranges[2 * r] : 0;
        const int64_t hi = key_ranges ? key_ranges[2 * r + 1] : N;
        oracle_row(q, k, v, N, D, scale, causal, rows[2 * r], rows[2 * r + 1], lo, hi,
                   s_row, o + r * D, lse + r);
    }
    free(scratch);
    (void)nthreads;
    return 0;
}

/* All keys of J(i) for every requested row. */
int oracle_attention_rows_f64(const double *q, const double *k, const double *v,
                              int64_t BH, int64_t N, int64_t D, double scale,
                              int causal, const int64_t *rows, int64_t nrows,
                              double *o, double *lse, int nthreads)
{
    return oracle_attention_rows_keyrange_f64(q, k, v, BH, N, D, scale, causal, rows, nrows,
                                              NULL, o, lse, nthreads);
}

/* Number of threads the parallel region uses (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
