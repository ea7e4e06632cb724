/*
 * FP64 CPU oracle for SANA-Video linear attention over rotated queries and keys.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the bench's CPU-baseline leg load this library.  The product (the CUDA
 * library) never calls it and shares no code, header or table with it.
 *
 * What it computes follows the page "PR #35728 完整报告 - [diffusion]
 * Accelerate SANA-Video linear attention in quality=high", section
 * 关键源码片段:
 *   - snippet `sana_video_linear_attention_site.py`, try_sana_video_linear_attention:
 *       scores = bmm(value, key_rotate^T)       (first GEMM, a D x D matrix per head)
 *       out    = (scores @ query_rotate) * normalizer
 *   - snippet `sana_video.py`, the FP32 fallback chain of forward(), same maths.
 * The pages keep tensors as [B, H, D, N] views; with contiguous [1, H, N, D]
 * storage the same quantities read
 *       KV[h][i][j]  = sum_m K_rot[h][m][i] * V[h][m][j]          (= scores^T)
 *       out[h][n][j] = (sum_i Q_rot[h][n][i] * KV[h][i][j]) / den[h][n]
 * where den is the denominator of the layer's normalizer (the layer divides by it).
 * Both quality tiers ('high', 'lossless') have this same exact target: they differ
 * only in rounding, so the oracle has no mode.
 *
 * Arithmetic: every input value (BF16 bit patterns, FP32 denominators) is exact
 * in FP64; products and sums are FP64 in the order written (m ascending for KV,
 * i ascending for the apply).  Build with -ffp-contract=off and no fast-math so
 * the order stays as written.  Loops over independent outputs are split across
 * OpenMP threads; no output's arithmetic depends on the split.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* BF16 is the top 16 bits of an IEEE binary32. */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Decode an array of BF16 bit patterns (used by tests to pin the decoding). */
void oracle_bf16_decode(int64_t count, const uint16_t *bits, double *out)
{
    for (int64_t e = 0; e < count; ++e)
        out[e] = bf16_to_f64(bits[e]);
}

/*
 * First GEMM: KV[h][i][j] = sum over m = 0..N-1 (ascending) of K[h][m][i] * V[h][m][j].
 * k, v: BF16 bits, [H][N][D].  kv: FP64 [H][D][D].
 */
int oracle_kv(int64_t H, int64_t N, int64_t D, const uint16_t *k, const uint16_t *v, double *kv)
{
    if (H < 0 || N < 0 || D < 1 || !k || !v || !kv)
        return 1;
    const int64_t rows_per_task = 8;
    const int64_t tasks_per_head = (D + rows_per_task - 1) / rows_per_task;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < H * tasks_per_head; ++t) {
        const int64_t h = t / tasks_per_head;
        const int64_t i0 = (t % tasks_per_head) * rows_per_task;
        const int64_t i1 = (i0 + rows_per_task < D) ? i0 + rows_per_task : D;
        double *acc = kv + (h * D + i0) * D;
        for (int64_t e = 0; e < (i1 - i0) * D; ++e)
            acc[e] = 0.0;
        for (int64_t m = 0; m < N; ++m) {
            const uint16_t *krow = k + (h * N + m) * D;
            const uint16_t *vrow = v + (h * N + m) * D;
            for (int64_t i = i0; i < i1; ++i) {
                const double a = bf16_to_f64(krow[i]);
                double *dst = acc + (i - i0) * D;
                for (int64_t j = 0; j < D; ++j)
                    dst[j] += a * bf16_to_f64(vrow[j]);
            }
        }
    }
    return 0;
}

/*
 * Second GEMM and normalisation for selected rows:
 *   out[r][j] = (sum over i = 0..D-1 (ascending) of Q[row_r][i] * KV[h_r][i][j]) / den[row_r]
 * rows[r] is a flat token index h*N + n (rows == NULL means all H*N rows in order).
 * q: BF16 bits [H][N][D]; kv: FP64 [H][D][D]; den: FP32 [H][N]; out: FP64 [n_rows][D].
 */
int oracle_apply_rows(int64_t H, int64_t N, int64_t D, const uint16_t *q, const double *kv,
                      const float *den, int64_t n_rows, const int64_t *rows, double *out)
{
    if (H < 0 || N < 0 || D < 1 || !q || !kv || !den || !out || n_rows < 0)
        return 1;
    if (!rows && n_rows != H * N)
        return 1;
    int bad = 0;
    int64_t r;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (r = 0; r < n_rows; ++r) {
        const int64_t flat = rows ? rows[r] : r;
        if (flat < 0 || flat >= H * N) {
            bad |= 1;
            continue;
        }
        const int64_t h = flat / N;
        const uint16_t *qrow = q + flat * D;
        const double *kvh = kv + h * D * D;
        const double d = (double)den[flat];
        for (int64_t j = 0; j < D; ++j) {
            double s = 0.0;
            for (int64_t i = 0; i < D; ++i)
                s += bf16_to_f64(qrow[i]) * kvh[i * D + j];
            out[r * D + j] = s / d;
        }
    }
    return bad;
}

/* The whole layer: KV for every head, then every output row.  out: FP64 [H][N][D]. */
int oracle_forward(int64_t H, int64_t N, int64_t D, const uint16_t *q, const uint16_t *k,
                   const uint16_t *v, const float *den, double *out)
{
    if (H < 0 || N < 0 || D < 1)
        return 1;
    double *kv = (double *)malloc((size_t)(H > 0 ? H : 1) * (size_t)D * (size_t)D * sizeof(double));
    if (!kv)
        return 2;
    int rc = oracle_kv(H, N, D, k, v, kv);
    if (rc == 0)
        rc = oracle_apply_rows(H, N, D, q, kv, den, H * N, NULL, out);
    free(kv);
    return rc;
}
