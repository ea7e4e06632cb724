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
 * The producer step (oracle_producer) restates what the model does before the two GEMMs
 * (page 1, snippet `sana_video.py`): ReLU on the normalised Q and K, interleaved RoPE on
 * the activated copies (only the rotated copies feed the GEMMs), and the normaliser from
 * the un-rotated activated copies:
 *       qa = relu(q), ka = relu(k)
 *       (y0, y1) of pair p of token n = (x0 c - x1 s, x0 s + x1 c), c = cos[n][p], s = sin[n][p]
 *       den[h][n] = sum_i qa[h][n][i] * (sum_m ka[h][m][i]) + eps
 * The rotation is fixed to IEEE binary32 operations in this order (each product and the
 * sum rounded to nearest), then rounded once to BF16 (nearest, ties to even), so that any
 * implementation following the same definition gets the same BF16 operands bit for bit.
 *
 * The softmax anchor layer (oracle_softmax_attention_rows) follows the page "[sglang]
 * SANA-Video 2.0 anchor attention의 FP32 upcast 제거로 720p 생성 52% 단축하기" (PR #49219),
 * section 코드 분석, 2. GatedSoftmaxAttention: F.scaled_dot_product_attention(q, k, v,
 * dropout_p=0.0) on [B, H, N, D] tensors - no mask, no dropout, default scale 1/sqrt(D):
 *       out[h][n][j] = sum_m w_m v[h][m][j] / sum_m w_m,   w_m = exp(s_m - max_m s_m),
 *       s_m = scale * sum_i q[h][n][i] k[h][m][i]
 *
 * Arithmetic: every input value (BF16 bit patterns, FP32 denominators) is exact
 * in FP64; products and sums are FP64 in the order written (m ascending for KV,
 * i ascending for the apply).  Build with -ffp-contract=off and no fast-math so
 * the order stays as written.  Loops over independent outputs are split across
 * OpenMP threads; no output's arithmetic depends on the split.
 */
#include <math.h>
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

/* IEEE binary32 -> BF16, round to nearest, ties to even (NaN stays a quiet NaN). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Round an array of binary32 values to BF16 bit patterns (tests pin the rounding). */
void oracle_f32_to_bf16(int64_t count, const float *in, uint16_t *out)
{
    for (int64_t e = 0; e < count; ++e)
        out[e] = f32_to_bf16_rne(in[e]);
}

/*
 * Producer step: q, k are the BF16 bits of the normalised projections [H][N][D] (before
 * ReLU), cos_t / sin_t the FP32 rotation tables [N][D/2].  Writes the BF16 bits of the
 * rotated activated copies q_rot, k_rot [H][N][D] and the FP64 denominators den [H][N].
 */
int oracle_producer(int64_t H, int64_t N, int64_t D, const uint16_t *q, const uint16_t *k, const float *cos_t,
                    const float *sin_t, double eps, uint16_t *q_rot, uint16_t *k_rot, double *den)
{
    if (H < 0 || N < 0 || D < 2 || D % 2 || !q || !k || !cos_t || !sin_t || !q_rot || !k_rot || !den)
        return 1;
    const int64_t P = D / 2;
    int64_t h;
#pragma omp parallel for schedule(dynamic, 1)
    for (h = 0; h < H; ++h) {
        double *ksum = (double *)calloc((size_t)D, sizeof(double));
        for (int64_t n = 0; n < N; ++n) {
            const int64_t row = (h * N + n) * D;
            for (int64_t i = 0; i < D; ++i) {
                const double ka = bf16_to_f64(k[row + i]);
                ksum[i] += ka > 0.0 ? ka : 0.0;
            }
        }
        for (int64_t n = 0; n < N; ++n) {
            const int64_t row = (h * N + n) * D;
            double dot = 0.0;
            for (int64_t i = 0; i < D; ++i) {
                const double qa = bf16_to_f64(q[row + i]);
                dot += (qa > 0.0 ? qa : 0.0) * ksum[i];
            }
            den[h * N + n] = dot + eps;
            for (int64_t p = 0; p < P; ++p) {
                const float c = cos_t[n * P + p], s = sin_t[n * P + p];
                for (int which = 0; which < 2; ++which) {
                    const uint16_t *src = which ? k : q;
                    uint16_t *dst = which ? k_rot : q_rot;
                    float x0 = (float)bf16_to_f64(src[row + 2 * p]);
                    float x1 = (float)bf16_to_f64(src[row + 2 * p + 1]);
                    x0 = x0 > 0.0f ? x0 : 0.0f;
                    x1 = x1 > 0.0f ? x1 : 0.0f;
                    const float a0 = x0 * c, b0 = x1 * s;
                    const float a1 = x0 * s, b1 = x1 * c;
                    dst[row + 2 * p] = f32_to_bf16_rne(a0 - b0);
                    dst[row + 2 * p + 1] = f32_to_bf16_rne(a1 + b1);
                }
            }
        }
        free(ksum);
    }
    return 0;
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

/*
 * The same second GEMM and normalisation with FP64 denominators, as the producer step
 * forms them (oracle_producer writes den in FP64; page 1, snippet `sana_video.py`, divides
 * the second product by the normaliser built from the un-rotated ReLU'd Q and K):
 *   out[r][j] = (sum over i = 0..D-1 (ascending) of Q[row_r][i] * KV[h_r][i][j]) / den64[row_r]
 * Arguments as oracle_apply_rows, except den64: FP64 [H][N].
 */
int oracle_apply_rows_f64den(int64_t H, int64_t N, int64_t D, const uint16_t *q, const double *kv,
                             const double *den64, int64_t n_rows, const int64_t *rows, double *out)
{
    if (H < 0 || N < 0 || D < 1 || !q || !kv || !den64 || !out || n_rows < 0)
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
        const double dd = den64[flat];
        for (int64_t j = 0; j < D; ++j) {
            double s = 0.0;
            for (int64_t i = 0; i < D; ++i)
                s += bf16_to_f64(qrow[i]) * kvh[i * D + j];
            out[r * D + j] = s / dd;
        }
    }
    return bad;
}

/*
 * Softmax attention for selected rows: rows[r] = h*N + n (rows == NULL: all H*N in order).
 * q, k, v: BF16 bits [H][N][D]; out: FP64 [n_rows][D].  Scores, weights and sums in FP64,
 * keys m ascending.
 */
int oracle_softmax_attention_rows(int64_t H, int64_t N, int64_t D, const uint16_t *q, const uint16_t *k,
                                  const uint16_t *v, double scale, int64_t n_rows, const int64_t *rows, double *out)
{
    if (H < 0 || N < 1 || D < 1 || !q || !k || !v || !out || n_rows < 0)
        return 1;
    if (!rows && n_rows != H * N)
        return 1;
    int bad = 0;
    int64_t r;
#pragma omp parallel reduction(| : bad)
    {
        double *s = (double *)malloc((size_t)N * sizeof(double));
        double *qd = (double *)malloc((size_t)D * sizeof(double));
        if (!s || !qd)
            bad |= 2;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            const int64_t flat = rows ? rows[r] : r;
            if (!s || !qd || flat < 0 || flat >= H * N) {
                bad |= 1;
                continue;
            }
            const int64_t h = flat / N;
            for (int64_t i = 0; i < D; ++i)
                qd[i] = bf16_to_f64(q[flat * D + i]);
            double smax = -INFINITY;
            for (int64_t m = 0; m < N; ++m) {
                const uint16_t *krow = k + (h * N + m) * D;
                double dot = 0.0;
                for (int64_t i = 0; i < D; ++i)
                    dot += qd[i] * bf16_to_f64(krow[i]);
                s[m] = scale * dot;
                if (s[m] > smax)
                    smax = s[m];
            }
            double wsum = 0.0;
            for (int64_t m = 0; m < N; ++m) {
                s[m] = exp(s[m] - smax);
                wsum += s[m];
            }
            double *dst = out + r * D;
            for (int64_t j = 0; j < D; ++j)
                dst[j] = 0.0;
            for (int64_t m = 0; m < N; ++m) {
                const uint16_t *vrow = v + (h * N + m) * D;
                for (int64_t j = 0; j < D; ++j)
                    dst[j] += s[m] * bf16_to_f64(vrow[j]);
            }
            for (int64_t j = 0; j < D; ++j)
                dst[j] /= wsum;
        }
        free(s);
        free(qd);
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
