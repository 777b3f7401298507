/*
 * fp64 CPU oracle for the causal attention score product and the ragged
 * dense layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or constant with
 * the CUDA library; the two meet only at the seeded input generators.
 *
 * Every function below is the plain definition written out, in fp64, over
 * inputs that are already bf16 (passed as their raw 16-bit patterns, so the
 * widening to double is exact). No blocking, no reordering, no fusion.
 *
 * Sources (the pages these definitions are read from):
 *  - "llm.c dev/cuda/trimat_forward.cu", the CPU referee `trimul_cpu`
 *    (Chapter I): input (B, T, 3, NH, HS), output (B, NH, T, T);
 *    out[b][nh][t][t2] = (Q[b][nh][t][:] . K[b][nh][t2][:]) * 1/sqrt(HS) for
 *    t2 <= t, and the causal mask value for t2 > t.
 *  - "DietCode tests/codegen/test_1_local_padding.py", test_local_padding
 *    docstring, the dense workload: Y[i, j] += X[i, k] * W[j, k], i.e.
 *    Y = X W^T with X [B*T, I], W [H, I], Y [B*T, H].
 *  - "Smallem" article 5 (kernels-gpu), its two-pass softmax: per row the
 *    maximum m and the sum of exp(x - m), then exp(x - m) / sum; applied to
 *    the causal scores of trimul_cpu (whose comment says it is taken from the
 *    attention forward pass, where a softmax over t2 <= t follows), masked
 *    positions t2 > t get probability 0.
 *  - "llm.c dev/cuda/trimat_forward.cu" again for fp32 inputs: the referee
 *    takes `const float* inp`, and `main` fills it with fp32 random numbers;
 *    oracle_trimul_f32 is the same definition over fp32 inputs, with no
 *    rounding of the inputs at all (fp32 widens to double exactly).
 *  - the same file, test_local_padding_ii docstring, the batched NT workload:
 *    Y[i, j, k] += X[i, j, l] * W[i, k, l] with X [B*NH, T, H/NH],
 *    W [B*NH, T, H/NH], Y [B*NH, T, T] (the unmasked, unscaled score product;
 *    the docstring prints X's last dimension as H/A, read here as H/NH).
 *
 * Readings taken where the pages leave a step open:
 *  - The score is divided by sqrt(HS) in fp64 (the definition), where the
 *    page multiplies an fp32 sum by an fp32 1/sqrtf(HS).
 *  - The masked value is written as a double NaN or -inf, chosen by the
 *    caller; the page writes NAN and remarks that -inf would also do.
 *  - HS = C / NH with C % NH == 0 (the page uses integer division; other
 *    shapes are rejected).
 *
 * Parity pins for each function live in the test-suite (exact rational brute
 * force, library fp64 matmul identity, closed forms, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exactly: a bf16 is the upper half of an fp32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
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

/*
 * One score row: out[b][h][t][0..T-1] of the trimat_forward referee.
 * Q[b][h][t][d] = qkv[b][t][0][h][d] and K[b][h][t2][d] = qkv[b][t2][1][h][d]
 * in the packed (B, T, 3, NH, HS) layout, so the key of head h sits C
 * elements after its query within the same (b, t) row of 3*C elements.
 */
static void score_row(double *dst, const uint16_t *qkv, int64_t T, int64_t C,
                      int64_t NH, int64_t b, int64_t h, int64_t t, double mask)
{
    const int64_t HS = C / NH;
    const int64_t C3 = 3 * C;
    const uint16_t *query = qkv + b * T * C3 + t * C3 + h * HS;
    const double root_hs = sqrt((double)HS);

    for (int64_t t2 = 0; t2 <= t; t2++) {
        const uint16_t *key = qkv + b * T * C3 + t2 * C3 + h * HS + C;
        double acc = 0.0;
        for (int64_t d = 0; d < HS; d++)
            acc += bf16_to_double(query[d]) * bf16_to_double(key[d]);
        dst[t2] = acc / root_hs;
    }
    for (int64_t t2 = t + 1; t2 < T; t2++)
        dst[t2] = mask;
}

static double mask_value(int mask_kind)
{
    return mask_kind == 1 ? -INFINITY : NAN;
}

static int check_trimul_shape(int64_t B, int64_t T, int64_t C, int64_t NH)
{
    if (B <= 0 || T <= 0 || C <= 0 || NH <= 0 || C % NH != 0)
        return -2;
    return 0;
}

/*
 * Full causal score tensor, (B, NH, T, T) doubles.
 * mask_kind: 0 -> NaN above the diagonal, 1 -> -inf.
 * Returns 0, or -2 for an invalid shape.
 */
int oracle_trimul(double *out, const uint16_t *qkv, int64_t B, int64_t T,
                  int64_t C, int64_t NH, int mask_kind)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    const double mask = mask_value(mask_kind);
    const int64_t rows = B * NH * T;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; r++) {
        const int64_t t = r % T;
        const int64_t h = (r / T) % NH;
        const int64_t b = r / (T * NH);
        score_row(out + r * T, qkv, T, C, NH, b, h, t, mask);
    }
    return 0;
}

/*
 * Selected score rows: for each of the n triples (b, h, t) in bht, writes the
 * T doubles of out[b][h][t][:] to out + i*T. Lets a full-size problem be
 * checked on sampled rows without materialising the whole tensor.
 */
int oracle_trimul_rows(double *out, const uint16_t *qkv, int64_t B, int64_t T,
                       int64_t C, int64_t NH, const int64_t *bht, int64_t n,
                       int mask_kind)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    for (int64_t i = 0; i < n; i++) {
        const int64_t b = bht[3 * i], h = bht[3 * i + 1], t = bht[3 * i + 2];
        if (b < 0 || b >= B || h < 0 || h >= NH || t < 0 || t >= T)
            return -2;
    }
    const double mask = mask_value(mask_kind);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n; i++)
        score_row(out + i * T, qkv, T, C, NH, bht[3 * i], bht[3 * i + 1],
                  bht[3 * i + 2], mask);
    return 0;
}

/*
 * The same score row over fp32 inputs (the referee's own input type):
 * out[b][h][t][0..T-1] with Q at qkv[b][t][0][h][:] and K at qkv[b][t2][1][h][:].
 */
static void score_row_f32(double *dst, const float *qkv, int64_t T, int64_t C,
                          int64_t NH, int64_t b, int64_t h, int64_t t, double mask)
{
    const int64_t HS = C / NH;
    const int64_t C3 = 3 * C;
    const float *query = qkv + b * T * C3 + t * C3 + h * HS;
    const double root_hs = sqrt((double)HS);

    for (int64_t t2 = 0; t2 <= t; t2++) {
        const float *key = qkv + b * T * C3 + t2 * C3 + h * HS + C;
        double acc = 0.0;
        for (int64_t d = 0; d < HS; d++)
            acc += (double)query[d] * (double)key[d];
        dst[t2] = acc / root_hs;
    }
    for (int64_t t2 = t + 1; t2 < T; t2++)
        dst[t2] = mask;
}

/* Full causal score tensor of fp32 inputs, (B, NH, T, T) doubles. */
int oracle_trimul_f32(double *out, const float *qkv, int64_t B, int64_t T,
                      int64_t C, int64_t NH, int mask_kind)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    const double mask = mask_value(mask_kind);
    const int64_t rows = B * NH * T;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; r++) {
        const int64_t t = r % T;
        const int64_t h = (r / T) % NH;
        const int64_t b = r / (T * NH);
        score_row_f32(out + r * T, qkv, T, C, NH, b, h, t, mask);
    }
    return 0;
}

/* Selected rows (b, h, t) of the fp32-input score tensor, n x T doubles. */
int oracle_trimul_f32_rows(double *out, const float *qkv, int64_t B, int64_t T,
                           int64_t C, int64_t NH, const int64_t *bht, int64_t n,
                           int mask_kind)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    for (int64_t i = 0; i < n; i++) {
        const int64_t b = bht[3 * i], h = bht[3 * i + 1], t = bht[3 * i + 2];
        if (b < 0 || b >= B || h < 0 || h >= NH || t < 0 || t >= T)
            return -2;
    }
    const double mask = mask_value(mask_kind);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n; i++)
        score_row_f32(out + i * T, qkv, T, C, NH, bht[3 * i], bht[3 * i + 1],
                      bht[3 * i + 2], mask);
    return 0;
}

/* One output row of the dense workload: Y[i][j] = sum_k X[i][k] * W[j][k]. */
static void dense_row(double *dst, const uint16_t *X, const uint16_t *W,
                      int64_t I, int64_t H, int64_t i)
{
    for (int64_t j = 0; j < H; j++) {
        double acc = 0.0;
        for (int64_t k = 0; k < I; k++)
            acc += bf16_to_double(X[i * I + k]) * bf16_to_double(W[j * I + k]);
        dst[j] = acc;
    }
}

/* Y = X W^T: X [M, I], W [H, I] row-major bf16; Y [M, H] doubles. */
int oracle_dense(double *Y, const uint16_t *X, const uint16_t *W, int64_t M,
                 int64_t I, int64_t H)
{
    if (M <= 0 || I <= 0 || H <= 0)
        return -2;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < M; i++)
        dense_row(Y + i * H, X, W, I, H, i);
    return 0;
}

/* Selected rows of Y = X W^T: rows[0..n-1] index X; output n x H doubles. */
int oracle_dense_rows(double *Y, const uint16_t *X, const uint16_t *W,
                      int64_t M, int64_t I, int64_t H, const int64_t *rows,
                      int64_t n)
{
    if (M <= 0 || I <= 0 || H <= 0)
        return -2;
    for (int64_t r = 0; r < n; r++)
        if (rows[r] < 0 || rows[r] >= M)
            return -2;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; r++)
        dense_row(Y + r * H, X, W, I, H, rows[r]);
    return 0;
}

/*
 * Batched NT product Y[i][j][k] = sum_l X[i][j][l] * W[i][k][l]
 * (test_local_padding_ii): X [batch, T1, D], W [batch, T2, D] bf16,
 * Y [batch, T1, T2] doubles. T1 and T2 may differ (the page uses T1 = T2).
 */
int oracle_bmm_nt(double *Y, const uint16_t *X, const uint16_t *W, int64_t batch,
                  int64_t T1, int64_t T2, int64_t D)
{
    if (batch <= 0 || T1 <= 0 || T2 <= 0 || D <= 0)
        return -2;
    const int64_t rows = batch * T1;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < rows; r++) {
        const int64_t i = r / T1, j = r % T1;
        const uint16_t *x = X + (i * T1 + j) * D;
        double *y = Y + (i * T1 + j) * T2;
        for (int64_t k = 0; k < T2; k++) {
            const uint16_t *w = W + (i * T2 + k) * D;
            double acc = 0.0;
            for (int64_t l = 0; l < D; l++)
                acc += bf16_to_double(x[l]) * bf16_to_double(w[l]);
            y[k] = acc;
        }
    }
    return 0;
}

/*
 * Causal softmax of the score rows: for each (b, h, t), over t2 <= t,
 * P[t2] = exp(s[t2] - m) / sum_{u <= t} exp(s[u] - m) with s = the trimul_cpu
 * score and m = max_{u <= t} s[u]; P[t2] = 0 for t2 > t. (B, NH, T, T) doubles.
 */
static void softmax_row(double *dst, const uint16_t *qkv, int64_t T, int64_t C,
                        int64_t NH, int64_t b, int64_t h, int64_t t)
{
    score_row(dst, qkv, T, C, NH, b, h, t, 0.0);
    double m = dst[0];
    for (int64_t t2 = 1; t2 <= t; t2++)
        if (dst[t2] > m)
            m = dst[t2];
    double sum = 0.0;
    for (int64_t t2 = 0; t2 <= t; t2++) {
        dst[t2] = exp(dst[t2] - m);
        sum += dst[t2];
    }
    for (int64_t t2 = 0; t2 <= t; t2++)
        dst[t2] /= sum;
    for (int64_t t2 = t + 1; t2 < T; t2++)
        dst[t2] = 0.0;
}

int oracle_causal_softmax(double *out, const uint16_t *qkv, int64_t B, int64_t T,
                          int64_t C, int64_t NH)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    const int64_t rows = B * NH * T;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; r++) {
        const int64_t t = r % T;
        const int64_t h = (r / T) % NH;
        const int64_t b = r / (T * NH);
        softmax_row(out + r * T, qkv, T, C, NH, b, h, t);
    }
    return 0;
}

/* Selected rows (b, h, t) of the causal softmax, n x T doubles. */
int oracle_causal_softmax_rows(double *out, const uint16_t *qkv, int64_t B, int64_t T,
                               int64_t C, int64_t NH, const int64_t *bht, int64_t n)
{
    if (check_trimul_shape(B, T, C, NH))
        return -2;
    for (int64_t i = 0; i < n; i++) {
        const int64_t b = bht[3 * i], h = bht[3 * i + 1], t = bht[3 * i + 2];
        if (b < 0 || b >= B || h < 0 || h >= NH || t < 0 || t >= T)
            return -2;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n; i++)
        softmax_row(out + i * T, qkv, T, C, NH, bht[3 * i], bht[3 * i + 1], bht[3 * i + 2]);
    return 0;
}
