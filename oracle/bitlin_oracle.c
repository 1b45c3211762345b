/*
 * CPU oracle for the Hadamard-folded 1-bit matrix-vector product.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * restatement of what the method computes, in double precision.  It is called
 * by the tests, by the package's smoke check and by the benchmark's CPU
 * baseline; the library's own path never calls, links or includes it, and it
 * shares no code with the CUDA kernels.
 *
 * Sources (page title, then the section the step comes from):
 *  - "ARCHITECTURE-SPEC" of the Pulse engine, section on the Hadamard fold:
 *    order of the activation transform (optional tiled->grouped head
 *    permutation, then x*signs, then a normalized Sylvester-Walsh transform in
 *    blocks of 1024 scaled by 1/32, then y = W @ x); the inverse order used by
 *    the embedding (h = signs * WHT(z)); the ssm_out permutation
 *    tiled [hd=128, nk=16, rep=3] -> grouped [hd, rep, nk].
 *  - "Inside the One-Bit Engine", first station (a weight is one bit: 1 means
 *    +1, 0 means -1, one shared scale per 128 weights; the shader accumulates
 *    a group sum of +-a and multiplies by the scale once per 128) and the
 *    station on the one-bit row format (bit k of a row is bit k&31 of word
 *    k>>5; the scale of k is scale[k>>7], IEEE binary16).
 *
 * Readings taken where the pages leave a step open:
 *  - "tiled [hd,nk,rep]" lists dimensions innermost first (ggml order), so the
 *    tiled offset of (d,k,r) is d + 128*(k + 16*r) and the grouped offset of
 *    (d,r,k) is d + 128*(r + 3*k); grouped[d,r,k] = tiled[d,k,r].
 *  - "Sylvester-Walsh" is the natural (Sylvester) ordering,
 *    H[i][j] = (-1)^popcount(i & j).  Parity on this point is unpinned: only
 *    real folded weights could tell it from the sequency ordering.
 *  - Blocks are contiguous and independent: block b holds x[1024b .. 1024b+1023].
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK 1024
#define ORACLE_GROUP 128

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero and subnormals: f * 2^-24 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16 value (8 significant bits, ties to
 * even), returned as a double.  bfloat16 keeps float32's exponent range. */
double oracle_round_bf16(double v)
{
    if (v == 0.0 || isnan(v) || isinf(v))
        return v;
    int e;
    double m = frexp(v, &e);           /* v = m * 2^e, 0.5 <= |m| < 1 */
    if (e - 1 < -126) {                /* bf16 subnormal range: fixed quantum 2^-133 */
        return ldexp(nearbyint(ldexp(v, 133)), -133);
    }
    double q = nearbyint(ldexp(m, 8)); /* 8 significant bits, current mode = nearest-even */
    return ldexp(q, e - 8);
}

/* Sylvester Hadamard entry H[i][j] = (-1)^popcount(i & j). */
static int hadamard_entry(unsigned i, unsigned j)
{
    return (__builtin_popcount(i & j) & 1) ? -1 : 1;
}

/* One block of the normalized transform by its definition:
 * out[i] = (1/32) * sum_j H[i][j] * in[j], 1024 x 1024 terms. */
void oracle_wht_block(const double* in, double* out)
{
    for (unsigned i = 0; i < ORACLE_BLOCK; ++i) {
        double s = 0.0;
        for (unsigned j = 0; j < ORACLE_BLOCK; ++j)
            s += hadamard_entry(i, j) * in[j];
        out[i] = s / 32.0;
    }
}

/* ssm_out head permutation (K = 6144): tiled [hd=128, nk=16, rep=3] ->
 * grouped [hd, rep, nk].  out[d + 128*(r + 3*k)] = in[d + 128*(k + 16*r)]. */
void oracle_permute_tiled_to_grouped(const double* in, double* out)
{
    for (int k = 0; k < 16; ++k)
        for (int r = 0; r < 3; ++r)
            for (int d = 0; d < 128; ++d)
                out[d + 128 * (r + 3 * k)] = in[d + 128 * (k + 16 * r)];
}

/* Activation transform applied right before the folded matmul, one token:
 * [permutation if perm] -> times signs -> blockwise normalized transform.
 * x is f64 here (the MLP block feeds it the f64 middle vector); oracle_rotate
 * below is the same for f32 activations.
 * Returns 0, or -1 if scratch memory could not be allocated. */
int oracle_rotate_f64(const double* x, int K, const float* signs, int perm, double* xt)
{
    double* t = (double*)malloc(sizeof(double) * (size_t)K);
    double* p = (double*)malloc(sizeof(double) * (size_t)K);
    if (!t || !p) {
        free(t);
        free(p);
        return -1;
    }
    for (int i = 0; i < K; ++i)
        t[i] = x[i];
    if (perm) {
        oracle_permute_tiled_to_grouped(t, p);
        for (int i = 0; i < K; ++i)
            t[i] = p[i];
    }
    for (int i = 0; i < K; ++i)
        t[i] *= (double)signs[i];
    for (int blk = 0; blk < K / ORACLE_BLOCK; ++blk)
        oracle_wht_block(t + blk * ORACLE_BLOCK, xt + blk * ORACLE_BLOCK);
    free(t);
    free(p);
    return 0;
}

int oracle_rotate(const float* x, int K, const float* signs, int perm, double* xt)
{
    double* t = (double*)malloc(sizeof(double) * (size_t)K);
    if (!t)
        return -1;
    for (int i = 0; i < K; ++i)
        t[i] = (double)x[i];
    int rc = oracle_rotate_f64(t, K, signs, perm, xt);
    free(t);
    return rc;
}

/* The embedding's inverse order: h = signs * WHT(z). */
void oracle_inverse_rotate(const double* z, int K, const float* signs, double* h)
{
    for (int blk = 0; blk < K / ORACLE_BLOCK; ++blk)
        oracle_wht_block(z + blk * ORACLE_BLOCK, h + blk * ORACLE_BLOCK);
    for (int i = 0; i < K; ++i)
        h[i] *= (double)signs[i];
}

/* Weight (n, k) as +-1: bit k&31 of word k>>5 of row n; 1 -> +1, 0 -> -1. */
static int weight_sign(const uint32_t* bits, int K, int n, int k)
{
    uint32_t word = bits[(size_t)n * (K / 32) + (k >> 5)];
    return ((word >> (k & 31)) & 1u) ? 1 : -1;
}

/* Rotated activations for M tokens, xt[M][K]; round_bf16 rounds each entry to
 * bfloat16 afterwards (the tensor-core path's operand precision). */
int oracle_rotate_tokens(const float* x, int M, int K, const float* signs, int perm,
                         int round_bf16, double* xt)
{
    int failed = 0;
    #pragma omp parallel for schedule(dynamic, 1) reduction(|:failed)
    for (int m = 0; m < M; ++m) {
        double* row = xt + (size_t)m * K;
        if (oracle_rotate(x + (size_t)m * K, K, signs, perm, row) != 0) {
            failed = 1;
            continue;
        }
        if (round_bf16)
            for (int i = 0; i < K; ++i)
                row[i] = oracle_round_bf16(row[i]);
    }
    return failed ? -1 : 0;
}

/* y[m][r] = sum_g scale(n, g) * sum_{k in group g} (+-1)(n, k) * xt[m][k],
 * for n = rows[r].  Each group sum is formed first and scaled once, as the
 * shader does. */
void oracle_product(const uint32_t* bits, const uint16_t* scales, const double* xt,
                    int M, int N, int K, const int64_t* rows, int nrows, double* y)
{
    const int G = K / ORACLE_GROUP;
    (void)N;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; ++m) {
        for (int r = 0; r < nrows; ++r) {
            const int n = (int)rows[r];
            const double* xm = xt + (size_t)m * K;
            double acc = 0.0;
            for (int g = 0; g < G; ++g) {
                double gsum = 0.0;
                for (int k = g * ORACLE_GROUP; k < (g + 1) * ORACLE_GROUP; ++k)
                    gsum += weight_sign(bits, K, n, k) * xm[k];
                acc += oracle_f16_to_f64(scales[(size_t)n * G + g]) * gsum;
            }
            y[(size_t)m * nrows + r] = acc;
        }
    }
}

/* Dequantized row n: w[k] = +-scale(n, k>>7), as the embedding lookup writes it. */
void oracle_dequant_row(const uint32_t* bits, const uint16_t* scales, int K, int n, double* w)
{
    const int G = K / ORACLE_GROUP;
    for (int k = 0; k < K; ++k)
        w[k] = weight_sign(bits, K, n, k) * oracle_f16_to_f64(scales[(size_t)n * G + (k >> 7)]);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
