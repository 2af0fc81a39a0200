/*
 * oracle.c -- plain CPU reference for the dense half-precision GEMM
 *
 *     D = alpha * A * B + beta * C
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes, and where that comes from:
 *
 *  - The element definition C[i,j] = sum over k in [0,K) of A[i,k] * B[k,j]
 *    ("矩阵乘法优化可视化学习文档", section 1 and the triple loop of section 3):
 *    loop i, then j, then k ascending, one accumulator per output element.
 *  - The multiply-accumulate D = A x B + C, with C allowed to alias D
 *    ("CUDA算子优化(5)：WMMA矩阵乘法", WMMA API section (5) mma_sync;
 *    "深入CUDA Tensor Core与WMMA", section 2.2).  The alpha/beta scaling is
 *    the BLAS reading of that accumulate: D = alpha*(A*B) + beta*C, with C
 *    not read at all when beta == 0.
 *  - Storage order: a row-major M x N matrix keeps element (i,j) at offset
 *    i*N + j, a column-major one at j*M + i ("深入CUDA Tensor Core与WMMA",
 *    section 3.2, the 2x3 example).  With a leading dimension ld >= the
 *    contiguous extent the offsets become i*ld + j and j*ld + i (same page,
 *    section 4.2, ldm).
 *  - Inputs are IEEE binary16 or bfloat16 bit patterns, decoded exactly to
 *    binary64 from the format definitions (no CUDA header is used).  The
 *    other tensor-core input types the pages list for Blackwell ("深入CUDA
 *    Tensor Core与WMMA", section 2.3: FP8 and TF32) are decoded the same
 *    way: the two 8-bit float formats E4M3 and E5M2 from their bit layouts,
 *    and TF32 operands -- stored as binary32 -- as the binary32 value
 *    itself (the product of the matrices as given; the reduced precision
 *    with which the tensor cores read them is a property of the device
 *    path, bounded by the tests' tolerance, and exact for inputs whose low
 *    13 fraction bits are zero).
 *  - Arithmetic is binary64 throughout.  Every product of two 11-bit (or
 *    8-bit) significands is exact in binary64; the K-sum has a relative
 *    error of at most K * 2^-53, far below any tolerance used against it.
 *  - The output is rounded ONCE, round-to-nearest-even, to the output type
 *    (float32 by the C conversion, which is IEEE RNE under the default
 *    rounding mode; binary16/bfloat16 by the encoder below).  This holds for
 *    the fp16-accumulate mode too: the oracle's value there is the exact
 *    result rounded once to binary16, and the fp16 accumulation of the
 *    device path is compared with it under the looser fp16 tolerance.
 *  - Alongside D it can return the unrounded value V and the error scale
 *    S[i,j] = |alpha| * sum_k |A[i,k] B[k,j]| + |beta * C[i,j]|.
 *
 * Threads only split the set of output rows (or sampled entries); the
 * arithmetic of each element is the single-accumulator loop above.
 *
 * Fused epilogue (the *_ep entry points).  The pages list epilogue fusion
 * -- bias, activation and scale applied before the write-back -- among the
 * standard GEMM optimisations ("矩阵乘法优化可视化学习文档", section 6, the
 * "Epilogue fusion" row, and section 8, the store step of the Triton
 * kernel) without fixing a formula.  The reading taken here:
 *     U[i,j] = alpha * r[i] * c[j] * sum_k A[i,k] B[k,j] + beta * C[i,j] + bias[j]
 *     D[i,j] = act(U[i,j])
 * with r (per-row scale), c (per-column scale) and bias given as float32
 * vectors (1, 1 and 0 when absent), act = identity, ReLU(u) = max(u, 0) or
 * GELU(u) = u * Phi(u) = u/2 * (1 + erf(u / sqrt 2)) (the exact form, erf
 * from the C library in binary64).  S becomes the error scale of U:
 * |alpha r c| * sum |A B| + |beta C| + |bias|.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Type and layout codes of this file (independent of the product's enums). */
enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3, OR_E5M2 = 4, OR_TF32 = 5 };
enum { OR_ROW = 0, OR_COL = 1 };

/* ---------------------------------------------------------------------- */
/* Format definitions                                                     */
/* ---------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * normal:    (-1)^s * 2^(e-15) * (1 + f/1024)  = (1024 + f) * 2^(e-25)
 * subnormal: (-1)^s * 2^-14 * (f/1024)         = f * 2^-24              */
double oracle_f16_decode(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * normal:    (128 + f) * 2^(e-134);  subnormal: f * 2^-133               */
double oracle_bf16_decode(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 7) & 0xff, f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return s ? -v : v;
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities, exponent 15 with fraction 7 is NaN (so the largest finite
 * value is 1.75 * 2^8 = 448).
 * normal:    (8 + f) * 2^(e-10);  subnormal: f * 2^-9                   */
double oracle_e4m3_decode(uint8_t h)
{
    int s = (h >> 7) & 1, e = (h >> 3) & 0xf, f = h & 0x7;
    double v;
    if (e == 0)
        v = ldexp((double)f, -9);
    else if (e == 15 && f == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + f), e - 10);
    return s ? -v : v;
}

/* E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits; exponent
 * 31 holds infinities (fraction 0) and NaNs, as in binary16.
 * normal:    (4 + f) * 2^(e-17);  subnormal: f * 2^-16                  */
double oracle_e5m2_decode(uint8_t h)
{
    int s = (h >> 7) & 1, e = (h >> 2) & 0x1f, f = h & 0x3;
    double v;
    if (e == 0)
        v = ldexp((double)f, -16);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(4 + f), e - 17);
    return s ? -v : v;
}

/* binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits.
 * normal:    (2^23 + f) * 2^(e-150);  subnormal: f * 2^-149             */
double oracle_f32_decode(uint32_t w)
{
    int s = (w >> 31) & 1, e = (w >> 23) & 0xff;
    uint32_t f = w & 0x7fffffu;
    double v;
    if (e == 0)
        v = ldexp((double)f, -149);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(8388608u + f), e - 150);
    return s ? -v : v;
}

/* Round-to-nearest-even of a binary64 value into a binary format with
 * `frac_bits` stored fraction bits and `exp_bits` exponent bits. */
static uint16_t encode_rne(double x, int frac_bits, int exp_bits)
{
    const int bias = (1 << (exp_bits - 1)) - 1;
    const int emin = 1 - bias;                 /* exponent of the smallest normal */
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (frac_bits + exp_bits)) : 0;
    const uint16_t exp_ones = (uint16_t)(((1u << exp_bits) - 1) << frac_bits);
    if (isnan(x))
        return sign | exp_ones | (uint16_t)(1u << (frac_bits - 1));  /* quiet NaN */
    double a = fabs(x);
    if (isinf(a))
        return sign | exp_ones;
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);               /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;              /* unbiased exponent of a */
    if (E < emin)
        E = emin;                /* subnormal range shares emin's quantum */
    /* a / quantum, exact: the quantum is a power of two */
    double n = ldexp(a, frac_bits - E);
    double fl = floor(n), rem = n - fl;
    double r = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    const double one = ldexp(1.0, frac_bits);  /* implicit leading bit */
    if (r < one)                                 /* stays subnormal (E == emin) */
        return sign | (uint16_t)r;
    if (r >= 2.0 * one) {                        /* carried into the next binade */
        r = one;
        E += 1;
    }
    int biased = E + bias;
    if (biased >= (1 << exp_bits) - 1)
        return sign | exp_ones;                  /* overflow -> infinity */
    return sign | (uint16_t)((unsigned)biased << frac_bits) | (uint16_t)(r - one);
}

uint16_t oracle_f16_encode(double x) { return encode_rne(x, 10, 5); }
uint16_t oracle_bf16_encode(double x) { return encode_rne(x, 7, 8); }

/* ---------------------------------------------------------------------- */
/* The GEMM definition                                                    */
/* ---------------------------------------------------------------------- */

typedef struct {
    int in_dtype;               /* OR_F16, OR_BF16, OR_E4M3, OR_E5M2 or OR_TF32 */
    const void *A, *B;          /* bit patterns: 16-bit, 8-bit or 32-bit elements */
    const void *C;              /* out_dtype elements, row-major, ld = ldc; may be NULL if beta == 0 */
    int64_t M, N, K, lda, ldb, ldc;
    int layoutA, layoutB;       /* OR_ROW / OR_COL */
    int out_dtype;              /* OR_F16 / OR_BF16 / OR_F32 */
    double alpha, beta;
    /* fused epilogue (all optional) */
    const float *bias;          /* N, added per column */
    const float *row_scale;     /* M, multiplies row i of alpha * A * B */
    const float *col_scale;     /* N, multiplies column j of alpha * A * B */
    int act;                    /* OR_ACT_* */
} gemm_args;

enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_GELU = 2 };

static double decode_in(int dt, uint16_t h)
{
    return dt == OR_F16 ? oracle_f16_decode(h) : oracle_bf16_decode(h);
}

/* element `off` of an input matrix of type dt */
static double input_at(int dt, const void *m, int64_t off)
{
    switch (dt) {
    case OR_E4M3: return oracle_e4m3_decode(((const uint8_t *)m)[off]);
    case OR_E5M2: return oracle_e5m2_decode(((const uint8_t *)m)[off]);
    case OR_TF32: return oracle_f32_decode(((const uint32_t *)m)[off]);
    default: return decode_in(dt, ((const uint16_t *)m)[off]);
    }
}

/* a(i,k): element (i,k) of the M x K matrix A in its storage order */
static double a_at(const gemm_args *g, int64_t i, int64_t k)
{
    int64_t off = g->layoutA == OR_ROW ? i * g->lda + k : k * g->lda + i;
    return input_at(g->in_dtype, g->A, off);
}

/* b(k,j): element (k,j) of the K x N matrix B in its storage order */
static double b_at(const gemm_args *g, int64_t k, int64_t j)
{
    int64_t off = g->layoutB == OR_ROW ? k * g->ldb + j : j * g->ldb + k;
    return input_at(g->in_dtype, g->B, off);
}

/* c(i,j): element (i,j) of the row-major M x N matrix C */
static double c_at(const gemm_args *g, int64_t i, int64_t j)
{
    int64_t off = i * g->ldc + j;
    if (g->out_dtype == OR_F32)
        return (double)((const float *)g->C)[off];
    return decode_in(g->out_dtype, ((const uint16_t *)g->C)[off]);
}

/* One output element: V = alpha * sum_k a(i,k) b(k,j) + beta * c(i,j),
 * S = |alpha| * sum_k |a(i,k) b(k,j)| + |beta * c(i,j)|. */
static void element(const gemm_args *g, int64_t i, int64_t j, double *v_out, double *s_out)
{
    double acc = 0.0, sabs = 0.0;
    for (int64_t k = 0; k < g->K; ++k) {
        double p = a_at(g, i, k) * b_at(g, k, j);
        acc += p;
        sabs += fabs(p);
    }
    double v = g->alpha * acc;
    double s = fabs(g->alpha) * sabs;
    if (g->row_scale || g->col_scale) {
        double sc = (g->row_scale ? (double)g->row_scale[i] : 1.0) *
                    (g->col_scale ? (double)g->col_scale[j] : 1.0);
        v *= sc;
        s *= fabs(sc);
    }
    if (g->beta != 0.0) {
        double c = c_at(g, i, j);
        v += g->beta * c;
        s += fabs(g->beta * c);
    }
    if (g->bias) {
        v += (double)g->bias[j];
        s += fabs((double)g->bias[j]);
    }
    if (g->act == OR_ACT_RELU)
        v = v > 0.0 ? v : 0.0;
    else if (g->act == OR_ACT_GELU)
        v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
    *v_out = v;
    *s_out = s;
}

static void store_out(int out_dtype, void *D, int64_t off, double v)
{
    if (out_dtype == OR_F32)
        ((float *)D)[off] = (float)v;
    else if (out_dtype == OR_F16)
        ((uint16_t *)D)[off] = oracle_f16_encode(v);
    else
        ((uint16_t *)D)[off] = oracle_bf16_encode(v);
}

typedef struct {
    const gemm_args *g;
    /* full mode */
    void *D;
    int64_t ldd;
    double *V, *S;              /* optional, M x N dense */
    int64_t row_begin, row_end;
    /* entries mode */
    const int64_t *ii, *jj;
    int64_t e_begin, e_end;
    double *Ve, *Se;
} work;

static void *run_rows(void *p)
{
    work *w = (work *)p;
    const gemm_args *g = w->g;
    for (int64_t i = w->row_begin; i < w->row_end; ++i)
        for (int64_t j = 0; j < g->N; ++j) {
            double v, s;
            element(g, i, j, &v, &s);
            if (w->D)
                store_out(g->out_dtype, w->D, i * w->ldd + j, v);
            if (w->V)
                w->V[i * g->N + j] = v;
            if (w->S)
                w->S[i * g->N + j] = s;
        }
    return NULL;
}

static void *run_entries(void *p)
{
    work *w = (work *)p;
    for (int64_t e = w->e_begin; e < w->e_end; ++e)
        element(w->g, w->ii[e], w->jj[e], &w->Ve[e], &w->Se[e]);
    return NULL;
}

static int check(const gemm_args *g)
{
    if (g->in_dtype != OR_F16 && g->in_dtype != OR_BF16 && g->in_dtype != OR_E4M3 && g->in_dtype != OR_E5M2 &&
        g->in_dtype != OR_TF32)
        return 1;
    if (g->out_dtype != OR_F16 && g->out_dtype != OR_BF16 && g->out_dtype != OR_F32)
        return 1;
    if (g->M < 0 || g->N < 0 || g->K < 0)
        return 1;
    if ((g->M > 0 && g->K > 0) && !g->A)
        return 1;
    if ((g->N > 0 && g->K > 0) && !g->B)
        return 1;
    if (g->beta != 0.0 && !g->C && g->M > 0 && g->N > 0)
        return 1;
    if (g->act != OR_ACT_NONE && g->act != OR_ACT_RELU && g->act != OR_ACT_GELU)
        return 1;
    return 0;
}

static int clamp_threads(int nthreads, int64_t units)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 512)
        nthreads = 512;
    if (units < nthreads)
        nthreads = units > 0 ? (int)units : 1;
    return nthreads;
}

/* Full product with the fused epilogue.  D (ldd), V and S may each be NULL.
 * Rows [0, M) are split over `nthreads` threads.  Returns 0 on success. */
int oracle_gemm_ep(int in_dtype, const void *A, const void *B, const void *C,
                   void *D, int64_t ldd, double *V, double *S,
                   int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                   int layoutA, int layoutB, int out_dtype, double alpha, double beta,
                   const float *bias, const float *row_scale, const float *col_scale, int act,
                   int nthreads)
{
    gemm_args g = {in_dtype, A, B, C, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                   out_dtype, alpha, beta, bias, row_scale, col_scale, act};
    if (check(&g))
        return 1;
    int nt = clamp_threads(nthreads, M);
    pthread_t th[512];
    work w[512];
    for (int t = 0; t < nt; ++t) {
        memset(&w[t], 0, sizeof(work));
        w[t].g = &g;
        w[t].D = D;
        w[t].ldd = ldd;
        w[t].V = V;
        w[t].S = S;
        w[t].row_begin = M * t / nt;
        w[t].row_end = M * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t)
        pthread_create(&th[t], NULL, run_rows, &w[t]);
    run_rows(&w[0]);
    for (int t = 1; t < nt; ++t)
        pthread_join(th[t], NULL);
    return 0;
}

/* Full product, plain epilogue (D = alpha A B + beta C). */
int oracle_gemm(int in_dtype, const void *A, const void *B, const void *C,
                void *D, int64_t ldd, double *V, double *S,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                int layoutA, int layoutB, int out_dtype, double alpha, double beta,
                int nthreads)
{
    return oracle_gemm_ep(in_dtype, A, B, C, D, ldd, V, S, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                          out_dtype, alpha, beta, NULL, NULL, NULL, OR_ACT_NONE, nthreads);
}

/* Selected entries (ii[e], jj[e]) only, with the fused epilogue: V and S. */
int oracle_gemm_entries_ep(int in_dtype, const void *A, const void *B, const void *C,
                           const int64_t *ii, const int64_t *jj, int64_t n_entries,
                           double *V, double *S,
                           int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           int layoutA, int layoutB, int out_dtype, double alpha, double beta,
                           const float *bias, const float *row_scale, const float *col_scale, int act,
                           int nthreads)
{
    gemm_args g = {in_dtype, A, B, C, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                   out_dtype, alpha, beta, bias, row_scale, col_scale, act};
    if (check(&g))
        return 1;
    for (int64_t e = 0; e < n_entries; ++e)
        if (ii[e] < 0 || ii[e] >= M || jj[e] < 0 || jj[e] >= N)
            return 1;
    int nt = clamp_threads(nthreads, n_entries);
    pthread_t th[512];
    work w[512];
    for (int t = 0; t < nt; ++t) {
        memset(&w[t], 0, sizeof(work));
        w[t].g = &g;
        w[t].ii = ii;
        w[t].jj = jj;
        w[t].Ve = V;
        w[t].Se = S;
        w[t].e_begin = n_entries * t / nt;
        w[t].e_end = n_entries * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t)
        pthread_create(&th[t], NULL, run_entries, &w[t]);
    run_entries(&w[0]);
    for (int t = 1; t < nt; ++t)
        pthread_join(th[t], NULL);
    return 0;
}

/* Selected entries, plain epilogue. */
int oracle_gemm_entries(int in_dtype, const void *A, const void *B, const void *C,
                        const int64_t *ii, const int64_t *jj, int64_t n_entries,
                        double *V, double *S,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        int layoutA, int layoutB, int out_dtype, double alpha, double beta,
                        int nthreads)
{
    return oracle_gemm_entries_ep(in_dtype, A, B, C, ii, jj, n_entries, V, S, M, N, K, lda, ldb, ldc,
                                  layoutA, layoutB, out_dtype, alpha, beta, NULL, NULL, NULL, OR_ACT_NONE,
                                  nthreads);
}

/* Round n binary64 values once, RNE, to out_dtype (for sampled entries). */
int oracle_round(const double *v, int64_t n, int out_dtype, void *out)
{
    if (out_dtype != OR_F16 && out_dtype != OR_BF16 && out_dtype != OR_F32)
        return 1;
    for (int64_t e = 0; e < n; ++e)
        store_out(out_dtype, out, e, v[e]);
    return 0;
}

/* Vector decoders for the tests (elements of the input type's width). */
void oracle_decode(const void *h, int64_t n, int dtype, double *out)
{
    for (int64_t e = 0; e < n; ++e)
        out[e] = input_at(dtype, h, e);
}
