/*
 * CPU oracle for the LLM.int8() mixed-precision decomposed matmul Y = X.W.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path.
 *
 * Every step is written out plainly in the order the pages give it; there is no
 * blocking, fusion or reordering of arithmetic.  Integer products are
 * accumulated in int64; the fp16 outlier product and the final merge are done
 * in double; the one place where floating point decides an integer (the int8
 * code) is done in fp32, the precision the GPU kernels use, with an explicit
 * rounding rule (round half away from zero).  Build with -ffp-contract=off and
 * without fast-math so that each float operation rounds exactly once.
 *
 * Sources (page title, section):
 *   [WALK]     "LLM.int8() paper walkthrough" (2kiu.com), sections 2.1-2.3
 *   [PITFALLS] "LLM.int8() quantization pitfalls guide" (codearts.csdn.net),
 *              sections 1, 2 (worked example) and 3.1-3.3
 *   [PRACTICE] "LLM quantization in practice: INT8 to QLoRA" (cnnetsun.cn),
 *              sections 3.2 (clamp after round) and 3.3 (symmetric absmax)
 *   [FABRIC]   "8-bit LLM quantization with Lightning Fabric" (aicoding.csdn.net),
 *              section 2.2 (per-output-channel weight scale; int32 result
 *              rescaled by scale_x * scale_w)
 *
 * Layouts (all row-major, caller-owned host memory):
 *   X   fp16 bits [M,K]     W   fp16 bits [K,N]     Y fp16 bits [M,N]
 *   (the *_fmt entry points take fmt = 1 for bfloat16 X, W and Y instead)
 *   Xq  int8 [M,K]          Wq  int8 [K,N]          C int64 [M,N]
 *   s_x float [M]           s_w float [N]           F double [M,N]
 *   is_outlier uint8 [K] (1 = column of X is an outlier dimension)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * IEEE binary16 <-> double, written from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 * ------------------------------------------------------------------------- */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round-to-nearest-even conversion of a double to binary16 (overflow -> inf). */
uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds to even -> inf */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = q * 2^-24, q rounded to nearest even;
         * q == 1024 encodes the smallest normal number, which is correct. */
        double q = nearbyint(ldexp(a, 24));
        return sign | (uint16_t)q;
    }
    int e;
    double m = frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 11)); /* 11 significant bits, RNE */
    e -= 1;                             /* a = (r/1024) * 2^e */
    if (r == 2048.0) {
        r = 1024.0;
        e += 1;
    }
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)r - 1024);
}

/* ---------------------------------------------------------------------------
 * bfloat16 <-> double, written from the format definition (1 sign bit, 8
 * exponent bits with bias 127, 7 fraction bits: the upper half of a binary32).
 * ------------------------------------------------------------------------- */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* subnormal: f * 2^-133 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* (1.f) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round-to-nearest-even conversion of a double to bfloat16 (overflow -> inf). */
uint16_t oracle_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7fc0;
    /* halfway between the largest finite value (2 - 2^-7) * 2^127 and 2^128 */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127))
        return sign | 0x7f80;
    if (a < ldexp(1.0, -126)) {
        /* subnormal range: value = q * 2^-133, q rounded to nearest even;
         * q == 128 encodes the smallest normal number, which is correct. */
        double q = nearbyint(ldexp(a, 133));
        return sign | (uint16_t)q;
    }
    int e;
    double m = frexp(a, &e);           /* a = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(ldexp(m, 8)); /* 8 significant bits, RNE */
    e -= 1;                            /* a = (r/128) * 2^e */
    if (r == 256.0) {
        r = 128.0;
        e += 1;
    }
    return sign | (uint16_t)((e + 127) << 7) | (uint16_t)((int)r - 128);
}

/* 16-bit floating-point element formats of X, W and Y: 0 = fp16, 1 = bf16. */
static double elem_to_double(uint16_t v, int fmt)
{
    return fmt ? oracle_bf16_to_double(v) : oracle_half_to_double(v);
}
static uint16_t double_to_elem(double v, int fmt)
{
    return fmt ? oracle_double_to_bf16(v) : oracle_double_to_half(v);
}
static float elem_to_float(uint16_t v, int fmt) { return (float)elem_to_double(v, fmt); }
static float half_to_float(uint16_t h) { return (float)oracle_half_to_double(h); }

/* ---------------------------------------------------------------------------
 * Symmetric absmax quantization of one value, as [PITFALLS] section 1 states it:
 *   scale_factor = 127 / max|x|,  q = round(x * scale_factor),
 * with the result clamped to [-127, 127] after rounding and before the cast to
 * int8 ([PRACTICE] section 3.2; symmetric range without -128, section 3.3).
 * Precision: fp32 for the scale factor and the product, each rounded once
 * (round-to-nearest-even); round() is C's round half away from zero.
 * A zero absmax gives scale factor 0, hence code 0.
 * ------------------------------------------------------------------------- */
float oracle_scale_factor(float absmax)
{
    return absmax > 0.0f ? 127.0f / absmax : 0.0f;
}

int8_t oracle_code(float x, float scale_factor)
{
    float p = x * scale_factor;
    float r = roundf(p);
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)r;
}

/* ---------------------------------------------------------------------------
 * A0. Weight quantization, one scale per output column ([WALK] section 2.1:
 * weights get a per-column scale; [FABRIC] section 2.2: one scale per output
 * neuron).  The column absmax runs over all K rows, because W is quantized
 * once, before any X is seen.
 * ------------------------------------------------------------------------- */
void oracle_quantize_weight_fmt(const uint16_t *W, int64_t K, int64_t N, int8_t *Wq, float *s_w, int fmt)
{
    for (int64_t n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(elem_to_float(W[k * N + n], fmt));
            if (a > amax)
                amax = a;
        }
        s_w[n] = amax;
        float sf = oracle_scale_factor(amax);
        for (int64_t k = 0; k < K; ++k)
            Wq[k * N + n] = oracle_code(elem_to_float(W[k * N + n], fmt), sf);
    }
}

void oracle_quantize_weight(const uint16_t *W, int64_t K, int64_t N, int8_t *Wq, float *s_w)
{
    oracle_quantize_weight_fmt(W, K, N, Wq, s_w, 0);
}

/* ---------------------------------------------------------------------------
 * Ablation, not a step of the path: per-tensor quantization, the coarse
 * granularity [FABRIC] section 3.4 contrasts with per-channel scales.  One
 * absmax over all n values of a tensor, then the same code rule as A0/A2.
 * ------------------------------------------------------------------------- */
void oracle_quantize_per_tensor(const uint16_t *A, int64_t n, int8_t *q, float *s)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(half_to_float(A[i]));
        if (a > amax)
            amax = a;
    }
    *s = amax;
    float sf = oracle_scale_factor(amax);
    for (int64_t i = 0; i < n; ++i)
        q[i] = oracle_code(half_to_float(A[i]), sf);
}

/* ---------------------------------------------------------------------------
 * A1. Outlier dimensions ([WALK] section 2.3): a K-column of X whose largest
 * magnitude exceeds the threshold t (default 6.0) is an outlier column.
 * "Exceeds" is read as strict: |x| > t.
 * ------------------------------------------------------------------------- */
void oracle_outlier_columns_fmt(const uint16_t *X, int64_t M, int64_t K, float t, uint8_t *is_outlier, int fmt)
{
    for (int64_t j = 0; j < K; ++j) {
        int out = 0;
        for (int64_t i = 0; i < M; ++i)
            if (fabsf(elem_to_float(X[i * K + j], fmt)) > t)
                out = 1;
        is_outlier[j] = (uint8_t)out;
    }
}

void oracle_outlier_columns(const uint16_t *X, int64_t M, int64_t K, float t, uint8_t *is_outlier)
{
    oracle_outlier_columns_fmt(X, M, K, t, is_outlier, 0);
}

/* ---------------------------------------------------------------------------
 * A2. Row quantization of the non-outlier part of X ([WALK] section 2.1:
 * activations get a per-row scale; section 2.3: only X_normal, the
 * non-outlier columns, is quantized).  The row absmax is taken over the
 * non-outlier columns; outlier columns get code 0 (they are carried by the
 * fp16 product instead).
 * ------------------------------------------------------------------------- */
void oracle_quantize_rows_fmt(const uint16_t *X, int64_t M, int64_t K, const uint8_t *is_outlier,
                              int8_t *Xq, float *s_x, int fmt)
{
    for (int64_t i = 0; i < M; ++i) {
        float amax = 0.0f;
        for (int64_t j = 0; j < K; ++j) {
            if (is_outlier[j])
                continue;
            float a = fabsf(elem_to_float(X[i * K + j], fmt));
            if (a > amax)
                amax = a;
        }
        s_x[i] = amax;
        float sf = oracle_scale_factor(amax);
        for (int64_t j = 0; j < K; ++j)
            Xq[i * K + j] = is_outlier[j] ? 0 : oracle_code(elem_to_float(X[i * K + j], fmt), sf);
    }
}

void oracle_quantize_rows(const uint16_t *X, int64_t M, int64_t K, const uint8_t *is_outlier,
                          int8_t *Xq, float *s_x)
{
    oracle_quantize_rows_fmt(X, M, K, is_outlier, Xq, s_x, 0);
}

/* ---------------------------------------------------------------------------
 * Row-parallel driver: rows are independent, so each thread takes a contiguous
 * block of rows and computes them with exactly the same loop as one thread.
 * ------------------------------------------------------------------------- */
typedef void (*row_fn)(void *ctx, int64_t r0, int64_t r1);
typedef struct {
    row_fn fn;
    void *ctx;
    int64_t r0, r1;
} row_job;

static void *row_job_run(void *p)
{
    row_job *j = (row_job *)p;
    j->fn(j->ctx, j->r0, j->r1);
    return NULL;
}

static void for_rows(row_fn fn, void *ctx, int64_t M, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > M)
        nthreads = (int)(M > 0 ? M : 1);
    if (nthreads == 1) {
        fn(ctx, 0, M);
        return;
    }
    pthread_t th[256];
    row_job jobs[256];
    int joined[256];
    int64_t per = (M + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t r0 = t * per, r1 = r0 + per < M ? r0 + per : M;
        joined[t] = 0;
        if (r0 >= r1)
            continue;
        jobs[t] = (row_job){fn, ctx, r0, r1};
        if (pthread_create(&th[t], NULL, row_job_run, &jobs[t]) == 0)
            joined[t] = 1;
        else
            row_job_run(&jobs[t]); /* no thread available: run it here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (joined[t])
            pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------------
 * A3. int8 x int8 -> integer matmul over all K ([FABRIC] section 2.2: int8
 * operands, integer result; [WALK] section 2.3: X_normal . W_normal in int8).
 * Accumulated in int64, so the result is exact for any K.  The outlier columns
 * of Xq are zero, so summing over all K equals summing over the non-outlier
 * columns.
 * ------------------------------------------------------------------------- */
typedef struct {
    const int8_t *Xq, *Wq;
    int64_t K, N;
    int64_t *C;
} imm_ctx;

static void imm_rows(void *p, int64_t r0, int64_t r1)
{
    imm_ctx *c = (imm_ctx *)p;
    for (int64_t i = r0; i < r1; ++i)
        for (int64_t n = 0; n < c->N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < c->K; ++k)
                acc += (int64_t)c->Xq[i * c->K + k] * (int64_t)c->Wq[k * c->N + n];
            c->C[i * c->N + n] = acc;
        }
}

void oracle_int8_matmul(const int8_t *Xq, const int8_t *Wq, int64_t M, int64_t K, int64_t N,
                        int64_t *C, int nthreads)
{
    imm_ctx c = {Xq, Wq, K, N, C};
    for_rows(imm_rows, &c, M, nthreads);
}

/* ---------------------------------------------------------------------------
 * A4. fp16 product of the outlier slice ([WALK] section 2.3: X_outlier and the
 * matching rows of W stay in 16-bit and are multiplied without quantization;
 * [PITFALLS] section 3.2: the outlier part is multiplied separately in 16-bit).
 * F[i,n] = sum over outlier columns k of X[i,k] * W[k,n], in double.
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *X, *W;
    const uint8_t *is_outlier;
    int64_t K, N;
    double *F;
    int fmt;
} omm_ctx;

static void omm_rows(void *p, int64_t r0, int64_t r1)
{
    omm_ctx *c = (omm_ctx *)p;
    for (int64_t i = r0; i < r1; ++i)
        for (int64_t n = 0; n < c->N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < c->K; ++k)
                if (c->is_outlier[k])
                    acc += elem_to_double(c->X[i * c->K + k], c->fmt) *
                           elem_to_double(c->W[k * c->N + n], c->fmt);
            c->F[i * c->N + n] = acc;
        }
}

void oracle_outlier_matmul_fmt(const uint16_t *X, const uint16_t *W, const uint8_t *is_outlier,
                               int64_t M, int64_t K, int64_t N, double *F, int nthreads, int fmt)
{
    omm_ctx c = {X, W, is_outlier, K, N, F, fmt};
    for_rows(omm_rows, &c, M, nthreads);
}

void oracle_outlier_matmul(const uint16_t *X, const uint16_t *W, const uint8_t *is_outlier,
                           int64_t M, int64_t K, int64_t N, double *F, int nthreads)
{
    oracle_outlier_matmul_fmt(X, W, is_outlier, M, K, N, F, nthreads, 0);
}

/* ---------------------------------------------------------------------------
 * A4 without a full fp16 copy of W: the dequantized weight.  Dequantization
 * multiplies a code by its scale ([PITFALLS] section 1 recovers the values
 * from the codes; [FABRIC] section 2.2: one scale per output column), here
 * absmax/127 since the scale is stored as the absmax.  When only the int8
 * codes of W are kept, an outlier row k of W is taken as
 *   w_hat[k,n] = fp16( fp32(q[k,n]) * fp32(s_w[n] / 127) ),
 * each fp32 operation rounded once to nearest even, then rounded to fp16 (the
 * operand precision of the outlier product).  s_w = 0 gives 0.
 * ------------------------------------------------------------------------- */
void oracle_dequantize_weight_fmt(const int8_t *Wq, const float *s_w, int64_t K, int64_t N, uint16_t *W_hat,
                                  int fmt)
{
    for (int64_t n = 0; n < N; ++n) {
        float r = s_w[n] / 127.0f;
        for (int64_t k = 0; k < K; ++k) {
            float p = (float)Wq[k * N + n] * r;
            W_hat[k * N + n] = double_to_elem((double)p, fmt);
        }
    }
}

void oracle_dequantize_weight(const int8_t *Wq, const float *s_w, int64_t K, int64_t N, uint16_t *W_hat)
{
    oracle_dequantize_weight_fmt(Wq, s_w, K, N, W_hat, 0);
}

/* ---------------------------------------------------------------------------
 * A5. Dequantize and merge ([PITFALLS] section 3.3: dequantize the 8-bit result,
 * then ADD the 16-bit result; [FABRIC] section 2.2: rescale the integer result
 * by scale_x * scale_w).  With s_x and s_w stored as absmax values, each code
 * carries a factor absmax/127, so the integer result is scaled by
 * s_x[i] * s_w[n] / 127^2.  Done in double, then rounded to fp16 (RNE).
 * ------------------------------------------------------------------------- */
void oracle_merge_fmt(const int64_t *C, const float *s_x, const float *s_w, const double *F,
                      int64_t M, int64_t N, uint16_t *Y, int fmt)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t n = 0; n < N; ++n) {
            double deq = (double)C[i * N + n] * (double)s_x[i] * (double)s_w[n] / 16129.0;
            double y = deq + (F ? F[i * N + n] : 0.0);
            Y[i * N + n] = double_to_elem(y, fmt);
        }
}

void oracle_merge(const int64_t *C, const float *s_x, const float *s_w, const double *F,
                  int64_t M, int64_t N, uint16_t *Y)
{
    oracle_merge_fmt(C, s_x, s_w, F, M, N, Y, 0);
}
