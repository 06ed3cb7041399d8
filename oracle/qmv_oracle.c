/*
 * qmv_oracle.c -- CPU fp64 oracle for the block-quantised weight x activation
 * product of single-stream decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  The CUDA library never
 * links, includes or calls it, and it shares no code, header or table with the
 * CUDA path.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *     y[m][n] = sum_k  x[m][k] * w[n][k]             (fp64)
 *     S[m][n] = sum_k |x[m][k] * w[n][k]|            (fp64, for the tolerance)
 *
 * Every kernel is checked against an fp64 CPU product over the same quantised
 * weights before it is timed (volta-kernel-bakeoff, "Making it fair").  A
 * decode step of one token is a sequence of such matrix-vector products, one
 * per weight matrix (H100-KERNEL-5X-ROADMAP, "Why the decode gap is
 * bandwidth, not arithmetic").
 *
 * Weight formats (GGUF; "Q4_0", "group_size 32" -- sm8x-bench, Q4_0 summary
 * and "Our kernel does what llama.cpp does"; Q8_0 -- H100-KERNEL-5X-ROADMAP,
 * "The measured baseline"):
 *   Q4_0 block, 18 bytes, 32 weights:  bytes 0..1 = fp16 scale d (little
 *     endian), bytes 2..17 = qs[0..15].  Element j<16 is the low nibble of
 *     qs[j], element j>=16 is the high nibble of qs[j-16]; w = (c - 8) * d.
 *   Q8_0 block, 34 bytes, 32 weights:  bytes 0..1 = fp16 d, bytes 2..33 =
 *     int8 codes q[0..31]; w = q * d.
 *   Plain 2-bit ("q2w": codes from -2 to 1 with an fp16 scale for every 32 weights, 2.5 bits
 *     per weight -- volta-kernel-bakeoff, "What's in the race", q2w_alu_v3),
 *     10 bytes, 32 weights: bytes 0..1 = fp16 d, bytes 2..9 = qs[0..7].  The
 *     pages fix the codes and the scale but not the bit order; it is read the
 *     way Q4_0 splits a byte (elements j and j+16), one step further: element
 *     j is bits 2*(j/8)..2*(j/8)+1 of qs[j % 8], an unsigned c in 0..3, so
 *     byte i holds elements i, i+8, i+16, i+24 from its low bits up; and
 *     w = (c - 2) * d.
 *   A row of W holds K/32 consecutive blocks; rows are dense (no padding).
 *   x is fp16 (IEEE binary16 bit patterns), row-major [M][K]; the _f32 entry
 *   points take fp32 activations instead (the bakeoff's fused_q4_v3_fp32in
 *   accepts fp32 and includes the narrowing in its time -- volta-kernel-
 *   bakeoff, "Results (one token, microseconds, lower is better)"), whose
 *   values enter the sums exactly: the product is defined on the activations
 *   the caller passes, and any narrowing a kernel does on the way is part of
 *   its rounding error, not of the definition.
 *
 * Parity pins: see tests/test_oracle.py (hand-computed fixtures under
 * tests/golden/, closed forms, invariants, exhaustive fp16 decode against
 * numpy, integer special cases against numpy matmul, planted mutations).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FMT_Q4_0 0
#define ORACLE_FMT_Q8_0 1
#define ORACLE_FMT_Q2W 2

/* IEEE 754 binary16 -> double, written out from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits; exponent 0 is
 * zero/subnormal (mantissa * 2^-24), exponent 31 is inf/NaN. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);
    } else if (expo == 31) {
        v = (mant == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25);
    }
    return sign ? -v : v;
}

/* float -> IEEE binary16, round to nearest with ties to even, written out from
 * the format's definition: |v| >= 65520 (the midpoint above 65504) is inf,
 * |v| < 2^-14 is a subnormal multiple of 2^-24, otherwise 10 mantissa bits
 * after the leading one.  The arithmetic is exact in double; rint rounds to
 * nearest even in the default rounding mode. */
uint16_t oracle_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    const double v = fabs((double)f);
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (v < ldexp(1.0, -14)) {
        const double n = rint(v * ldexp(1.0, 24));       /* 0..1024; 1024 is the smallest normal */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int e2;
    const double m = frexp(v, &e2);                       /* v = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                                       /* v = (2m) * 2^e, 2m in [1, 2) */
    double mant = rint((2.0 * m - 1.0) * 1024.0);
    if (mant >= 1024.0) { mant = 0.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)mant);
}

int64_t oracle_block_bytes(int fmt)
{
    if (fmt == ORACLE_FMT_Q4_0) return 18;
    if (fmt == ORACLE_FMT_Q8_0) return 34;
    if (fmt == ORACLE_FMT_Q2W) return 10;
    return -1;
}

/* Dequantise one Q4_0 block of 32 weights into w[0..31]. */
static void dequant_block_q4_0(const uint8_t *blk, double *w)
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    double d = oracle_half_to_double(dbits);
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 16; ++j) {
        int lo = qs[j] & 0x0f;
        int hi = qs[j] >> 4;
        w[j] = (double)(lo - 8) * d;
        w[j + 16] = (double)(hi - 8) * d;
    }
}

/* Dequantise one plain 2-bit block of 32 weights into w[0..31]. */
static void dequant_block_q2w(const uint8_t *blk, double *w)
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    double d = oracle_half_to_double(dbits);
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 32; ++j) {
        int c = (qs[j % 8] >> (2 * (j / 8))) & 3;
        w[j] = (double)(c - 2) * d;
    }
}

/* Dequantise one Q8_0 block of 32 weights into w[0..31]. */
static void dequant_block_q8_0(const uint8_t *blk, double *w)
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    double d = oracle_half_to_double(dbits);
    const int8_t *q = (const int8_t *)(blk + 2);
    for (int j = 0; j < 32; ++j) {
        w[j] = (double)q[j] * d;
    }
}

/* Dequantise row n of W (K weights) into w[0..K-1]. */
int oracle_dequant_row(int fmt, const uint8_t *W, int64_t n, int64_t K, double *w)
{
    int64_t bb = oracle_block_bytes(fmt);
    if (bb < 0 || K % 32 != 0) return -1;
    int64_t nblk = K / 32;
    const uint8_t *row = W + n * nblk * bb;
    for (int64_t b = 0; b < nblk; ++b) {
        if (fmt == ORACLE_FMT_Q4_0)
            dequant_block_q4_0(row + b * bb, w + 32 * b);
        else if (fmt == ORACLE_FMT_Q8_0)
            dequant_block_q8_0(row + b * bb, w + 32 * b);
        else
            dequant_block_q2w(row + b * bb, w + 32 * b);
    }
    return 0;
}

/* Activations widened to fp64 (exact for both fp16 and fp32). */
static double *widen_half(const uint16_t *x, int64_t n)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (xd)
        for (int64_t i = 0; i < n; ++i) xd[i] = oracle_half_to_double(x[i]);
    return xd;
}

static double *widen_float(const float *x, int64_t n)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (xd)
        for (int64_t i = 0; i < n; ++i) xd[i] = (double)x[i];
    return xd;
}

/* y and S for the listed rows, from fp64 activations xd[M][K]. */
static int qmv_rows_xd(int fmt, const uint8_t *W, const double *xd,
                       int64_t N, int64_t K, int64_t M,
                       const int64_t *rows, int64_t nrows,
                       double *y, double *S, int nthreads)
{
    int failed = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads) reduction(| : failed)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t n = rows ? rows[r] : r;
        double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!w || n < 0 || n >= N) { failed = 1; free(w); continue; }
        oracle_dequant_row(fmt, W, n, K, w);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = xd[m * K + k] * w[k];
                acc += p;
                sabs += fabs(p);
            }
            y[m * nrows + r] = acc;
            S[m * nrows + r] = sabs;
        }
        free(w);
    }
    (void)nthreads;
    return failed ? -3 : 0;
}

/* y and S for the rows listed in rows[0..nrows-1] (all rows when rows is NULL,
 * then nrows = N).  Outputs are [M][nrows] row-major. */
int oracle_qmv_rows(int fmt, const uint8_t *W, const uint16_t *x,
                    int64_t N, int64_t K, int64_t M,
                    const int64_t *rows, int64_t nrows,
                    double *y, double *S, int nthreads)
{
    if (oracle_block_bytes(fmt) < 0 || K % 32 != 0 || N < 0 || M < 0) return -1;
    if (rows == NULL) nrows = N;
    double *xd = widen_half(x, M * K);
    if (!xd) return -2;
    int rc = qmv_rows_xd(fmt, W, xd, N, K, M, rows, nrows, y, S, nthreads);
    free(xd);
    return rc;
}

/* oracle_qmv_rows with fp32 activations x[M][K]. */
int oracle_qmv_rows_f32(int fmt, const uint8_t *W, const float *x,
                        int64_t N, int64_t K, int64_t M,
                        const int64_t *rows, int64_t nrows,
                        double *y, double *S, int nthreads)
{
    if (oracle_block_bytes(fmt) < 0 || K % 32 != 0 || N < 0 || M < 0) return -1;
    if (rows == NULL) nrows = N;
    double *xd = widen_float(x, M * K);
    if (!xd) return -2;
    int rc = qmv_rows_xd(fmt, W, xd, N, K, M, rows, nrows, y, S, nthreads);
    free(xd);
    return rc;
}

/* Full product: y[M][N], S[M][N]. */
int oracle_qmv(int fmt, const uint8_t *W, const uint16_t *x,
               int64_t N, int64_t K, int64_t M, double *y, double *S, int nthreads)
{
    return oracle_qmv_rows(fmt, W, x, N, K, M, NULL, N, y, S, nthreads);
}

/* Several experts, one token each, in one call (the bakeoff's moe_*
 * contenders run 8 to 10 experts in a single launch -- volta-kernel-bakeoff,
 * "What's in the race"; each expert has distinct weights and its own token, so
 * a wrong index changes the result -- "Making it fair").
 * Slot s uses expert e = idx[s] of a pool of n_experts experts stored back to
 * back (expert e starts e * N * (K/32) blocks in), token x[s][0..K-1], and
 * writes y[s][0..N-1], S[s][0..N-1].  An index outside [0, n_experts) is an
 * error (returns -4, outputs of that slot untouched). */
int oracle_moe(int fmt, const uint8_t *W_pool, const int32_t *idx, int64_t n_experts,
               const uint16_t *x, int64_t N, int64_t K, int64_t n_slots,
               double *y, double *S, int nthreads)
{
    int64_t bb = oracle_block_bytes(fmt);
    if (bb < 0 || K % 32 != 0) return -1;
    int64_t expert_bytes = N * (K / 32) * bb;
    int rc = 0;
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = idx[s];
        if (e < 0 || e >= n_experts) { rc = -4; continue; }
        int r = oracle_qmv(fmt, W_pool + (int64_t)e * expert_bytes, x + s * K,
                           N, K, 1, y + s * N, S + s * N, nthreads);
        if (r != 0) return r;
    }
    return rc;
}

/* The MLP's gate + up + SwiGLU at decode, as one product over two tables that
 * share the activations (gate and up handled as one stacked table --
 * volta-kernel-bakeoff, "A few tokens at once"; W1, W3 and SwiGLU fused so the
 * activations are read once -- SovereignKernel diary, phase 6).  SwiGLU with
 * its usual swish: the gate product goes through
 * silu(g) = g / (1 + e^-g) and multiplies the up product:
 *
 *     g[m][n] = sum_k x[m][k] * wg[n][k]        u[m][n] = sum_k x[m][k] * wu[n][k]
 *     y[m][n] = silu(g[m][n]) * u[m][n]
 *
 * For the listed rows (all rows when rows is NULL, then nrows = N); every
 * output is [M][nrows] row-major and fp64: y, g, u and the S sums of the two
 * products (the tolerance of a fused result is derived from them). */
static int swiglu_rows_xd(int fmt, const uint8_t *Wg, const uint8_t *Wu, const double *xd,
                          int64_t N, int64_t K, int64_t M, const int64_t *rows, int64_t nrows,
                          double *y, double *g, double *u, double *Sg, double *Su, int nthreads)
{
    int rc = qmv_rows_xd(fmt, Wg, xd, N, K, M, rows, nrows, g, Sg, nthreads);
    if (rc != 0) return rc;
    rc = qmv_rows_xd(fmt, Wu, xd, N, K, M, rows, nrows, u, Su, nthreads);
    if (rc != 0) return rc;
    for (int64_t i = 0; i < M * nrows; ++i) {
        const double gate = g[i];
        y[i] = gate / (1.0 + exp(-gate)) * u[i];
    }
    return 0;
}

int oracle_swiglu_rows(int fmt, const uint8_t *Wg, const uint8_t *Wu, const uint16_t *x,
                       int64_t N, int64_t K, int64_t M, const int64_t *rows, int64_t nrows,
                       double *y, double *g, double *u, double *Sg, double *Su, int nthreads)
{
    if (oracle_block_bytes(fmt) < 0 || K % 32 != 0 || N < 0 || M < 0) return -1;
    if (rows == NULL) nrows = N;
    double *xd = widen_half(x, M * K);
    if (!xd) return -2;
    int rc = swiglu_rows_xd(fmt, Wg, Wu, xd, N, K, M, rows, nrows, y, g, u, Sg, Su, nthreads);
    free(xd);
    return rc;
}

/* oracle_swiglu_rows with fp32 activations x[M][K]. */
int oracle_swiglu_rows_f32(int fmt, const uint8_t *Wg, const uint8_t *Wu, const float *x,
                           int64_t N, int64_t K, int64_t M, const int64_t *rows, int64_t nrows,
                           double *y, double *g, double *u, double *Sg, double *Su, int nthreads)
{
    if (oracle_block_bytes(fmt) < 0 || K % 32 != 0 || N < 0 || M < 0) return -1;
    if (rows == NULL) nrows = N;
    double *xd = widen_float(x, M * K);
    if (!xd) return -2;
    int rc = swiglu_rows_xd(fmt, Wg, Wu, xd, N, K, M, rows, nrows, y, g, u, Sg, Su, nthreads);
    free(xd);
    return rc;
}

/* Activations quantised to 8 bits per block of 32 (Q8_1: llama.cpp and the
 * sm8x kernel convert the activations to this form once per call and then
 * take an int8 dot -- sm8x-bench, "Our kernel does what llama.cpp does").  For each
 * block of each token, in fp32 with round-to-nearest (the same precision the
 * kernel decides the codes in):
 *     amax = max |x_i|,  d = amax / 127,  id = 1 / d (0 when d = 0),
 *     q_i = round(x_i * id)   (ties away from zero),
 * and the block keeps d as fp16 (its stored scale) and sum_i q_i.
 * Outputs: q int8 [M][K], d_bits uint16 [M][K/32], sumq int32 [M][K/32]. */
int oracle_quantize_q8_1(const uint16_t *x, int64_t M, int64_t K, int8_t *q, uint16_t *d_bits, int32_t *sumq)
{
    if (K % 32 != 0 || M < 0) return -1;
    const int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t *xb = x + m * K + b * 32;
            float xf[32];
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                xf[i] = (float)oracle_half_to_double(xb[i]);
                const float a = fabsf(xf[i]);
                if (a > amax) amax = a;
            }
            const float d = amax / 127.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            int32_t s = 0;
            for (int i = 0; i < 32; ++i) {
                const float t = xf[i] * id;
                const int c = (int)roundf(t);
                q[m * K + b * 32 + i] = (int8_t)c;
                s += c;
            }
            d_bits[m * nb + b] = oracle_float_to_half(d);
            sumq[m * nb + b] = s;
        }
    }
    return 0;
}

/* The product with Q8_1 activations: y[m][n] = sum_k w[n][k] * q[m][k] * d[m][k/32]
 * with d the block's stored fp16 scale (the plain product on the activations
 * the quantised form stands for); S likewise with absolute values. */
int oracle_qmv_q8_1_rows(int fmt, const uint8_t *W, const int8_t *q, const uint16_t *d_bits,
                         int64_t N, int64_t K, int64_t M, const int64_t *rows, int64_t nrows,
                         double *y, double *S, int nthreads)
{
    if (oracle_block_bytes(fmt) < 0 || K % 32 != 0 || N < 0 || M < 0) return -1;
    if (rows == NULL) nrows = N;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!xd) return -2;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            xd[m * K + k] = (double)q[m * K + k] * oracle_half_to_double(d_bits[m * (K / 32) + k / 32]);
    int rc = qmv_rows_xd(fmt, W, xd, N, K, M, rows, nrows, y, S, nthreads);
    free(xd);
    return rc;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
