/*
 * qmv.h -- C ABI of the block-quantised weight x activation product used by
 * single-stream LLM decode, for one NVIDIA GB300 (sm_103a).
 *
 * The operation, for every call below (one token's decode step multiplies its
 * activation row by each weight matrix in turn -- H100-KERNEL-5X-ROADMAP,
 * "Why the decode gap is bandwidth, not arithmetic"):
 *
 *     y[m][n] = sum_k x[m][k] * w[n][k],   0 <= m < M, 0 <= n < N, 0 <= k < K
 *
 * where w is the dequantised weight matrix W[N x K].
 *
 * Weight layout (GGUF; "Q4_0", "group_size 32" -- sm8x-bench, Q4_0 summary and
 * "Our kernel does what llama.cpp does"; Q8_0 -- H100-KERNEL-5X-ROADMAP, "The
 * measured baseline"):
 *   - W is row-major: row n is K/32 consecutive blocks, rows are dense
 *     (row stride = (K/32) * block bytes, no padding).
 *   - Q4_0 block = 18 bytes: fp16 scale d (little endian) then 16 bytes qs;
 *     element j < 16 is the low nibble of qs[j], element j >= 16 the high
 *     nibble of qs[j-16]; w = (c - 8) * d.
 *   - Q8_0 block = 34 bytes: fp16 scale d then 32 int8 codes q; w = q * d.
 * Activations x: fp16, row-major [M][K].  Output y: fp32, row-major [M][N],
 * overwritten (never accumulated into).  Accumulation is fp32.
 *
 * Accuracy contract: per output, |y - y_exact| <= 2e-3 * (sum_k |x w| + 1e-6),
 * with y_exact the fp64 dequantise-then-dot (volta-kernel-bakeoff, "Making it
 * fair": CPU double-precision reference; "A few tokens at once": checked like
 * cuBLAS fp16, 2e-3, large and tiny activations planted).  This bound is the
 * acceptance bar on activations like the pages' (N(0,1), their large plant of
 * +-20000..60000 and tiny plant of x 1e-4) and on whole blocks of +-65504.
 * What holds for every input follows from the arithmetic of the decode
 * kernels, which sum eight products per fp16 partial sum with weights
 * pre-scaled to |w'| <= 1/8 (Q4_0: (c - 8)/64, Q8_0: q/1024; 2-bit: 1/16):
 *   - for finite fp16 activations and finite scales every output is finite:
 *     no fp16 partial sum can overflow (after eight products of at most
 *     65504/8 each, round-to-nearest stays at or below 65504);
 *   - |y - y_exact| <= about 2^-8 * sum_k |x w| + 2^-25 * P * K * max |d|,
 *     P the pre-scale (64, 1024, 32): eight fp16 roundings of at most 2^-11
 *     of a partial sum each, plus at most half a subnormal step (2^-25) per
 *     rounding when products fall below fp16's normal range.
 * Activations must be finite fp16.  Exceptions, each stated at its
 * declaration: the *_f32 calls take fp32 activations (rounded to fp16 in the
 * kernel), the *_q8_1 calls compute the product on the activations quantised
 * to Q8_1 (their own accuracy statement), and the prefill calls -- and the
 * several-token Q4_0 / Q8_0 decode calls that run on the tensor cores (at
 * qmv_q4_0) -- round each dequantised weight to fp16 and sum its products in
 * fp32 (so |d| <= 8188 for Q4_0, |d| <= 511 for Q8_0 keeps every weight
 * finite; within the 2e-3 bar above).
 *
 * Conventions common to every entry point:
 *   - All array pointers are DEVICE pointers on the current CUDA device, owned
 *     by the caller; the library never allocates, frees or retains them.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they enqueue work on `stream` and return; the host never
 *     blocks (except qmv_device_status, which synchronises `stream`).
 *   - Argument errors are reported before anything is enqueued.  Errors found
 *     on the device (an expert index out of range) are recorded in a device
 *     status word read by qmv_device_status(); the kernel never traps.
 *   - N == 0 or M == 0: nothing to do, QMV_OK, nothing enqueued.
 *     K == 0: y is filled with zeros (an empty sum).
 *   - The library is thread-safe for concurrent calls on different streams.
 *   - Weights are read-only inputs.  By default the decode and prefill kernels
 *     use programmatic dependent launch: a call may begin streaming (and, for
 *     prefill, dequantising) W while the previous kernel on `stream` is still
 *     finishing, and reads x / writes y only after that kernel has completed.
 *     So W must not be written by the kernel that runs immediately before a
 *     call on the same stream; if it is (in-place re-quantisation, a weight
 *     loader), call qmv_set_pdl(0) first.  Every declaration below that takes
 *     W is subject to this condition.
 */
#ifndef QMV_H
#define QMV_H

#include <stdint.h>

#if defined(__GNUC__)
#define QMV_API __attribute__((visibility("default")))
#else
#define QMV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *qmv_stream_t;

typedef enum {
    QMV_OK = 0,
    QMV_ERR_NULL = 1,      /* a required pointer is NULL                        */
    QMV_ERR_ALIGN = 2,     /* W not 16-byte aligned, x not 2-byte, y not 4-byte */
    QMV_ERR_SHAPE = 3,     /* N, K, M or a count out of range, K % 32 != 0      */
    QMV_ERR_LAUNCH = 4,    /* the CUDA launch failed (cudaGetLastError)         */
    QMV_ERR_DEVICE = 5,    /* a device-side error was recorded                  */
    QMV_ERR_CUDA = 6       /* another CUDA runtime call failed                  */
} qmv_status;

/* Device status word bits (qmv_device_status). */
#define QMV_DEV_BAD_EXPERT  0x1   /* an expert index was outside [0, n_experts) */
#define QMV_DEV_TIMEOUT     0x2   /* a bounded wait in a kernel gave up          */

/*
 * Q4_0 decode GEMV.  Prior art: the bakeoff's fused_q4 kernels (a warp per
 * row, codes unpacked in registers, fp32 sums; v2 builds halves from codes by
 * OR-ing them into the 0x6400 pattern -- volta-kernel-bakeoff, "What's in the
 * race") and the sm8x kernel (several rows per warp to keep more loads in
 * flight, launch shape chosen per table -- sm8x-bench, summary).
 *   W : Q4_0 bytes [N][K/32*18], 16-byte aligned.
 *   x : fp16 [M][K], 2-byte aligned.        y : fp32 [M][N], 4-byte aligned.
 *   N >= 0, K >= 0 with K % 32 == 0, 0 <= M <= 8.
 * K % 256 == 0 (16-byte aligned rows) with x 16-byte aligned takes the
 * streaming kernel; other K or alignments take a slower generic kernel with
 * the same results contract.  When the activations of all M tokens do not fit
 * in shared memory (e.g. 8 tokens of K = 14336 in fp16) the call runs as a
 * few launches over token subsets, each streaming W again.  These rules hold
 * for every decode call below.
 * Several tokens on the tensor cores (qmv_q4_0 and qmv_q8_0 only): with
 * K % 256 == 0 and W, x 16-byte aligned, calls of 8 tokens, and of 4..7 tokens
 * with K >= 2560, run on the prefill kernel's 16-token tiles (the weights
 * dequantised into tensor memory, fp32 accumulation; split along K over a
 * cluster of up to 8 CTAs where the 128-row tiles alone would leave SMs idle,
 * the partial tiles added in a fixed order).  Measured on the GB300 they are
 * faster there (e.g. Q8_0 12288x2560 at eight tokens 21.9 -> 13.0 us, Q4_0
 * 4096x14336 43.4 -> 15.3 us); the weight rounding is that of the prefill
 * call (the preamble).
 * W must not be written by the kernel right before this call on `stream`
 * while programmatic dependent launch is on (see the preamble).
 */
QMV_API qmv_status qmv_q4_0(const void *W, const void *x, float *y,
                    int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Q8_0 decode GEMV, same contract as qmv_q4_0 with 34-byte Q8_0 blocks (the
 * bakeoff's fused_q8 contender streams 8-bit weights -- volta-kernel-bakeoff,
 * "What's in the race"; k_q8_gemm -- H100-KERNEL-5X-ROADMAP, "Lever 1").
 *   W : Q8_0 bytes [N][K/32*34], 16-byte aligned.  0 <= M <= 8.
 */
QMV_API qmv_status qmv_q8_0(const void *W, const void *x, float *y,
                    int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Q4_0 decode GEMV against activations quantised to Q8_1, with integer dots
 * (the sm8x kernel and llama.cpp convert the activations to 8-bit blocks once
 * and take the Q4_0 dot with dp4a on nibbles masked by 0x0F0F0F0F --
 * sm8x-bench, "Our kernel does what llama.cpp does").  Here each CTA quantises
 * the activations while it stages them: no separate quantisation launch.
 *   W, y, N, K, M (<= 8), errors and asynchrony as for qmv_q4_0; x fp16 [M][K].
 * The activations are replaced by Q8_1 blocks (see qmv_quantize_q8_1), so the
 * result is the product on the quantised activations:
 *     y[m][n] = sum over blocks b of d_w * d_x[m][b] * sum_i (c_i - 8) * q[m][i],
 * which differs from the exact product by up to sum_k |w| * (d/2 + |q| * |fp16(d) - d|)
 * per output (d the block's fp32 scale).  Against that quantised product the
 * kernel's only rounding is the fp32 accumulation of the per-block terms.
 */
QMV_API qmv_status qmv_q4_0_q8_1(const void *W, const void *x, float *y,
                         int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Q8_1 quantisation of fp16 activations, exactly as qmv_q4_0_q8_1 and
 * qmv_q8_0_q8_1 perform it inside their kernel: per block of 32 values of a row, in fp32 with
 * round-to-nearest, amax = max |x|, d = amax / 127, id = 1 / d (0 for an
 * all-zero block) and q = round(x * id) with ties away from zero; the block's
 * scale is d rounded to fp16.  Values must be finite.
 *   x      : DEVICE fp16 [M][K], 16-byte aligned; K % 32 == 0.
 *   q      : DEVICE int8 [M][K] (8-byte aligned), the codes.
 *   d_bits : DEVICE uint16 [M][K/32] (2-byte aligned), the fp16 scales' bits.
 *   sumq   : DEVICE int32 [M][K/32] (4-byte aligned), each block's code sum.
 * (llama.cpp's Q8_1 block stores d and d * sum(q) beside its 32 codes; these
 * are the same quantities in three plain arrays.)
 * Asynchronous on `stream`; with programmatic dependent launch on, the next
 * call of this library may start streaming its weights while this one runs and
 * reads the codes only after it has completed.
 */
QMV_API qmv_status qmv_quantize_q8_1(const void *x, int8_t *q, uint16_t *d_bits, int32_t *sumq,
                             int64_t M, int64_t K, qmv_stream_t stream);

/*
 * qmv_q4_0_q8_1 with the activations already in Q8_1 (as qmv_quantize_q8_1
 * writes them): the two steps of the sm8x kernel and llama.cpp, quantise once
 * and then take the int8 dot against several tables that share the
 * activations.  The result equals qmv_q4_0_q8_1 on the fp16 activations those
 * blocks came from, bit for bit.
 *   q      : DEVICE int8 [M][K], 16-byte aligned (K % 256 == 0 for the
 *            streaming kernel; other K run the generic kernel).
 *   d_bits : DEVICE uint16 [M][K/32] (fp16 scales), 2-byte aligned.
 *   sumq   : DEVICE int32 [M][K/32] (code sums), 4-byte aligned.
 *   W, y, N, K, M (<= 8), errors and asynchrony as for qmv_q4_0.
 */
QMV_API qmv_status qmv_q4_0_q8_1_pre(const void *W, const int8_t *q, const uint16_t *d_bits, const int32_t *sumq,
                             float *y, int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Q8_0 decode GEMV against activations quantised to Q8_1, with signed integer
 * dots.  The pages give the Q8_1 integer dot for Q4_0 weights only
 * (sm8x-bench, "Our kernel does what llama.cpp does"); this call carries it to
 * Q8_0, whose codes are already signed bytes, so a block's dot is a plain
 * int8 x int8 sum with no nibble split and no code-sum correction:
 *     y[m][n] = sum over blocks b of d_w * d_x[m][b] * sum_i c_i * q[m][i].
 * Quantisation of the activations, error bound against the exact product and
 * the kernel's rounding as for qmv_q4_0_q8_1.
 *   W : Q8_0 bytes [N][K/32*34], 16-byte aligned; x fp16 [M][K].
 *   y, N, K, M (<= 8), errors and asynchrony as for qmv_q8_0.
 */
QMV_API qmv_status qmv_q8_0_q8_1(const void *W, const void *x, float *y,
                         int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * qmv_q8_0_q8_1 with the activations already in Q8_1 (as qmv_quantize_q8_1
 * writes them; the code sums are not needed).  Equal to qmv_q8_0_q8_1 on the
 * fp16 activations those blocks came from, bit for bit.
 *   q      : DEVICE int8 [M][K], 16-byte aligned (K % 256 == 0 for the
 *            streaming kernel; other K run the generic kernel).
 *   d_bits : DEVICE uint16 [M][K/32] (fp16 scales), 2-byte aligned.
 *   W, y, N, K, M (<= 8), errors and asynchrony as for qmv_q8_0.
 */
QMV_API qmv_status qmv_q8_0_q8_1_pre(const void *W, const int8_t *q, const uint16_t *d_bits,
                             float *y, int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Plain 2-bit decode GEMV (the bakeoff's q2w format: codes -2..1 with one fp16
 * scale per 32 weights, 2.5 bits per weight -- volta-kernel-bakeoff, "What's
 * in the race" and the Results table's 2-bit column), same contract as
 * qmv_q4_0 with 10-byte blocks:
 *   W : [N][K/32*10] bytes, 16-byte aligned; a block is fp16 d (little
 *       endian) then qs[0..7]; element j of the block is bits 2*(j/8) and
 *       2*(j/8)+1 of qs[j % 8], an unsigned c in 0..3, and w = (c - 2) * d.
 *       (The pages leave the bit order open; this is Q4_0's split of a byte
 *       into elements j and j+16 carried one step further.)
 *   0 <= M <= 8; K % 256 == 0 takes the streaming kernel, other K the
 *   generic one.
 */
QMV_API qmv_status qmv_q2w(const void *W, const void *x, float *y,
                   int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Several experts, each with its own token, in ONE launch (the bakeoff's moe_*
 * contenders run 8 to 10 experts this way -- volta-kernel-bakeoff, "What's in
 * the race"; every expert gets distinct weights and its own token, so that a
 * wrong index shows up as a wrong result -- "Making it fair").
 *   W_pool     : n_experts Q4_0 experts of N x K each, back to back
 *                (expert e starts at byte e * N * (K/32) * 18), 16-byte aligned.
 *   expert_idx : DEVICE int32 [M]; slot s uses expert expert_idx[s].
 *                Duplicates are allowed.
 *   x          : fp16 [M][K] (row s = token of slot s).
 *   y          : fp32 [M][N] (row s = output of slot s).
 *   1 <= n_experts, 0 <= M <= 64.
 * An index outside [0, n_experts) sets QMV_DEV_BAD_EXPERT in the device status
 * word and fills that slot's row of y with NaN; other slots are unaffected.
 * Row s of y is bit-identical to qmv_q4_0 on expert expert_idx[s] with token
 * x[s] (same inner loop and reduction order).
 */
QMV_API qmv_status qmv_moe(const void *W_pool, const int32_t *expert_idx, int64_t n_experts,
                   const void *x, float *y, int64_t N, int64_t K, int64_t M,
                   qmv_stream_t stream);

/*
 * The MLP's gate + up + SwiGLU in one call (decode, 1..8 tokens): two Q4_0
 * tables that share the activations, read together, with the activation
 * function applied before anything is written --
 *     y[m][n] = silu(g) * u,  g = sum_k x[m][k] wg[n][k],  u = sum_k x[m][k] wu[n][k],
 *     silu(g) = g / (1 + e^-g)
 * (the bakeoff treats gate and up as one stacked table with a single pass
 * over the activations -- volta-kernel-bakeoff, "A few tokens at once"; the
 * diary's phase-6 kernel fuses W1, W3 and SwiGLU so that the activations are
 * read once and only the activated output is stored -- SovereignKernel diary,
 * phase 6).  The two tables stay separate arrays; the kernel interleaves their
 * rows as it streams them.
 *   W_gate, W_up : Q4_0 bytes [N][K/32*18] each, 16-byte aligned (W_up may
 *                  be NULL only when K == 0).
 *   x : fp16 [M][K].  y : fp32 [M][N] (overwritten).  M <= 8.
 * Accuracy: g and u each carry the product's bound above; through silu,
 * |y - y_exact| <= 2e-3 * (1.1 * Sg * (|u| + 2e-3 * Su) + |silu(g)| * Su)
 * with Sg, Su the two products' sums of |x w| (1.1 bounds |silu'|).
 * Errors and asynchrony as for qmv_q4_0.
 */
QMV_API qmv_status qmv_q4_0_swiglu(const void *W_gate, const void *W_up, const void *x, float *y,
                           int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * qmv_q4_0 and qmv_q4_0_swiglu with fp32 activations (the bakeoff's
 * fused_q4_v3_fp32in takes fp32 in and counts the narrowing to fp16 in its
 * time -- volta-kernel-bakeoff, "Results (one token, microseconds, lower is
 * better)" and "A few tokens at once").  The narrowing happens inside the
 * kernel, while each CTA stages the activations into shared memory, at every
 * token count: no separate conversion launch and no fp16 copy in memory.
 *   x : fp32 [M][K], 4-byte aligned (16-byte aligned with K % 256 == 0 for the
 *       streaming kernel; otherwise the generic kernel runs).  Every value is
 *       rounded to fp16 (nearest even) before the product, so the results
 *       equal those of qmv_q4_0 / qmv_q4_0_swiglu on x rounded to fp16
 *       (bit-identical: the same kernel runs after staging), except where
 *       qmv_q4_0 takes the tensor cores (several tokens, at qmv_q4_0): this
 *       call always streams, and the two then agree within the accuracy
 *       bound.  Values must lie
 *       within fp16's range (|x| < 65520): larger ones round to +-inf.
 *   W, W_gate, W_up, y, N, K, M, errors and asynchrony as for the fp16 calls.
 * Accuracy against the exact product on the fp32 values: the bounds above,
 * which also cover the rounding of x (at most 2^-11 of each |x w|).
 */
QMV_API qmv_status qmv_q4_0_f32(const void *W, const float *x, float *y,
                        int64_t N, int64_t K, int64_t M, qmv_stream_t stream);
QMV_API qmv_status qmv_q4_0_swiglu_f32(const void *W_gate, const void *W_up, const float *x, float *y,
                               int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Q4_0 prefill GEMM for many tokens (M >= 1, intended for M >= 64).  Prior
 * art: the bakeoff's tc_q4, which dequantises a tile into shared memory for the
 * tensor cores (volta-kernel-bakeoff, "What's in the race"), and the plan to
 * dequantise inside the tensor-core multiply ("What we'd do next", item 3).
 * On sm_103a: packed
 * W tiles staged by bulk copies, dequantised to fp16 straight into tensor
 * memory, where tcgen05.mma reads them beside its fp32 accumulators.
 *   W : Q4_0 bytes [N][K/32*18], 16-byte aligned.  The tensor-core kernel
 *       takes K % 256 == 0 (any N: a ragged last 128-row tile is masked);
 *       other K take the generic kernel.
 *   x : fp16 [M][K], 16-byte aligned.  y : fp32 [M][N].
 *   0 <= M <= 2^24 (QMV_ERR_SHAPE above).  Above 65535 * 256 tokens the
 *   token tiles would exceed the grid's y limit, and the generic kernel takes
 *   the call.
 * Calls of up to 16 tokens run on 16-token tiles, split along K over a
 * cluster of up to 8 CTAs where the 128-row tiles alone would leave SMs idle
 * (the same launch as the several-token decode calls above).
 * W must not be written by the kernel right before this call on `stream`
 * while programmatic dependent launch is on (see the preamble).
 */
QMV_API qmv_status qmm_q4_0_prefill(const void *W, const void *x, float *y,
                            int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * The same many-token GEMM for Q8_0 weights (the roadmap's measured Q8_0
 * baseline -- roadmap, "The measured baseline" -- taken to many tokens): each
 * 34-byte block's int8 codes times its fp16 scale, rounded once to fp16, in
 * tensor memory; fp32 accumulation.
 *   W : Q8_0 bytes [N][K/32*34], 16-byte aligned.  The tensor-core kernel
 *       takes K % 256 == 0; other K take the generic kernel.
 *   x, y, M, errors and asynchrony as for qmm_q4_0_prefill.
 * W must not be written by the kernel right before this call on `stream`
 * while programmatic dependent launch is on (see the preamble).
 */
QMV_API qmv_status qmm_q8_0_prefill(const void *W, const void *x, float *y,
                            int64_t N, int64_t K, int64_t M, qmv_stream_t stream);

/*
 * Reads and clears the device status word (QMV_DEV_* bits) of the current
 * device, in one atomic step enqueued on `stream` (so it follows every kernel
 * enqueued before it on `stream`; a bit that a kernel on another stream sets
 * meanwhile is kept for the next read, never lost).  Synchronises `stream`.
 * *out receives the bits.  Returns QMV_ERR_NULL for out == NULL, QMV_ERR_CUDA
 * or QMV_ERR_LAUNCH on a runtime error.
 */
QMV_API qmv_status qmv_device_status(qmv_stream_t stream, int32_t *out);

/*
 * Read-only bandwidth probe (a measurement utility, not part of the product):
 * streams `bytes` of device memory through per-warp shared-memory rings filled
 * by bulk (TMA) copies, the way the decode kernels stream their weights, with
 * no arithmetic on the bytes.  Timing it over a buffer several times the L2
 * gives the read roofline the decode kernels are compared with, beside the
 * copy bandwidth (sm8x-bench reports its kernels against a measured bandwidth
 * probe as well as the spec figure -- sm8x-bench, methodology bullets).
 *   buf   : DEVICE, 16-byte aligned, `bytes` long; bytes % 256 == 0.
 *   out   : DEVICE uint32, 4-byte aligned: receives the XOR, over every
 *           256-byte-aligned offset o < bytes, of the four 32-bit little-endian
 *           words at buf + o .. o + 15 (proof that the bytes were consumed).
 * Asynchronous on `stream`; bytes == 0 writes 0.  QMV_ERR_SHAPE for a
 * negative or unaligned size, QMV_ERR_NULL / QMV_ERR_ALIGN as usual.
 */
QMV_API qmv_status qmv_read_probe(const void *buf, int64_t bytes, uint32_t *out, qmv_stream_t stream);

/* Programmatic dependent launch for the decode, prefill and Q8_1 quantisation
 * kernels: 1 = on (default), 0 = off (plain stream order).  Process-wide;
 * affects later calls. */
QMV_API void qmv_set_pdl(int enable);

/* Static description of a status code. */
QMV_API const char *qmv_status_str(qmv_status s);

/* Library version, e.g. "qmv 0.1.0 sm_103a". */
QMV_API const char *qmv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
