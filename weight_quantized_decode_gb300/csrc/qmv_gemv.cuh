// qmv_gemv.cuh -- the streaming decode GEMV for GGUF Q4_0 / Q8_0 on sm_103a,
// and the one-launch multi-expert variant built on the same inner loop.
//
// Design (GB300-first; the pages' V100/RTX-3090 kernels are prior art):
//   * Unit of work: 8 consecutive blocks of one row = 256 weights
//     (144 bytes Q4_0, 272 bytes Q8_0; both are whole multiples of 16 bytes,
//     so a unit is a run of aligned 128-bit words when K % 256 == 0).
//   * Each warp is its own streaming engine: it owns a ring of S shared-memory
//     stages and fills them with bulk (TMA) copies, one per row chunk, that
//     signal an mbarrier on arrival.  A stage holds RG = 32/G rows x SP*G units.
//   * Lane (r, q) of the warp (r = lane / G, q = lane % G) reads unit q (+G...)
//     of row r from the stage with 128-bit shared loads (a 144-/272-byte lane
//     stride is bank-conflict-free), unpacks nibbles/bytes with the fp16
//     0x6400|n trick, and accumulates half2 products per block, scaled to fp32
//     per block (the bakeoff's v2 unpack and its v2w variant, which takes a
//     full 32-weight block per lane step -- volta-kernel-bakeoff, "What's in
//     the race").
//   * G lanes per row, RG = 32/G rows per warp (several rows per warp keep
//     more loads in flight, and the launch shape is chosen per table --
//     sm8x-bench, summary); the G partial sums of a row are combined with warp
//     shuffles (the diary's kernel gives a whole warp to each row and reduces
//     it with shuffles -- SovereignKernel diary, Phase 3): xor butterflies when G is a power of
//     two; a G that does not divide 32 (a tuning choice, e.g. G = 10 for rows
//     of 10 units) leaves lanes RG*G.. idle and sums the G partials in lane
//     order.
//   * Activations live in shared memory for the whole call, permuted once per
//     CTA into the pair order the unpack produces and padded so that the G
//     distinct units a warp reads at once fall in distinct banks.  For M > 1
//     one unpacked weight register serves all M tokens (the bakeoff's
//     few-token kernel reuses each load across rows and tokens --
//     volta-kernel-bakeoff, "A few tokens at once").
//   * Rows are split across CTAs in balanced contiguous ranges; within a CTA
//     the row groups are dealt to warps round-robin.
//   * Programmatic dependent launch: the first S stages of W are requested
//     before griddepcontrol.wait; x is read and y written only after it.
#pragma once

#include "qmv_common.cuh"

namespace qmv {

enum Fmt : int { kQ4_0 = 0, kQ8_0 = 1, kQ2W = 2 };

template <int FMT>
struct FmtTraits;

template <>
struct FmtTraits<kQ4_0> {
    static constexpr int kBlockBytes = 18;
    static constexpr int kUnitBytes = 144;    // 8 blocks
    static constexpr int kUnitWords = 36;
    static constexpr float kPrescale = kQ4Prescale;
};

template <>
struct FmtTraits<kQ8_0> {
    static constexpr int kBlockBytes = 34;
    static constexpr int kUnitBytes = 272;
    static constexpr int kUnitWords = 68;
    static constexpr float kPrescale = kQ8Prescale;
};

// Plain 2-bit: fp16 d then 8 code bytes per 32 weights (2.5 bits per weight).
template <>
struct FmtTraits<kQ2W> {
    static constexpr int kBlockBytes = 10;
    static constexpr int kUnitBytes = 80;
    static constexpr int kUnitWords = 20;
    static constexpr float kPrescale = kQ2Prescale;
};

constexpr int kUnitWeights = 256;
constexpr int kXUnitBytes = 528;   // 512 bytes of permuted activations + 16 bytes pad
// Q8_1 activations: per unit the 256 codes of its 8 blocks in element order,
// then per block (fp32 scale, 8 * code sum), then 16 bytes pad (336 = 5 * 16
// mod 128: the G units a warp reads at once fall in distinct banks).
constexpr int kXQ8UnitBytes = 336;

struct GemvParams {
    const uint8_t *W;            // weights; for the multi-expert call, the expert pool; fused SwiGLU: gate
    const uint8_t *W2;           // fused SwiGLU: the up table (else nullptr)
    const __half *x;             // [n_problems * M][K] fp16 activations
    const float *xf;             // fp32 activations of the same shape (XF32 kernels; x is then unused)
    float *y;                    // [n_problems * M][N]
    const int32_t *expert_idx;   // multi-expert call only (else nullptr)
    int64_t N;                   // rows per problem
    int64_t K;
    int64_t n_experts;
    int64_t row_bytes;           // (K/32) * block bytes
    int64_t rows_total;          // n_problems * N
    int n_problems;              // 1 for a plain GEMV, slots for the multi-expert call
    int max_local_problems;      // most problems one CTA's row range can touch
    int U;                       // units per row = K / 256
    int G;                       // lanes per row (1..32; RG = 32 / G rows per warp)
    int SP;                      // passes per stage (odd)
    int S;                       // stages in each warp's ring
    int early;                   // stages requested before griddepcontrol.wait (the rest after the
                                 // activation loads); the multi-expert call requests none early
    int xq8;                     // Q4_0 or Q8_0 against Q8_1-quantised activations (integer dots)
    const int8_t *xq;            // activations already in Q8_1 (codes [M][K]); else quantised in the kernel
    const uint16_t *xq_d;        //   their fp16 scales' bits [M][K/32]
    const int32_t *xq_s;         //   and code sums [M][K/32]
    int *status;                 // device status word
    int test_skip_copy;          // failure-detection test only: CTA 0's warp 0 never requests its first
                                 // stage, so its bounded wait runs out (0 in every normal call)
    unsigned long long *phase;   // phase-timeline builds only (QMV_PHASE_STAMPS): [count, records...]
    unsigned int phase_seq;      //   this launch's sequence number
};

// Phase timeline: a build switch (QMV_PHASE_STAMPS), off by default, that
// adds no work to the product build.  Each CTA records global-timer stamps at
// entry, when griddepcontrol.wait returns (the previous grid has completed),
// when the activations are staged, and when its first and last warps finish.
constexpr int kPhaseWords = 7;   // seq << 32 | cta, t_entry, t_wait, t_staged, t_first_done, t_last_done, smid
constexpr int kPhaseCap = 1 << 18;

// Shared-memory bytes the kernel needs for a configuration.
__host__ __device__ inline size_t gemv_smem_bytes(int fmt, int M, int n_problems, int U, int warps, int S, int SP,
                                                   bool xq8 = false)
{
    const size_t unit_bytes = fmt == kQ4_0 ? 144 : (fmt == kQ2W ? 80 : 272);
    const size_t xbytes = static_cast<size_t>(n_problems) * M * U * (xq8 ? kXQ8UnitBytes : kXUnitBytes);
    const size_t ring = static_cast<size_t>(warps) * S * 32 * SP * unit_bytes;
    const size_t bars = static_cast<size_t>(warps) * S * 8;
    const size_t idx = (static_cast<size_t>(n_problems) * 4 + 15) / 16 * 16;   // expert indices (multi-expert call)
    return xbytes + ring + bars + idx;
}

// Permuted activation layout.  Within a block, the activation of element e
// (0..31) is stored at slot x_perm_slot(parity, e) (0..31), so that each
// 16-byte group of slots lines up with the half2 pairs one unpacked 32-bit word
// of codes produces.  Even blocks of a unit start 2 bytes into a 32-bit word,
// so their first word is re-formed with a PRMT as qs bytes (0, 1, 14, 15)
// [Q4_0], (0, 1, 30, 31) [Q8_0] or (0, 1, 6, 7) [2-bit, whose second word is
// then bytes (2..5)]; the other words are aligned.
template <int FMT>
__host__ __device__ __forceinline__ int x_perm_slot(int block_parity, int e)
{
    if (FMT == kQ4_0) {
        const int hi = e >= 16 ? 1 : 0;
        const int qi = e - 16 * hi;             // qs byte index 0..15
        int word, bp;
        if (block_parity) { word = qi >> 2; bp = qi & 3; }
        else if (qi < 2) { word = 0; bp = qi; }
        else if (qi >= 14) { word = 0; bp = qi - 12; }
        else { word = (qi + 2) >> 2; bp = (qi + 2) & 3; }
        // unpack_q4_word pairs: 0 = (lo b0, lo b2), 1 = (lo b1, lo b3),
        //                       2 = (hi b0, hi b2), 3 = (hi b1, hi b3)
        const int pair = (bp & 1) + 2 * hi;
        const int second = bp >> 1;
        return word * 8 + pair * 2 + second;
    } else if (FMT == kQ2W) {
        const int plane = e >> 3, qi = e & 7;     // code byte qi, bits 2*plane
        int word, bp;
        if (block_parity) { word = qi >> 2; bp = qi & 3; }
        else if (qi < 2 || qi >= 6) { word = 0; bp = qi < 2 ? qi : qi - 4; }
        else { word = 1; bp = qi - 2; }
        // unpack_q2_word pairs: 2p = (plane p of b0, of b2), 2p+1 = (of b1, of b3)
        const int pair = 2 * plane + (bp & 1);
        const int second = bp >> 1;
        return word * 16 + pair * 2 + second;
    } else {
        const int qi = e;
        int word, bp;
        if (block_parity) { word = qi >> 2; bp = qi & 3; }
        else if (qi < 2) { word = 0; bp = qi; }
        else if (qi >= 30) { word = 0; bp = qi - 28; }
        else { word = (qi + 2) >> 2; bp = (qi + 2) & 3; }
        // unpack_q8_word pairs: 0 = (b0, b2), 1 = (b1, b3)
        const int pair = bp & 1;
        const int second = bp >> 1;
        return word * 4 + pair * 2 + second;
    }
}

// ---- per-unit dot products ------------------------------------------------------

// acc += d * (a.lo + a.hi + b.lo + b.hi), with fp16 inputs, exact products and
// fp32 accumulation (mixed-precision fma.rn.f32.f16); d is the block's fp16
// scale in the low 16 bits of `dbits`.
__device__ __forceinline__ void acc_block(float &acc, uint32_t dbits, __half2 a, __half2 b)
{
    const uint32_t ua = *reinterpret_cast<uint32_t *>(&a);
    const uint32_t ub = *reinterpret_cast<uint32_t *>(&b);
    const unsigned short dh = static_cast<unsigned short>(dbits);
    asm("{\n\t.reg .b16 d, a0, a1, b0, b1;\n\t"
        "mov.b16 d, %1;\n\t"
        "mov.b32 {a0, a1}, %2;\n\t"
        "mov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, d, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, d, %0;\n\t"
        "fma.rn.f32.f16 %0, b0, d, %0;\n\t"
        "fma.rn.f32.f16 %0, b1, d, %0;\n\t}"
        : "+f"(acc)
        : "h"(dh), "r"(ua), "r"(ub));
}

// acc[m] += sum over the 8 blocks of one unit of d_b * (partial_b / prescale).
// wsrc: the unit's bytes in shared memory; xsrc: the unit's permuted
// activations for token 0; xstride: bytes between tokens.
template <int M>
__device__ __forceinline__ void dot_unit_q4_0(const uint8_t *wsrc, const uint8_t *xsrc, int xstride,
                                              float (&acc)[M])
{
    uint32_t w[36];
#pragma unroll
    for (int c = 0; c < 9; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(wsrc + 16 * c);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    float part[2][M];
#pragma unroll
    for (int m = 0; m < M; ++m) part[0][m] = part[1][m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int h = b >> 1;
        uint32_t q[4];
        uint32_t dsrc;
        if ((b & 1) == 0) {
            dsrc = w[9 * h] & 0xffffu;
            q[0] = __byte_perm(w[9 * h], w[9 * h + 4], 0x5432);
            q[1] = w[9 * h + 1];
            q[2] = w[9 * h + 2];
            q[3] = w[9 * h + 3];
        } else {
            dsrc = w[9 * h + 4] >> 16;
            q[0] = w[9 * h + 5];
            q[1] = w[9 * h + 6];
            q[2] = w[9 * h + 7];
            q[3] = w[9 * h + 8];
        }
        // Two independent half2 chains per token (words 0-1 and 2-3), joined
        // in fp32: shorter dependency chains, each half sums 8 products.
        __half2 ha[M], hb[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            ha[m] = __float2half2_rn(0.0f);
            hb[m] = __float2half2_rn(0.0f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 wv[4];
            unpack_q4_word(q[j], wv);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xsrc + m * xstride + b * 64 + j * 16);
                __half2 &h = (j < 2) ? ha[m] : hb[m];
                h = __hfma2(wv[0], as_h2(xv.x), h);
                h = __hfma2(wv[1], as_h2(xv.y), h);
                h = __hfma2(wv[2], as_h2(xv.z), h);
                h = __hfma2(wv[3], as_h2(xv.w), h);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc_block(part[b & 1][m], dsrc, ha[m], hb[m]);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] += part[0][m] + part[1][m];
}

template <int M>
__device__ __forceinline__ void dot_unit_q8_0(const uint8_t *wsrc, const uint8_t *xsrc, int xstride,
                                              float (&acc)[M])
{
    uint32_t w[68];
#pragma unroll
    for (int c = 0; c < 17; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(wsrc + 16 * c);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    float part[2][M];
#pragma unroll
    for (int m = 0; m < M; ++m) part[0][m] = part[1][m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int h = b >> 1;
        uint32_t q[8];
        uint32_t dsrc;
        if ((b & 1) == 0) {
            dsrc = w[17 * h] & 0xffffu;
            q[0] = __byte_perm(w[17 * h], w[17 * h + 8], 0x5432);
#pragma unroll
            for (int j = 1; j < 8; ++j) q[j] = w[17 * h + j];
        } else {
            dsrc = w[17 * h + 8] >> 16;
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = w[17 * h + 9 + j];
        }
        __half2 ha[M], hb[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            ha[m] = __float2half2_rn(0.0f);
            hb[m] = __float2half2_rn(0.0f);
        }
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            __half2 wa[2], wb[2];
            unpack_q8_word(q[j], wa);
            unpack_q8_word(q[j + 1], wb);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xsrc + m * xstride + b * 64 + j * 8);
                __half2 &h = (j < 4) ? ha[m] : hb[m];
                h = __hfma2(wa[0], as_h2(xv.x), h);
                h = __hfma2(wa[1], as_h2(xv.y), h);
                h = __hfma2(wb[0], as_h2(xv.z), h);
                h = __hfma2(wb[1], as_h2(xv.w), h);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc_block(part[b & 1][m], dsrc, ha[m], hb[m]);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] += part[0][m] + part[1][m];
}

// Plain 2-bit: a unit is 80 bytes = 20 words; blocks 2h, 2h+1 share words
// 5h..5h+4 as (d, c0, c1) (c2..c5) (c6, c7, d') (c'0..c'3) (c'4..c'7).
template <int M>
__device__ __forceinline__ void dot_unit_q2w(const uint8_t *wsrc, const uint8_t *xsrc, int xstride,
                                             float (&acc)[M])
{
    uint32_t w[20];
#pragma unroll
    for (int c = 0; c < 5; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(wsrc + 16 * c);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    float part[2][M];
#pragma unroll
    for (int m = 0; m < M; ++m) part[0][m] = part[1][m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int h = b >> 1;
        uint32_t q[2];
        uint32_t dsrc;
        if ((b & 1) == 0) {
            dsrc = w[5 * h] & 0xffffu;
            q[0] = __byte_perm(w[5 * h], w[5 * h + 2], 0x5432);   // code bytes 0, 1, 6, 7
            q[1] = w[5 * h + 1];                                  // code bytes 2..5
        } else {
            dsrc = w[5 * h + 2] >> 16;
            q[0] = w[5 * h + 3];
            q[1] = w[5 * h + 4];
        }
        // One half2 chain per word and token (8 products per half), joined in fp32.
        __half2 ha[M], hb[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            ha[m] = __float2half2_rn(0.0f);
            hb[m] = __float2half2_rn(0.0f);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            __half2 wv[8];
            unpack_q2_word(q[j], wv);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const uint8_t *xp = xsrc + m * xstride + b * 64 + j * 32;
                const uint4 x0 = *reinterpret_cast<const uint4 *>(xp);
                const uint4 x1 = *reinterpret_cast<const uint4 *>(xp + 16);
                __half2 &hh = (j == 0) ? ha[m] : hb[m];
                hh = __hfma2(wv[0], as_h2(x0.x), hh);
                hh = __hfma2(wv[1], as_h2(x0.y), hh);
                hh = __hfma2(wv[2], as_h2(x0.z), hh);
                hh = __hfma2(wv[3], as_h2(x0.w), hh);
                hh = __hfma2(wv[4], as_h2(x1.x), hh);
                hh = __hfma2(wv[5], as_h2(x1.y), hh);
                hh = __hfma2(wv[6], as_h2(x1.z), hh);
                hh = __hfma2(wv[7], as_h2(x1.w), hh);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc_block(part[b & 1][m], dsrc, ha[m], hb[m]);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] += part[0][m] + part[1][m];
}

// Q4_0 weights against Q8_1 activations: per block, integer dots of the codes
// (low nibbles against codes 0..15, high nibbles -- left in place, so 16 times
// their value -- against codes 16..31), minus 8 * sum(q), scaled by d_w * d_x.
template <int M>
__device__ __forceinline__ void dot_unit_q4_0_q81(const uint8_t *wsrc, const uint8_t *xsrc, int xstride,
                                                  float (&acc)[M])
{
    uint32_t w[36];
#pragma unroll
    for (int c = 0; c < 9; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(wsrc + 16 * c);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int h = b >> 1;
        uint32_t qw[4];
        uint32_t dsrc;
        if ((b & 1) == 0) {
            // qs starts 2 bytes into word 9h: realign to qs bytes 4k..4k+3
            dsrc = w[9 * h] & 0xffffu;
#pragma unroll
            for (int k = 0; k < 4; ++k) qw[k] = __byte_perm(w[9 * h + k], w[9 * h + k + 1], 0x5432);
        } else {
            dsrc = w[9 * h + 4] >> 16;
#pragma unroll
            for (int k = 0; k < 4; ++k) qw[k] = w[9 * h + 5 + k];
        }
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            lo[k] = qw[k] & 0x0F0F0F0Fu;
            hi[k] = qw[k] & 0xF0F0F0F0u;
        }
        const float dw = half_lo_to_float(dsrc);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint8_t *xp = xsrc + m * xstride;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(xp + b * 32);
            const uint4 x1 = *reinterpret_cast<const uint4 *>(xp + b * 32 + 16);
            const float2 meta = *reinterpret_cast<const float2 *>(xp + 256 + b * 8);   // (d_x, 8 * sum q)
            int sl = dp4a_us(lo[0], x0.x, 0);
            sl = dp4a_us(lo[1], x0.y, sl);
            sl = dp4a_us(lo[2], x0.z, sl);
            sl = dp4a_us(lo[3], x0.w, sl);
            int sh = dp4a_us(hi[0], x1.x, 0);
            sh = dp4a_us(hi[1], x1.y, sh);
            sh = dp4a_us(hi[2], x1.z, sh);
            sh = dp4a_us(hi[3], x1.w, sh);
            const int sumi = sl + (sh >> 4) - __float_as_int(meta.y);
            acc[m] = fmaf(static_cast<float>(sumi), dw * meta.x, acc[m]);
        }
    }
}

// Q8_0 against Q8_1 activations: both operands are signed bytes, so a block's
// dot is eight signed dp4a and its contribution d_w * d_x * sum(c_w * c_x); the
// codes carry no offset, so the activations' code sums are not needed.  An
// even block's codes start 2 bytes into a 4-byte word: each of its code words
// is re-formed from two adjacent words with one PRMT (the activations are
// staged in natural order).
template <int M>
__device__ __forceinline__ void dot_unit_q8_0_q81(const uint8_t *wsrc, const uint8_t *xsrc, int xstride,
                                                  float (&acc)[M])
{
    uint32_t w[68];
#pragma unroll
    for (int c = 0; c < 17; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(wsrc + 16 * c);
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int h = b >> 1;
        uint32_t qw[8];
        uint32_t dsrc;
        if ((b & 1) == 0) {
            dsrc = w[17 * h] & 0xffffu;
#pragma unroll
            for (int k = 0; k < 8; ++k) qw[k] = __byte_perm(w[17 * h + k], w[17 * h + k + 1], 0x5432);
        } else {
            dsrc = w[17 * h + 8] >> 16;
#pragma unroll
            for (int k = 0; k < 8; ++k) qw[k] = w[17 * h + 9 + k];
        }
        const float dw = half_lo_to_float(dsrc);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint8_t *xp = xsrc + m * xstride;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(xp + b * 32);
            const uint4 x1 = *reinterpret_cast<const uint4 *>(xp + b * 32 + 16);
            const float dx = *reinterpret_cast<const float *>(xp + 256 + b * 8);
            int s = __dp4a(static_cast<int>(qw[0]), static_cast<int>(x0.x), 0);
            s = __dp4a(static_cast<int>(qw[1]), static_cast<int>(x0.y), s);
            s = __dp4a(static_cast<int>(qw[2]), static_cast<int>(x0.z), s);
            s = __dp4a(static_cast<int>(qw[3]), static_cast<int>(x0.w), s);
            s = __dp4a(static_cast<int>(qw[4]), static_cast<int>(x1.x), s);
            s = __dp4a(static_cast<int>(qw[5]), static_cast<int>(x1.y), s);
            s = __dp4a(static_cast<int>(qw[6]), static_cast<int>(x1.z), s);
            s = __dp4a(static_cast<int>(qw[7]), static_cast<int>(x1.w), s);
            acc[m] = fmaf(static_cast<float>(s), dw * dx, acc[m]);
        }
    }
}

// ---- the streaming kernel ----------------------------------------------------------

// Warp-collective wait for phase `parity` of `bar`: one vote when the stage
// has landed (the common case), a bounded wait otherwise.
__device__ __forceinline__ bool stage_wait(uint64_t *bar, uint32_t parity, int *status)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return mbar_wait_warp(bar, parity, status);
}

// MOE = the one-launch multi-expert form: problem p is expert slot p with its
// own token, weights from expert_idx[p] of the pool.  Otherwise one problem
// of M tokens.  SWIGLU = the MLP's gate + up + SwiGLU in one pass: rows
// 2n / 2n+1 are row n of the gate / up table (the two tables handled as one
// stacked table -- volta-kernel-bakeoff, "A few tokens at once"), a CTA owns
// whole pairs, and y[m][n] = silu(g) * u is formed in the epilogue, so only
// the activated result reaches memory (SovereignKernel diary, phase 6).
// XF32 = the activations arrive as fp32 (p.xf) and are rounded to fp16 while
// they are staged, so the product that follows is the fp16 one (the bakeoff's
// fp32in kernels convert inside the kernel for the same reason: a separate
// conversion pass costs a launch -- volta-kernel-bakeoff, "Results (one token,
// microseconds, lower is better)").
// XQ8 = the activations are quantised to Q8_1 while they are staged (or copied
// in, already quantised) and the block products are integer dots (plain Q4_0
// and Q8_0 calls only).
template <int FMT, int M, int MAXT, bool MOE, bool SWIGLU = false, bool XF32 = false, bool XQ8 = false>
__global__ void __launch_bounds__(MAXT, 1) qmv_stream_kernel(const GemvParams p)
{
    using T = FmtTraits<FMT>;
    static_assert(!XQ8 || ((FMT == kQ4_0 || FMT == kQ8_0) && !MOE && !SWIGLU && !XF32),
                  "Q8_1 activations: plain Q4_0 and Q8_0 calls only");
    constexpr int XUB = XQ8 ? kXQ8UnitBytes : kXUnitBytes;   // activation bytes per unit and token
    constexpr float kPre = XQ8 ? 1.0f : T::kPrescale;           // the integer dot carries no pre-scale
    extern __shared__ __align__(128) uint8_t smem[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int U = p.U, G = p.G, SP = p.SP, S = p.S;
#ifdef QMV_PHASE_STAMPS
    __shared__ unsigned long long ph_t[4];   // entry, wait, staged, first warp done
    __shared__ unsigned long long ph_last;
    if (threadIdx.x == 0) {
        ph_t[0] = global_timer_ns();
        ph_t[3] = ~0ull;
        ph_last = 0;
    }
#endif
    const int RG = 32 / G;
    // Row indices fit in 32 bits (checked on the host).
    const uint32_t N = static_cast<uint32_t>(p.N);

    // Shared-memory carve-up: activations, then per-warp rings, then barriers.
    const size_t xbytes = static_cast<size_t>(p.max_local_problems) * M * U * XUB;
    const int slot_bytes = 32 * SP * T::kUnitBytes;
    uint8_t *xs = smem;
    uint8_t *ring = smem + xbytes + static_cast<size_t>(warp) * S * slot_bytes;
    uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + xbytes + static_cast<size_t>(warps) * S * slot_bytes);
    uint64_t *bars = bars_all + warp * S;
    int32_t *sidx = reinterpret_cast<int32_t *>(bars_all + warps * S);   // this CTA's expert indices

    // This CTA's contiguous range of (problem, row) pairs.
    const uint32_t R = static_cast<uint32_t>(p.rows_total);
    // (SwiGLU: whole gate/up pairs, so row0 is even and nrows even.)
    const uint32_t row0 = SWIGLU ? 2u * static_cast<uint32_t>((static_cast<uint64_t>(R / 2) * blockIdx.x) / gridDim.x)
                                 : static_cast<uint32_t>((static_cast<uint64_t>(R) * blockIdx.x) / gridDim.x);
    const uint32_t row1 = SWIGLU ? 2u * static_cast<uint32_t>((static_cast<uint64_t>(R / 2) * (blockIdx.x + 1)) / gridDim.x)
                                 : static_cast<uint32_t>((static_cast<uint64_t>(R) * (blockIdx.x + 1)) / gridDim.x);
    const int nrows = static_cast<int>(row1 - row0);
    // Problems (expert slots) this CTA touches; always 0..0 for the plain GEMV.
    const int prob_lo = (MOE && nrows > 0) ? static_cast<int>(row0 / N) : 0;
    const int prob_hi = MOE ? (nrows > 0 ? static_cast<int>((row1 - 1) / N) : -1) : 0;
    const int ngroups = (nrows + RG - 1) / RG;
    const int my_groups = (ngroups > warp) ? (ngroups - warp + warps - 1) / warps : 0;
    const int units_per_stage = SP * G;
    const int T_stages = (U + units_per_stage - 1) / units_per_stage;
    const int total = my_groups * T_stages;
    const uint32_t lane_chunk_bytes = static_cast<uint32_t>(units_per_stage) * T::kUnitBytes;
    const uint8_t *cta_rows = p.W + static_cast<int64_t>(row0) * p.row_bytes;   // plain GEMV only

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    __syncwarp();

    // ---- copy issue: stages are requested strictly in order ----------------------
    int issued = 0;          // stages requested
    int is_slot = 0;         // slot of the next stage to request
    int is_t = 0;            // its stage index within the row group
    int is_g = warp;         // its row group (CTA-local)
    const uint8_t *is_row = nullptr;   // multi-expert call: row of lane r < RG in the current group (null: none)
    const uint64_t l2_policy = l2_evict_first_policy();   // weights stream through L2 once

    // One elected lane requests the row chunks of a stage in a loop (except in
    // the multi-expert call): a copy whose operands differ per lane is issued
    // one lane at a time anyway, at several times the cost (on the GB300, 32
    // per-lane 256-byte copies took ~1760 cycles to issue, the same 32 from one
    // lane ~420).
    auto issue_next = [&]() {
        const int u0 = is_t * units_per_stage;
        const int u1 = min(U, u0 + units_per_stage);
        const uint32_t bytes = static_cast<uint32_t>(u1 - u0) * T::kUnitBytes;
        const size_t off = static_cast<size_t>(u0) * T::kUnitBytes;
        const int lr0 = is_g * RG;
        const int nr = min(RG, nrows - lr0);   // rows of the group (at least one while stages remain)
        // (test only) the first stage of CTA 0's warp 0 is expected but never
        // requested: nothing is in flight into that slot when its wait gives up
        const bool skip = p.test_skip_copy && blockIdx.x == 0 && warp == 0 && issued == 0;
        if constexpr (MOE) {
            // Per-lane copies here (lane r requests group row r): each row's
            // expert id comes from shared memory, and rows whose id is out of
            // range request nothing (their dot products read zeros).  Measured
            // ahead of an elected lane's loop for the multi-expert call.
            if (is_t == 0) {
                is_row = nullptr;
                if (lane < nr) {
                    const uint32_t row = row0 + static_cast<uint32_t>(lr0 + lane);
                    const uint32_t prob = row / N;
                    const uint32_t n = row - prob * N;
                    const int64_t e = sidx[prob - prob_lo];
                    if (e >= 0 && e < p.n_experts) is_row = p.W + (e * p.N + n) * p.row_bytes;
                }
            }
            const uint32_t my_bytes = is_row ? bytes : 0u;
            const uint32_t total_bytes = __reduce_add_sync(0xffffffffu, my_bytes);
            if (lane == 0) mbar_arrive_expect_tx(&bars[is_slot], total_bytes);
            __syncwarp();
            if (my_bytes && !skip)
                bulk_g2s_hint(ring + static_cast<size_t>(is_slot) * slot_bytes + lane * lane_chunk_bytes, is_row + off,
                              my_bytes, &bars[is_slot], l2_policy);
        } else if (elect_one()) {
            uint8_t *dst = ring + static_cast<size_t>(is_slot) * slot_bytes;
            mbar_arrive_expect_tx(&bars[is_slot], static_cast<uint32_t>(nr) * bytes);
            if (!skip)
                for (int i = 0; i < nr; ++i) {
                    const uint8_t *src;
                    if (SWIGLU) {
                        const uint32_t row = row0 + static_cast<uint32_t>(lr0 + i);
                        src = ((row & 1u) ? p.W2 : p.W) + static_cast<int64_t>(row >> 1) * p.row_bytes;
                    } else {
                        src = cta_rows + static_cast<int64_t>(lr0 + i) * p.row_bytes;
                    }
                    bulk_g2s_hint(dst + i * lane_chunk_bytes, src + off, bytes, &bars[is_slot], l2_policy);
                }
        }
        __syncwarp();
        ++issued;
        if (++is_slot == S) is_slot = 0;
        if (++is_t == T_stages) {
            is_t = 0;
            is_g += warps;
        }
    };

    // Request the first stage before waiting for the previous kernel (W is
    // never written by it).  The expert indices may be, so the multi-expert
    // call waits first.  The remaining prefetch is requested after this
    // thread's activation loads: the activations are on the critical path and
    // must not queue behind megabytes of weight traffic.
    // The multi-expert call requests its first p.early stages as soon as it
    // has the indices, ahead of its activation loads (it has no weights in
    // flight before then).
    const int prefetch = total < S ? total : S;
    const int early_n = prefetch < p.early ? prefetch : p.early;
    int early = MOE ? 0 : early_n;
    for (int i = 0; i < early; ++i) issue_next();

    pdl_wait_prior_grid();
#ifdef QMV_PHASE_STAMPS
    if (threadIdx.x == 0) ph_t[1] = global_timer_ns();
#endif

    if (MOE) {
        // The CTA's expert indices, once, before any copy needs them.
        for (int i = threadIdx.x; i <= prob_hi - prob_lo; i += blockDim.x) sidx[i] = p.expert_idx[prob_lo + i];
        __syncthreads();
        for (int i = 0; i < early_n; ++i) issue_next();
        early = early_n;
    }

    // Stage the activations: permuted pair order, 528-byte padded units.  Each
    // thread builds whole 16-byte chunks of the permuted layout from four
    // 4-byte loads (pairs of consecutive activations) and four PRMTs.  The
    // (token, chunk) items of all the CTA's tokens are dealt out together, up
    // to kStageItems per thread per round with all their loads in flight, so
    // long rows and several tokens cost few L2 round trips.
    if (XQ8 && p.xq) {
        // Activations already in Q8_1: copy the codes (16 per load) and the
        // blocks' (scale, 8 * code sum) into the staged layout.
        const int chunks = static_cast<int>(p.K / 16);
        for (int it = threadIdx.x; it < M * chunks; it += blockDim.x) {
            const int tok = it / chunks, c = it - tok * chunks;
            const int blk = c >> 1;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.xq + static_cast<int64_t>(tok) * p.K) + c);
            *reinterpret_cast<uint4 *>(xs + static_cast<size_t>(tok) * U * XUB + (blk >> 3) * XUB + (blk & 7) * 32 +
                                       (c & 1) * 16) = v;
        }
        const int nb = static_cast<int>(p.K / 32);
        for (int it = threadIdx.x; it < M * nb; it += blockDim.x) {
            const int tok = it / nb, blk = it - tok * nb;
            const int64_t j = static_cast<int64_t>(tok) * nb + blk;
            const float dxq = __half2float(__ushort_as_half(__ldg(p.xq_d + j)));
            int sum8 = 0;   // Q8_0 codes carry no offset: the code sums are not read
            if constexpr (FMT == kQ4_0) sum8 = 8 * __ldg(p.xq_s + j);
            *reinterpret_cast<float2 *>(xs + static_cast<size_t>(tok) * U * XUB + (blk >> 3) * XUB + 256 +
                                        (blk & 7) * 8) = make_float2(dxq, __int_as_float(sum8));
        }
        for (int i = early; i < prefetch; ++i) issue_next();
    } else if constexpr (XQ8) {
        // Q8_1: each item is a 16-byte chunk of 8 activations, read with one
        // load; the four chunks of a 32-block sit in four adjacent lanes of one
        // round (chunks per token and the round are multiples of 4), which
        // share the block's max and code sum with shuffles.
        constexpr int kQItems = (M == 1) ? 2 : 4;
        const int ntok = M;
        const int chunks = static_cast<int>(p.K / 8);
        const int items = ntok * chunks;
        const int round = kQItems * blockDim.x;
        const int dq = round / chunks, dr = round - dq * chunks;
        int tk[kQItems], ck[kQItems];
#pragma unroll
        for (int b = 0; b < kQItems; ++b) {
            const int it = b * blockDim.x + threadIdx.x;
            tk[b] = it / chunks;
            ck[b] = it - tk[b] * chunks;
        }
        bool first = true;
        for (int it0 = 0; it0 < items || first; it0 += round) {
            uint4 xv[kQItems];
            bool ok[kQItems];
            int cidx[kQItems], tidx[kQItems];
#pragma unroll
            for (int b = 0; b < kQItems; ++b) {
                ok[b] = it0 + b * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x) < items;
                cidx[b] = ck[b];
                tidx[b] = tk[b];
                xv[b] = make_uint4(0u, 0u, 0u, 0u);
                if (ok[b])
                    xv[b] = __ldg(reinterpret_cast<const uint4 *>(p.x + static_cast<int64_t>(tk[b]) * p.K) + ck[b]);
            }
#pragma unroll
            for (int b = 0; b < kQItems; ++b) {
                ck[b] += dr;
                tk[b] += dq;
                if (ck[b] >= chunks) {
                    ck[b] -= chunks;
                    ++tk[b];
                }
            }
            if (first) {
                first = false;
                for (int i = early; i < prefetch; ++i) issue_next();
            }
#pragma unroll
            for (int b = 0; b < kQItems; ++b) {
                float dxq;
                int sq;
                const uint2 codes = q8_1_chunk(xv[b], dxq, sq);    // all lanes: it shuffles
                if (ok[b]) {
                    const int c = cidx[b];
                    const int blk = c >> 2, sub = c & 3;
                    uint8_t *xu = xs + static_cast<size_t>(tidx[b]) * U * XUB + (blk >> 3) * XUB;
                    *reinterpret_cast<uint2 *>(xu + (blk & 7) * 32 + sub * 8) = codes;
                    if (sub == 0)
                        *reinterpret_cast<float2 *>(xu + 256 + (blk & 7) * 8) = make_float2(dxq, __int_as_float(8 * sq));
                }
            }
        }
    } else {
        constexpr bool kOneToken = (M == 1 && !MOE);
        constexpr int kStageItems = 4;
        const int ntok = (prob_hi - prob_lo + 1) * M;
        const int chunks = static_cast<int>(p.K / 8);          // 16-byte chunks per token (4 per block)
        const int items = ntok * chunks;
        // Item slot b of this thread is item it0 + b * blockDim + threadIdx
        // = (token tk[b], chunk ck[b]); both advance by a fixed step per round.
        const int round = kStageItems * blockDim.x;
        const int dq = kOneToken ? 0 : round / chunks, dr = kOneToken ? round : round - dq * chunks;
        int tk[kStageItems], ck[kStageItems];
#pragma unroll
        for (int b = 0; b < kStageItems; ++b) {
            const int it = b * blockDim.x + threadIdx.x;
            tk[b] = kOneToken ? 0 : it / chunks;
            ck[b] = it - tk[b] * chunks;
        }
        bool first = true;
        for (int it0 = 0; it0 < items || first; it0 += round) {
            uint32_t a[kStageItems][4];
            float2 af[XF32 ? kStageItems : 1][4];    // fp32 pairs, rounded when stored
            int cidx[kStageItems], tidx[kStageItems];
#pragma unroll
            for (int b = 0; b < kStageItems; ++b) {
                const int it = it0 + b * blockDim.x + threadIdx.x;
                cidx[b] = -1;
                tidx[b] = 0;
                if (it < items) {
                    const int tok = tk[b];
                    const int c = ck[b];
                    cidx[b] = c;
                    tidx[b] = tok;
                    const int blk = c >> 2, sub = c & 3;
                    int i0, i2, i4, i6;    // first element of each loaded pair (in half units)
                    if (FMT == kQ4_0) {
                        // word `sub` of the block: bytes b0,b1 from (i0, i0+1), b2,b3 from (i2, i2+1);
                        // low nibbles are elements i, high nibbles i + 16.
                        if (blk & 1) { i0 = 4 * sub; i2 = 4 * sub + 2; }
                        else if (sub == 0) { i0 = 0; i2 = 14; }
                        else { i0 = 4 * sub - 2; i2 = 4 * sub; }
                        i4 = i0 + 16;
                        i6 = i2 + 16;
                    } else if (FMT == kQ2W) {
                        // planes 2*(sub & 1) and 2*(sub & 1) + 1 of word sub >> 1: bytes
                        // b0,b1 from (i0, i0+1), b2,b3 from (i2, i2+1); byte i holds
                        // elements i + 8 * plane.  Even blocks: words (0,1,6,7), (2..5).
                        const int wd = sub >> 1, p0 = 2 * (sub & 1);
                        int b0, b2;
                        if (blk & 1) { b0 = 4 * wd; b2 = 4 * wd + 2; }
                        else if (wd == 0) { b0 = 0; b2 = 6; }
                        else { b0 = 2; b2 = 4; }
                        i0 = b0 + 8 * p0;
                        i2 = b2 + 8 * p0;
                        i4 = i0 + 8;
                        i6 = i2 + 8;
                    } else {
                        // words 2*sub and 2*sub+1 of the block (Q8_0: four codes per word)
                        const int w0 = 2 * sub, w1 = 2 * sub + 1;
                        if (blk & 1) { i0 = 4 * w0; i2 = 4 * w0 + 2; }
                        else if (w0 == 0) { i0 = 0; i2 = 30; }
                        else { i0 = 4 * w0 - 2; i2 = 4 * w0; }
                        if (blk & 1) { i4 = 4 * w1; i6 = 4 * w1 + 2; }
                        else { i4 = 4 * w1 - 2; i6 = 4 * w1; }
                    }
                    const int64_t xoff = (static_cast<int64_t>(prob_lo) * M + tok) * p.K;
                    if constexpr (XF32) {
                        // one 8-byte load per pair; all loads of the round are
                        // issued before any of them is rounded to a half2 word
                        const float2 *xb = reinterpret_cast<const float2 *>(p.xf + xoff) + blk * 16;
                        af[b][0] = __ldg(xb + (i0 >> 1));
                        af[b][1] = __ldg(xb + (i2 >> 1));
                        af[b][2] = __ldg(xb + (i4 >> 1));
                        af[b][3] = __ldg(xb + (i6 >> 1));
                    } else {
                        const uint32_t *xb = reinterpret_cast<const uint32_t *>(p.x + xoff) +
                                             blk * 16;     // 32 halves = 16 words per block
                        a[b][0] = __ldg(xb + (i0 >> 1));
                        a[b][1] = __ldg(xb + (i2 >> 1));
                        a[b][2] = __ldg(xb + (i4 >> 1));
                        a[b][3] = __ldg(xb + (i6 >> 1));
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < kStageItems; ++b) {
                ck[b] += dr;
                tk[b] += dq;
                if (!kOneToken && ck[b] >= chunks) {
                    ck[b] -= chunks;
                    ++tk[b];
                }
            }
            if (first) {
                first = false;
                for (int i = early; i < prefetch; ++i) issue_next();
            }
#pragma unroll
            for (int b = 0; b < kStageItems; ++b) {
                if (cidx[b] >= 0) {
                    const int c = cidx[b];
                    const int blk = c >> 2, sub = c & 3;
                    uint8_t *xd = xs + static_cast<size_t>(tidx[b]) * U * kXUnitBytes;
                    if constexpr (XF32) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) a[b][k] = float2_to_half2_bits(af[b][k]);
                    }
                    // pairs (first of each, first of each) and (second, second)
                    const uint4 v = make_uint4(__byte_perm(a[b][0], a[b][1], 0x5410), __byte_perm(a[b][0], a[b][1], 0x7632),
                                               __byte_perm(a[b][2], a[b][3], 0x5410), __byte_perm(a[b][2], a[b][3], 0x7632));
                    *reinterpret_cast<uint4 *>(xd + (blk >> 3) * kXUnitBytes + (blk & 7) * 64 + sub * 16) = v;
                }
            }
        }
    }
    __syncthreads();
    pdl_allow_next_grid();
#ifdef QMV_PHASE_STAMPS
    if (threadIdx.x == 0) ph_t[2] = global_timer_ns();
#endif

    const int r = lane / G;
    const int q = lane - r * G;
    const bool lane_on = r < RG;             // G that does not divide 32 leaves lanes RG*G.. idle
    const bool g_pow2 = (G & (G - 1)) == 0;
    const int xstride = U * XUB;             // bytes between tokens of a problem
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;

    bool alive = true;
    int consumed = 0;
    int slot = 0;
    uint32_t phase = 0;
    int t = 0;
    int g = warp;
    int lr = 0;
    uint32_t prob = 0;
    bool row_ok = false;
    const uint8_t *xrow = xs;
    const uint8_t *lane_stage = ring + r * lane_chunk_bytes;

    for (int i = 0; i < total; ++i) {
        if (t == 0) {
            lr = g * RG + r;
            row_ok = lane_on && lr < nrows;
            if (MOE) {
                prob = row_ok ? (row0 + lr) / N : static_cast<uint32_t>(prob_lo);
                if (row_ok) {
                    const int64_t e = sidx[prob - prob_lo];
                    row_ok = (e >= 0 && e < p.n_experts);
                }
                xrow = xs + static_cast<size_t>(prob - prob_lo) * M * xstride;
            }
        }
        if (!stage_wait(&bars[slot], phase, p.status)) {
            alive = false;
            break;
        }
        consumed = i + 1;
        const uint8_t *stage = lane_stage + static_cast<size_t>(slot) * slot_bytes;
        if (row_ok) {
            const int u0 = t * units_per_stage + q;
            for (int pass = 0; pass < SP; ++pass) {
                const int u = u0 + pass * G;
                if (u < U) {
                    if constexpr (XQ8 && FMT == kQ8_0)
                        dot_unit_q8_0_q81<M>(stage + (pass * G + q) * T::kUnitBytes, xrow + u * XUB, xstride, acc);
                    else if constexpr (XQ8)
                        dot_unit_q4_0_q81<M>(stage + (pass * G + q) * T::kUnitBytes, xrow + u * XUB, xstride, acc);
                    else if (FMT == kQ4_0)
                        dot_unit_q4_0<M>(stage + (pass * G + q) * T::kUnitBytes, xrow + u * kXUnitBytes, xstride, acc);
                    else if (FMT == kQ2W)
                        dot_unit_q2w<M>(stage + (pass * G + q) * T::kUnitBytes, xrow + u * kXUnitBytes, xstride, acc);
                    else
                        dot_unit_q8_0<M>(stage + (pass * G + q) * T::kUnitBytes, xrow + u * kXUnitBytes, xstride, acc);
                }
            }
        }
        // This lane's reads of the stage (generic proxy) are ordered before
        // the bulk copy that refills the slot (async proxy).
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (issued < total) issue_next();

        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
        if (++t == T_stages) {
            t = 0;
            g += warps;
            // Combine the G partial sums of each row.
            if (g_pow2) {
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    for (int off = G >> 1; off > 0; off >>= 1)
                        acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
                }
            } else {
                // G lanes per row, G not a power of two: the row's first lane
                // adds the G partial sums in lane order.
                const int src0 = (lane_on ? r : 0) * G;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float sum = 0.0f;
                    for (int j = 0; j < G; ++j) sum += __shfl_sync(0xffffffffu, acc[m], src0 + j);
                    acc[m] = sum;
                }
            }
            if (SWIGLU) {
                // The up row (lr + 1) sits G lanes further on in the same group.
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const float up = __shfl_down_sync(0xffffffffu, acc[m], G);
                    if (q == 0 && lane_on && lr < nrows && (lr & 1) == 0) {
                        const float gate = acc[m] * kPre;
                        p.y[static_cast<int64_t>(m) * p.N + ((row0 + lr) >> 1)] =
                            gate / (1.0f + __expf(-gate)) * (up * kPre);
                    }
                }
            } else if (q == 0 && lane_on && lr < nrows) {
                const uint32_t row = row0 + lr;
                if (MOE) {
                    const uint32_t n = row - prob * N;
                    if (!row_ok) atomicOr(p.status, kDevBadExpert);
                    p.y[static_cast<int64_t>(prob) * p.N + n] =
                        row_ok ? acc[0] * kPre : __int_as_float(0x7fc00000);
                } else {
#pragma unroll
                    for (int m = 0; m < M; ++m) p.y[static_cast<int64_t>(m) * p.N + row] = acc[m] * kPre;
                }
            }
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m] = 0.0f;
        }
    }

    if (!alive) {
        // A wait gave up: let every copy this warp requested land before the
        // CTA (and its shared memory) goes away; each wait is bounded again.
        // Each slot holds at most one outstanding stage.
        if (lane == 0) {
            for (int j = consumed; j < issued; ++j)
                mbar_wait_bounded(&bars[j % S], static_cast<uint32_t>((j / S) & 1), nullptr);
        }
        __syncwarp();
    }
#ifdef QMV_PHASE_STAMPS
    if (lane == 0) {
        const unsigned long long t = global_timer_ns();
        atomicMin(&ph_t[3], t);
        atomicMax(&ph_last, t);
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.phase) {
        const unsigned long long i = atomicAdd(p.phase, 1ull);
        if (i < kPhaseCap) {
            unsigned smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            unsigned long long *rec = p.phase + 1 + i * kPhaseWords;
            rec[0] = (static_cast<unsigned long long>(p.phase_seq) << 32) | blockIdx.x;
            rec[1] = ph_t[0];
            rec[2] = ph_t[1];
            rec[3] = ph_t[2];
            rec[4] = ph_t[3];
            rec[5] = ph_last;
            rec[6] = smid;
        }
    }
#endif
}

// ---- the generic kernel (any K % 32 == 0, any M, activations from global) ----------

// Activation i as the product sees it: fp16, or fp32 rounded to fp16 (nearest
// even) exactly as the streaming kernel stages it.
__device__ __forceinline__ float load_x(const GemvParams &p, int64_t i)
{
    return p.xf ? __half2float(__float2half_rn(p.xf[i])) : __half2float(p.x[i]);
}

// Signed code of weight j of a block (before its scale), for the generic kernel.
template <int FMT>
__device__ __forceinline__ int weight_code(const uint8_t *blk, int j)
{
    if (FMT == kQ4_0) return (j < 16 ? (blk[2 + j] & 0xF) : (blk[2 + j - 16] >> 4)) - 8;
    if (FMT == kQ2W) return ((blk[2 + (j & 7)] >> (2 * (j >> 3))) & 3) - 2;
    return static_cast<int8_t>(blk[2 + j]);
}

template <int FMT>
__global__ void __launch_bounds__(256) qmv_generic_kernel(const GemvParams p, int M)
{
    const int lane = threadIdx.x & 31;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int bb = FmtTraits<FMT>::kBlockBytes;
    const int64_t nblk = p.K / 32;
    pdl_wait_prior_grid();
    // Fused SwiGLU (W2 set): one warp per output row n, both products.
    const bool swiglu = p.W2 != nullptr;
    const int64_t nout = swiglu ? p.N : p.rows_total;
    for (int64_t row = gw; row < nout; row += nw) {
        const int64_t prob = row / p.N;
        const int64_t n = row - prob * p.N;
        int64_t e = 0;
        bool ok = true;
        if (p.expert_idx) {
            e = p.expert_idx[prob];
            ok = (e >= 0 && e < p.n_experts);
        }
        for (int m0 = 0; m0 < M; m0 += 8) {
            float acc[8], gacc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = gacc[j] = 0.0f;
            for (int t = 0; t < (swiglu ? 2 : 1); ++t) {
                if (t == 1) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        gacc[j] = acc[j];
                        acc[j] = 0.0f;
                    }
                }
                if (ok && p.xq8) {
                    // Q8_1 activations: each block's codes decided as the streaming
                    // kernel decides them, then an integer dot per block.
                    const uint8_t *wr = p.W + (e * p.N + n) * p.row_bytes;
                    for (int64_t b = lane; b < nblk; b += 32) {
                        const uint8_t *blk = wr + b * bb;
                        const float dw = __half2float(__ushort_as_half(
                            static_cast<unsigned short>(blk[0] | (blk[1] << 8))));
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) {
                            if (m0 + mm >= M) continue;
                            const int64_t tok = prob * M + m0 + mm;
                            int s = 0;
                            float dxq;
                            if (p.xq) {   // activations already in Q8_1
                                const int8_t *qb = p.xq + tok * p.K + b * 32;
                                for (int j = 0; j < 32; ++j) s += weight_code<FMT>(blk, j) * qb[j];
                                dxq = __half2float(__ushort_as_half(p.xq_d[tok * (p.K / 32) + b]));
                            } else {
                                const __half *xb = p.x + tok * p.K + b * 32;
                                float amax = 0.0f;
                                for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(__half2float(xb[j])));
                                const float d = __fdiv_rn(amax, 127.0f);
                                const float id = d != 0.0f ? __frcp_rn(d) : 0.0f;
                                for (int j = 0; j < 32; ++j) {
                                    const int code = static_cast<int>(roundf(__fmul_rn(__half2float(xb[j]), id)));
                                    s += weight_code<FMT>(blk, j) * code;
                                }
                                dxq = __half2float(__float2half_rn(d));
                            }
                            acc[mm] = fmaf(static_cast<float>(s), dw * dxq, acc[mm]);
                        }
                    }
                } else if (ok) {
                    const uint8_t *wr = (t == 1 ? p.W2 : p.W) + (e * p.N + n) * p.row_bytes;
                    for (int64_t b = lane; b < nblk; b += 32) {
                        const uint8_t *blk = wr + b * bb;
                        const float d = __half2float(__ushort_as_half(
                            static_cast<unsigned short>(blk[0] | (blk[1] << 8))));
                        for (int j = 0; j < 32; ++j) {
                            const float wv = static_cast<float>(weight_code<FMT>(blk, j)) * d;
#pragma unroll
                            for (int mm = 0; mm < 8; ++mm) {
                                if (m0 + mm < M)
                                    acc[mm] = fmaf(wv, load_x(p, (prob * M + m0 + mm) * p.K + b * 32 + j), acc[mm]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int mm = 0; mm < 8; ++mm)
                    for (int off = 16; off > 0; off >>= 1) acc[mm] += __shfl_xor_sync(0xffffffffu, acc[mm], off);
            }
            if (lane == 0) {
                if (!ok) atomicOr(p.status, kDevBadExpert);
                for (int mm = 0; mm < 8 && m0 + mm < M; ++mm) {
                    float v = acc[mm];
                    if (swiglu) v = gacc[mm] / (1.0f + __expf(-gacc[mm])) * acc[mm];
                    p.y[(prob * M + m0 + mm) * p.N + n] = ok ? v : __int_as_float(0x7fc00000);
                }
            }
        }
    }
}

}  // namespace qmv
