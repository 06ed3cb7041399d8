// qmv_common.cuh -- device-side building blocks shared by the decode and
// prefill kernels: inline-PTX wrappers for mbarriers, bulk (TMA) copies,
// programmatic dependent launch, and the fp16 magic-number unpack of GGUF
// Q4_0 / Q8_0 codes.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qmv {

// Device status bits (mirrors QMV_DEV_* in include/qmv.h).
constexpr int kDevBadExpert = 0x1;
constexpr int kDevTimeout = 0x2;

// A bounded wait gives up after this many nanoseconds of global time.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread (up to `hint_ns`) until
// the phase completes, instead of returning at once: a waiting thread then
// takes no issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kSuspendHintNs = 20000;

// Wait for phase `parity` of `bar`, giving up after kWaitLimitNs.  Called by a
// single thread.  Returns false (and records kDevTimeout) on give-up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            if (status) atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Warp-collective bounded wait: every lane of the warp calls it; the result is
// warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, int *status)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
        // The phase has completed; every lane observes it before touching data.
        while (!mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) {
        }
    }
    return ok;
}

// One lane of a converged warp (the same lane on every call with all lanes
// active).  The tensor-core and tensor-copy issue paths run inside such a
// block of a warp that executes the loop as a whole: measured on the GB300,
// a loop run by a lone lane issued 64-column MMAs at ~105 cycles each, the
// same loop run by the converged warp with an elected issuer at ~50.
__device__ __forceinline__ bool elect_one()
{
    uint32_t e;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(e));
    return e != 0;
}

// ---- bulk copies (TMA, non-tensor) --------------------------------------------

// Global -> shared bulk copy that signals `bar` with complete_tx.  dst, src and
// bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// An L2 policy that evicts the streamed lines first: weights are read once per
// call and should not push the (small, reused) activations out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache-eviction hint.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---- programmatic dependent launch ---------------------------------------------

__device__ __forceinline__ void pdl_wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_allow_next_grid()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- integer helpers ------------------------------------------------------------

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ __half2 as_h2(uint32_t u)
{
    return *reinterpret_cast<__half2 *>(&u);
}

// Two fp32 values rounded to fp16 (nearest even) as one half2 word: .x in
// the low half, as two consecutive fp16 activations sit in memory.
__device__ __forceinline__ uint32_t float2_to_half2_bits(float2 v)
{
    const __half2 h = __float22half2_rn(v);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float half_lo_to_float(uint32_t u)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu)));
}

__device__ __forceinline__ float half_hi_to_float(uint32_t u)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16)));
}

// ---- fp16 magic-number unpack -----------------------------------------------------
//
// The half with bit pattern 0x6400 | n is exactly 1024 + n for 0 <= n < 1024
// (the unpack of the bakeoff's v2 kernel -- volta-kernel-bakeoff, "What's in
// the race").  One LOP3 places two nibbles (or, after a
// PRMT, two bytes) into the mantissas of a half2; one HFMA2 then removes the
// 1024 offset and the code bias and applies a power-of-two pre-scale, exactly.
//
// The weights come out pre-scaled so that no fp16 partial sum can overflow,
// whatever the (finite) fp16 activations: a lane sums two code words, i.e.
// eight products, in each half of a half2 chain before the chain goes to fp32,
// and the page's rule for that case is to divide the centred code by 64
// instead of 32 (volta-kernel-bakeoff, "A few tokens at once").  Q4_0 weights
// enter as (c - 8) / 64 and Q8_0 weights as q / 1024, so |w'| <= 1/8 and one
// product is at most 65504 / 8 = 8188 in magnitude.  Round-to-nearest is
// monotone, so after i products a partial sum is at most B_i with B_1 = 8188
// and B_i = fp16(B_{i-1} + 8188): 8188, 16376, 24560, 32752, 40928, 49120,
// 57312, 65504 -- finite after all eight (a CPU test replays this sequence
// against the constants below).  The plain 2-bit weights enter as (c - 2) / 32
// (|w'| <= 1/16: at most 32752 after eight products).  The fp32 block sums are
// multiplied back by the pre-scale at the end (exact: a power of two).
constexpr float kQ4Prescale = 64.0f;
constexpr float kQ8Prescale = 1024.0f;
constexpr float kQ2Prescale = 32.0f;

// Q4_0: one 32-bit word of qs holding bytes (b0, b1, b2, b3) -> four half2
// weights (c - 8) / 64:  w[0] = (lo b0, lo b2)   w[1] = (lo b1, lo b3)
//           w[2] = (hi b0, hi b2)   w[3] = (hi b1, hi b3)
// Low nibbles of qs[i] are element i of the block, high nibbles element i+16.
__device__ __forceinline__ void unpack_q4_word(uint32_t v, __half2 (&w)[4])
{
    const uint32_t magic = 0x64006400u;
    const uint32_t v8 = v >> 8;
    const uint32_t l02 = and_or(v, 0x000F000Fu, magic);   // 1024 + n
    const uint32_t l13 = and_or(v8, 0x000F000Fu, magic);
    const uint32_t h02 = and_or(v, 0x00F000F0u, magic);   // 1024 + 16 n
    const uint32_t h13 = and_or(v8, 0x00F000F0u, magic);
    // (1024 + n) / 64 - 1032 / 64 = (n - 8) / 64
    const __half2 s_lo = __halves2half2(__ushort_as_half(0x2400), __ushort_as_half(0x2400));  // 2^-6
    const __half2 b_lo = __halves2half2(__ushort_as_half(0xCC08), __ushort_as_half(0xCC08));  // -16.125
    // (1024 + 16 n) / 1024 - 1.125 = (n - 8) / 64
    const __half2 s_hi = __halves2half2(__ushort_as_half(0x1400), __ushort_as_half(0x1400));  // 2^-10
    const __half2 b_hi = __halves2half2(__ushort_as_half(0xBC80), __ushort_as_half(0xBC80));  // -1.125
    w[0] = __hfma2(as_h2(l02), s_lo, b_lo);
    w[1] = __hfma2(as_h2(l13), s_lo, b_lo);
    w[2] = __hfma2(as_h2(h02), s_hi, b_hi);
    w[3] = __hfma2(as_h2(h13), s_hi, b_hi);
}

// Q8_0: one 32-bit word holding int8 codes (q0, q1, q2, q3) -> two half2
// weights w[0] = (q0, q2) / 1024, w[1] = (q1, q3) / 1024.  Biasing each byte by
// +128 (XOR 0x80) makes it an unsigned mantissa: 0x6400 | (q + 128) = 1152 + q.
__device__ __forceinline__ void unpack_q8_word(uint32_t v, __half2 (&w)[2])
{
    const uint32_t u = v ^ 0x80808080u;
    const uint32_t h02 = __byte_perm(u, 0x64646464u, 0x4240);   // (0x64|b0, 0x64|b2)
    const uint32_t h13 = __byte_perm(u, 0x64646464u, 0x4341);   // (0x64|b1, 0x64|b3)
    // (1152 + q) / 1024 - 1.125 = q / 1024
    const __half2 s = __halves2half2(__ushort_as_half(0x1400), __ushort_as_half(0x1400));  // 2^-10
    const __half2 b = __halves2half2(__ushort_as_half(0xBC80), __ushort_as_half(0xBC80));  // -1.125
    w[0] = __hfma2(as_h2(h02), s, b);
    w[1] = __hfma2(as_h2(h13), s, b);
}

// Plain 2-bit: one 32-bit word of code bytes (b0, b1, b2, b3), each holding
// four codes c in 0..3 at bits 0-1, 2-3, 4-5, 6-7 (planes 0..3) -> eight half2
// weights (c - 2) / 32:
//   w[2p] = (plane p of b0, plane p of b2)   w[2p+1] = (plane p of b1, plane p of b3)
// Plane p lands in the mantissa as c * 4^p: 0x6400 | (c << 2p) is the half
// 1024 + c * 4^p, and (1024 + c * 4^p) * 2^-(2p+5) - (2^(5-2p) + 1/16) =
// (c - 2) / 32, a value fp16 holds exactly, so one HFMA2 per pair is exact.
__device__ __forceinline__ void unpack_q2_word(uint32_t v, __half2 (&w)[8])
{
    const uint32_t magic = 0x64006400u;
    const uint32_t v8 = v >> 8;
    constexpr unsigned short kScale[4] = {0x2800, 0x2000, 0x1800, 0x1000};   // 2^-5, 2^-7, 2^-9, 2^-11
    constexpr unsigned short kBias[4] = {0xD002, 0xC808, 0xC020, 0xB880};    // -32.0625, -8.0625, -2.0625, -0.5625
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t mask = 0x00030003u << (2 * p);
        const __half2 s = __halves2half2(__ushort_as_half(kScale[p]), __ushort_as_half(kScale[p]));
        const __half2 b = __halves2half2(__ushort_as_half(kBias[p]), __ushort_as_half(kBias[p]));
        w[2 * p] = __hfma2(as_h2(and_or(v, mask, magic)), s, b);
        w[2 * p + 1] = __hfma2(as_h2(and_or(v8, mask, magic)), s, b);
    }
}

// ---- Q8_1 activations (8-bit codes per block of 32) ---------------------------------
//
// Per block of 32 activations, decided in fp32 with round-to-nearest: amax =
// max |x|, d = amax / 127, id = 1 / d (0 for an all-zero block), code =
// round(x * id) with ties away from zero.  The block keeps d rounded to fp16
// (its stored scale) and the sum of its codes (for the -8 * sum(q) term of a
// Q4_0 dot).  Quantising the activations this way before an int8 dot is what
// llama.cpp and the sm8x kernel do (sm8x-bench, "Our kernel does what
// llama.cpp does").

// One 8-activation chunk (16 bytes of fp16) of a 32-block whose four chunks are
// held by lanes 4l..4l+3 of the warp.  Every lane of the warp calls this (lanes
// without a chunk pass zeros).  Returns the chunk's eight codes in memory
// order; dq and sumq receive the block's fp16-rounded scale and code sum.
__device__ __forceinline__ uint2 q8_1_chunk(uint4 xv, float &dq, int &sumq)
{
    float f[8];
    const uint32_t wv[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __half22float2(as_h2(wv[k]));
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __frcp_rn(d) : 0.0f;
    int s = 0;
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int code = static_cast<int>(roundf(__fmul_rn(f[i], id)));
        s += code;
        packed[i >> 2] |= (static_cast<uint32_t>(code) & 0xffu) << (8 * (i & 3));
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    sumq = s;
    dq = __half2float(__float2half_rn(d));
    return make_uint2(packed[0], packed[1]);
}

// d = sum over four bytes of a (unsigned) times b (signed), plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

}  // namespace qmv
