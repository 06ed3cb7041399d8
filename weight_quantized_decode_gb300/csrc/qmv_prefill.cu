// qmv_prefill.cu -- Q4_0 / Q8_0 prefill GEMM on the 5th-generation tensor
// cores (tcgen05.mma with fp32 accumulators in tensor memory), sm_103a; also
// the several-token decode calls the launch rule sends here.
//
//   y[m][n] = sum_k x[m][k] * w[n][k]     (tokens m; W in GGUF Q4_0 or Q8_0)
//
// Prior art on the pages: the bakeoff's tc_q4 contender, which dequantises a
// weight tile into shared memory and multiplies it with 16x16x16 WMMA
// fragments (volta-kernel-bakeoff, "What's in the race"), and the Marlin-style
// plan of "What we'd do next" item 3 (dequantise inside the tensor-core
// multiply itself).  The GB300 form:
//
//   * One CTA computes a 128-row (weights) x TN-column (tokens) tile of y^T in
//     tensor memory (one or two such weight tiles): weights are the MMA's M
//     side (128 lanes), tokens its N side (16, or 64..256 columns of fp32).
//   * The dequantised weights never touch shared memory: the dequantising
//     warps write them straight into tensor memory (tcgen05.st), and the MMA
//     reads its A operand from there.  Shared memory then carries only the
//     packed weights and the activation tiles.
//   * Roles by warp: the dequantising warps (8; 16 in 16-token tiles) -- warp
//     w writes tensor-memory lane quarter w mod 4, the only lanes its
//     sub-partition can reach; then the MMA warp, which allocates tensor memory
//     and issues the MMAs from one elected lane; then two copy producers, one
//     streaming packed 128-row x 256-K weight tiles (144 bytes per row for
//     Q4_0, 272 for Q8_0) and one 64-K activation tiles, with TMA tensor
//     copies into their own shared-memory rings; the activation tiles land in
//     the 128-byte-swizzled K-major layout the tensor core reads.  The MMA and
//     copy loops run as whole warps (warp-collective waits, an elected issuer).
//   * Dequantisation uses fp16 bit tricks (Q4_0: 0x6400|n, w = (c - 8) * d;
//     Q8_0: 0x64 above the sign-flipped code, w = q * d), one 32-weight block
//     per thread and atom, computed before the wait for its tensor-memory slot
//     and stored as 16 columns of half2.
//   * tcgen05.mma (kind::f16, 128 x TN x 16, A from tensor memory) four times
//     per 64-K atom; a ring slot holds KSUB atoms (4, 2 or 1 for 16/64-, 128-
//     and wider token tiles); tcgen05.commit releases the slot's activation
//     tile and weight atoms, and finally signals the epilogue.
//   * 16-token tiles may split K over a cluster of up to 8 CTAs along z; each
//     CTA stores its partial rows into their owner's shared memory and the
//     owner adds them in rank order after one cluster barrier.
//   * The epilogue reads the accumulators with tcgen05.ld (warp w reads lane
//     quarter w mod 4, the warps of a quarter split the columns) and stores y
//     with coalesced fp32 stores.
// Operands are fp16: the activations arrive as fp16 and each dequantised
// weight is rounded once to fp16.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/qmv.h"
#include "qmv_common.cuh"
#include "qmv_launch.h"
#include "qmv_prefill.h"
#include "qmv_prefill_plan.h"

namespace qmv {

namespace {

// Threads of a CTA: the dequantising warps (8; 16 in the 16-token tiles,
// whose kernels need few registers and whose slots are whole 256-K chunks),
// then the MMA warp and the two copy producers.
constexpr int kThreads = kPrefillThreads;                          // 11 warps
constexpr int kThreadsSmall = prefill_threads(true);               // 19 warps

struct PrefillParams {
    float *y;
    int *status;
    int64_t N, K, M;
    int TN;            // token columns per tile = the MMA's N (multiple of 64, <= 256)
    int WT;            // 128-row weight tiles per CTA (1 or 2)
    int NW;            // packed-weight ring slots (256-K chunks of WT tiles)
    int NSA;           // weight-atom ring slots (tensor memory)
    int NSB;           // activation ring slots (shared memory)
    int KSUB;          // 64-K atoms per slot (1, 2 or 4): MMAs per barrier round = 4 * KSUB * WT
    int cluster;       // CTAs per cluster sharing each activation tile by multicast (1 or 2)
    uint32_t tmem_cols;
    int test_skip_copy;   // failure-detection test only: CTA (0, 0) never requests its first packed tile
    unsigned long long *phase;   // phase-timeline builds only (QMV_PHASE_STAMPS): [count, records...]
    unsigned int phase_seq;
};

#ifdef QMV_PHASE_STAMPS
// Phase-timeline record (QMV_PHASE_STAMPS builds): seq << 32 | CTA, global-timer
// stamps at entry, after set-up, at the first MMA, after the last commit, when
// the accumulator is complete and at exit, and the SM clock cycles between the
// first MMA and the last commit.
constexpr int kPrefillPhaseWords = 8;
constexpr int kPrefillPhaseCap = 1 << 16;
constexpr int kTraceSlotsDev = 128;
constexpr int kTraceCols = 8;
__device__ unsigned long long g_prefill_trace_dev[kTraceSlotsDev * kTraceCols];
#define QMV_TRACE(j, k)                                                                                     \
    do {                                                                                                  \
        if (blockIdx.x == 0 && blockIdx.y == 0 && (j) < kTraceSlotsDev)                                   \
            g_prefill_trace_dev[(j) * kTraceCols + (k)] = global_timer_ns();                              \
    } while (0)
#else
#define QMV_TRACE(j, k) \
    do {                \
    } while (0)
#endif

// ---- tcgen05 / TMA wrappers -------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// tma_load_2d delivered to every CTA of `mask` in the cluster, at the same
// shared-memory offsets (destination and barrier) in each.
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                               uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the canonical layout a TMA SWIZZLE_128B box produces).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 bytes
    d |= static_cast<uint64_t>(1) << 46;                 // descriptor version for sm_100 family
    d |= static_cast<uint64_t>(2) << 61;                 // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 accumulator,
// M = 128, N = tn.
__host__ __device__ __forceinline__ uint32_t f16_idesc(int tn)
{
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                    // A, B format: f16
           | (static_cast<uint32_t>(tn >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(kBM >> 4) << 24);  // M / 16
}

// Four K=16 steps over one 64-K atom with A in tensor memory: A advances by
// 8 columns (16 fp16) and the B descriptor by 32 bytes (2 in its 16-byte
// address field) per step.  `first` clears the accumulator.
__device__ __forceinline__ void mma_f16_atom_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                                bool first)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        ".reg .b32 a1, a2, a3;\n\t"
        ".reg .b64 b1, b2, b3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, 0, 0;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n\t}"
        ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(first ? 0 : 1)
        : "memory");
}

// 16 consecutive 32-bit tensor-memory columns of this thread's lane (the warp
// writes its lane quarter: taddr carries the quarter's first lane).
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Arrive on the barrier at this offset in every CTA of `mask` once the MMAs
// issued so far are complete.
__device__ __forceinline__ void mma_commit_mc(uint64_t *bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(smem_u32(bar)), "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Warp-collective wait_or_abort: every lane calls it and gets the same answer.
// The common case (phase already complete) stays converged; otherwise lane 0
// waits and the others follow.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                   int *status)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok)   // the phase has completed: every lane observes it before going on
        while (!mbar_try_wait(bar, parity)) {
        }
    return ok;
}

// Dequantise one 32-weight Q4_0 block (scale bits `dbits`, codes in 4 aligned
// words q[0..3] = qs[0..15]) into 32 fp16 weights in natural K order:
// out[0..3] = elements 0..7, out[4..7] = 8..15, out[8..11] = 16..23,
// out[12..15] = 24..31 (each entry a half2 of consecutive elements).
__device__ __forceinline__ void dequant_block_f16(uint32_t dbits, const uint32_t (&q)[4], uint32_t (&out)[16])
{
    const __half d = __ushort_as_half(static_cast<unsigned short>(dbits));
    const __half2 d2 = __halves2half2(d, d);
    const uint32_t magic = 0x64006400u;
    const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));    // 1/16
    const __half2 m72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));    // -72
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t t01 = __byte_perm(q[i], 0u, 0x4140);   // (b0, b1) in the low bytes of two halves
        const uint32_t t23 = __byte_perm(q[i], 0u, 0x4342);   // (b2, b3)
        const __half2 lo01 = __hsub2(as_h2(and_or(t01, 0x000F000Fu, magic)), c1032);      // c - 8, exact
        const __half2 lo23 = __hsub2(as_h2(and_or(t23, 0x000F000Fu, magic)), c1032);
        const __half2 hi01 = __hfma2(as_h2(and_or(t01, 0x00F000F0u, magic)), s16, m72);   // c - 8, exact
        const __half2 hi23 = __hfma2(as_h2(and_or(t23, 0x00F000F0u, magic)), s16, m72);
        const __half2 a = __hmul2(lo01, d2), b = __hmul2(lo23, d2);
        const __half2 c = __hmul2(hi01, d2), e = __hmul2(hi23, d2);
        // word i holds qs[4i..4i+3]: elements 4i..4i+3 (low) and 16+4i..16+4i+3 (high)
        out[2 * i] = *reinterpret_cast<const uint32_t *>(&a);
        out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&b);
        out[8 + 2 * i] = *reinterpret_cast<const uint32_t *>(&c);
        out[8 + 2 * i + 1] = *reinterpret_cast<const uint32_t *>(&e);
    }
}

// Dequantise one 34-byte Q8_0 block (fp16 scale, then 32 int8 codes) from
// the nine 32-bit words of a packed 256-K row chunk that hold it: EVEN blocks
// start a word (scale in the low half of v[0], code pair j in v[(j + 1) / 2]),
// odd blocks start half a word in (scale in the upper half of v[0], code
// pair j in v[1 + j / 2]).  A code byte b becomes the fp16 1024 + (b ^ 0x80)
// = 1152 + code (the sign flip makes it unsigned, 0x64 its exponent byte);
// subtracting 1152 is exact, and the product with the scale is rounded once.
// Output j is the half2 of elements (2j, 2j + 1).
template <bool EVEN>
__device__ __forceinline__ void dequant_block_q8_f16(const uint32_t *v, uint32_t (&out)[16])
{
    const uint32_t dbits = EVEN ? (v[0] & 0xffffu) : (v[0] >> 16);
    const __half d = __ushort_as_half(static_cast<unsigned short>(dbits));
    const __half2 d2 = __halves2half2(d, d);
    const __half2 c1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t word = EVEN ? v[(j + 1) >> 1] : v[1 + (j >> 1)];
        // EVEN: pair j sits in bytes 2, 3 (j even) or 0, 1 (j odd) of its word
        const uint32_t sel = EVEN ? ((j & 1) ? 0x4140u : 0x4342u) : ((j & 1) ? 0x4342u : 0x4140u);
        const uint32_t t = __byte_perm(word ^ 0x80808080u, 0x64646464u, sel);
        const __half2 c = __hsub2(as_h2(t), c1152);   // the codes, exact
        const __half2 w = __hmul2(c, d2);
        out[j] = *reinterpret_cast<const uint32_t *>(&w);
    }
}

// 16 consecutive 32-bit tensor-memory columns of this thread's lane into v.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Sixteen floats (16-byte aligned) to this shared-memory location of cluster
// CTA `rank`.
__device__ __forceinline__ void st_cluster_f32x16(const float *local, uint32_t rank, const uint32_t (&v)[16])
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(remote + 16u * i), "r"(v[4 * i]),
                     "r"(v[4 * i + 1]), "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                     : "memory");
}

// SMALL: 16-token tiles (one weight tile, no multicast), which may be split
// along K over a cluster; the other tiles compile without that code.
template <int WT, int CL, int FMT, bool SMALL>
__global__ void __launch_bounds__(SMALL ? kThreadsSmall : kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const PrefillParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment of the activation tiles (required by the 128-byte swizzle).
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int NW = p.NW, NSA = p.NSA, NSB = p.NSB, TN = p.TN, KSUB = p.KSUB;
    // Equal ring depths without a cluster: one set of release barriers
    // (aempty) serves both rings, and a slot is released with one commit.
    const bool one_ring = NSA == NSB && CL == 1;
    uint32_t crank = 0u;
    if constexpr (CL > 1) crank = cluster_rank();
    const uint16_t cmask = static_cast<uint16_t>((1u << CL) - 1u);
    const int b_atom_bytes = TN * kKB * 2;                  // one 64-K activation atom
    const int b_slot_bytes = KSUB * b_atom_bytes;
    // One weight row's 256-K chunk (144 bytes Q4_0, 272 Q8_0) and the TMA
    // coordinate step per chunk (bytes for Q4_0; the Q8_0 map counts 16-bit
    // elements, its 272-byte box row being wider than a box's 256 elements).
    constexpr int kRowB = prefill_row_bytes(FMT);
    constexpr int kTileB = kBM * kRowB;
    constexpr int kWCoord = FMT == kPfQ8_0 ? kRowB / 2 : kRowB;
    const int w_slot_bytes = WT * kTileB;                   // one 256-K chunk of the CTA's WT weight tiles
    uint8_t *b_tiles = smem;
    uint8_t *w_tiles = b_tiles + NSB * b_slot_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_tiles + NW * w_slot_bytes);
    uint64_t *wfull = bars;             // [NW]
    uint64_t *wempty = wfull + NW;      // [NW]
    uint64_t *afull = wempty + NW;      // [NSA] dequantised atoms written to tensor memory
    uint64_t *aempty = afull + NSA;     // [NSA] the slot's MMAs are done: its weight atoms are free
    uint64_t *bfull = aempty + NSA;     // [NSB] activation atoms landed
    uint64_t *bempty = bfull + NSB;     // [NSB] every cluster CTA's MMAs of the slot are done: its
                                        //       activation tile may be refilled in all of them
    uint64_t *accfull = bempty + NSB;   // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accfull + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // split K: the receive buffer for other CTAs' partial rows (16-token tiles)
    float *red_buf = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + 512);

    constexpr int kDeqWarps = SMALL ? 16 : 8;                  // warps 0 .. kDeqWarps-1
    constexpr int kMmaWarp = kDeqWarps, kWProducerWarp = kDeqWarps + 1, kXProducerWarp = kDeqWarps + 2;
    constexpr int kWarps = kDeqWarps + 3;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
#ifdef QMV_PHASE_STAMPS
    __shared__ unsigned long long phs[7];   // entry, setup, first MMA, last commit, acc ready, clk0, clk1
    if (threadIdx.x == 0) phs[0] = global_timer_ns();
#endif
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBM * WT;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TN;
    // Split K (16-token tiles): CTA z of the cluster along z takes chunks
    // [c_first, c_first + nC).
    const int64_t chunks_all = p.K / kKChunk;
    const int c_first = SMALL ? static_cast<int>(chunks_all * blockIdx.z / gridDim.z) : 0;
    const int nC = SMALL ? static_cast<int>(chunks_all * (blockIdx.z + 1) / gridDim.z) - c_first
                         : static_cast<int>(chunks_all);            // packed 256-K chunks
    const int nK = SMALL ? nC * (kKChunk / kKB) / KSUB : static_cast<int>(p.K / (kKB * KSUB));   // slots

    if (threadIdx.x == 0) {
        for (int i = 0; i < NW; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], kDeqWarps);
        }
        for (int i = 0; i < NSA; ++i) {
            mbar_init(&afull[i], kDeqWarps);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < NSB; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], CL);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, p.tmem_cols);
    tc_fence_before();
    // The peer CTAs' barriers are initialised before any multicast copy or
    // commit can reach them.
    if constexpr (CL > 1)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Columns [t * TN, (t + 1) * TN) hold weight tile t's accumulator; weight
    // atom (slot s, atom a, tile t) follows at A0 + ((s * KSUB + a) * WT + t) * 32,
    // A0 = WT * TN rounded up to 32 columns (16-token tiles: 32).
    const uint32_t tmem_a0 = tmem_base + (SMALL ? 32u : static_cast<uint32_t>(WT * TN));
#ifdef QMV_PHASE_STAMPS
    if (threadIdx.x == 0) phs[1] = global_timer_ns();
#endif
    // The next kernel of the stream may be scheduled now (its CTAs start on
    // free SMs and stream their own weights); it reads what this kernel
    // writes only after its own griddepcontrol.wait.
    pdl_allow_next_grid();

    bool ok = true;
    if (warp == kWProducerWarp) {
        // ---------------- packed weights: TMA tensor copies, NW deep ----------------
        // The whole warp runs the loop; one elected lane issues the copies.
        // W is never written by the kernel before this one (a documented
        // condition of the call), so its copies do not wait for it.
        int issued = 0, slot = 0;
        uint32_t phase = 1;            // an empty slot starts "released"
        for (int c = 0; c < nC; ++c) {
            if (!warp_wait_or_abort(&wempty[slot], phase, abort_flag, p.status)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(&wfull[slot], static_cast<uint32_t>(w_slot_bytes));
                // (test only) the first chunk of CTA (0, 0) is expected but never
                // requested, so the waits on it run out and the CTA aborts
                if (!(p.test_skip_copy && c == 0 && blockIdx.x == 0 && blockIdx.y == 0))
                    for (int t = 0; t < WT; ++t)   // rows past N read zeros
                        tma_load_2d(w_tiles + slot * w_slot_bytes + t * kTileB, &wmap, (c_first + c) * kWCoord,
                                    static_cast<int>(n0) + t * kBM, &wfull[slot]);
            }
            __syncwarp();
            ++issued;
            if (++slot == NW) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (!ok && lane == 0)   // let the copies already requested land before the CTA exits
            for (int c = (issued > NW ? issued - NW : 0); c < issued; ++c)
                mbar_wait_bounded(&wfull[c % NW], (c / NW) & 1, nullptr);
    } else if (warp == kXProducerWarp) {
        // ---------------- activations: TMA tensor copies, one per atom ----------------
        // With a cluster, this CTA loads rows [crank * TN / CL, ...) of every
        // atom and multicasts them into the same offsets of all the cluster's
        // CTAs; a slot is refilled once every CTA's MMAs have released it.
        // The whole warp runs the loop; one elected lane issues the copies.
        pdl_wait_prior_grid();
        const int rows = TN / CL;
        const int row_off_bytes = static_cast<int>(crank) * rows * 128;
        int issued = 0, s = 0;
        uint32_t phase = 1;
        for (int j = 0; j < nK; ++j) {
            if (!warp_wait_or_abort(one_ring ? &aempty[s] : &bempty[s], phase, abort_flag, p.status)) {
                ok = false;
                break;
            }
            if (elect_one()) {
                mbar_arrive_expect_tx(&bfull[s], b_slot_bytes);
                for (int a = 0; a < KSUB; ++a) {
                    uint8_t *dst = b_tiles + s * b_slot_bytes + a * b_atom_bytes + row_off_bytes;
                    const int xk = ((SMALL ? c_first * (kKChunk / kKB) : 0) + j * KSUB + a) * kKB;
                    if constexpr (CL > 1)
                        tma_load_2d_mc(dst, &xmap, xk, static_cast<int>(m0) + static_cast<int>(crank) * rows,
                                       &bfull[s], cmask);
                    else
                        tma_load_2d(dst, &xmap, xk, static_cast<int>(m0), &bfull[s]);
                }
                QMV_TRACE(j, 0);
            }
            __syncwarp();
            ++issued;
            if (++s == NSB) {
                s = 0;
                phase ^= 1u;
            }
        }
        if (!ok && lane == 0)
            for (int j = (issued > NSB ? issued - NSB : 0); j < issued; ++j)
                mbar_wait_bounded(&bfull[j % NSB], (j / NSB) & 1, nullptr);
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue: the warp runs the loop, one elected lane issues ----------------
        const uint32_t idesc = f16_idesc(TN);
        // Descriptor of activation slot 0's first atom; a slot (or a 16-wide
        // K step: 32 bytes = 2 in the 16-byte address field) is a plain addition.
        const uint64_t b_desc0 = sw128_desc(smem_u32(b_tiles));
        const uint64_t b_step = static_cast<uint64_t>(b_slot_bytes) >> 4;
        const uint64_t b_atom_step = static_cast<uint64_t>(b_atom_bytes) >> 4;
        const uint32_t a_slot_cols = static_cast<uint32_t>(KSUB * WT * kAtomCols);
        int committed = 0, sa = 0, sb = 0;
        uint32_t pha = 0, phb = 0;
        uint64_t b_desc = b_desc0;
        uint32_t a_tmem = tmem_a0;
        for (int j = 0; j < nK; ++j) {
            if (!warp_wait_or_abort(&bfull[sb], phb, abort_flag, p.status)) {
                ok = false;
                break;
            }
            if (lane == 0) QMV_TRACE(j, 1);
            if (!warp_wait_or_abort(&afull[sa], pha, abort_flag, p.status)) {
                ok = false;
                break;
            }
            // Order the MMAs after the barrier waits (the tcgen05 ops are
            // asynchronous to this thread) and after the weight atoms'
            // tensor-memory stores the barrier published.
            tc_fence_after();
            // The same lane issues every MMA and every commit: a commit tracks
            // the MMAs its own thread issued.
            if (elect_one()) {
                QMV_TRACE(j, 2);
#ifdef QMV_PHASE_STAMPS
                if (j == 0) {
                    phs[2] = global_timer_ns();
                    phs[5] = clock64();
                }
#endif
                for (int a = 0; a < KSUB; ++a)
                    for (int t = 0; t < WT; ++t)
                        mma_f16_atom_ts(tmem_base + static_cast<uint32_t>(t * TN),
                                        a_tmem + static_cast<uint32_t>((a * WT + t) * kAtomCols),
                                        b_desc + a * b_atom_step, idesc, j == 0 && a == 0);
                mma_commit(&aempty[sa]);
                if constexpr (CL > 1)
                    mma_commit_mc(&bempty[sb], cmask);
                else if (!one_ring)
                    mma_commit(&bempty[sb]);
                QMV_TRACE(j, 3);
            }
            __syncwarp();
            ++committed;
            if (++sa == NSA) {
                sa = 0;
                pha ^= 1u;
                a_tmem = tmem_a0;
            } else {
                a_tmem += a_slot_cols;
            }
            if (++sb == NSB) {
                sb = 0;
                phb ^= 1u;
                b_desc = b_desc0;
            } else {
                b_desc += b_step;
            }
        }
        if (elect_one()) {
            mma_commit(accfull);
#ifdef QMV_PHASE_STAMPS
            phs[3] = global_timer_ns();
            phs[6] = clock64();
#endif
        }
        __syncwarp();
        if (!ok && committed > 0 && lane == 0) mbar_wait_bounded(accfull, 0, nullptr);
    } else if constexpr (SMALL) {
        // ---------------- dequantising warps 0..15, 16-token tiles ----------------
        // One weight tile and one ring slot per 256-K chunk.  Four warps per
        // tensor-memory lane quarter (warp w writes lanes 32 * (w mod 4) .. +31):
        // part p = w / 4 dequantises blocks p and p + 4 of the chunk (atoms
        // p / 2 and p / 2 + 2, half p mod 2), loading only those blocks' words.
        constexpr int kBW = FMT == kPfQ8_0 ? 9 : 5;   // 32-bit words holding one block
        const int quarter = warp & 3;
        const int part = warp >> 2;
        const int r = 32 * quarter + lane;         // weight row within the tile
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
        int slot = 0, sa = 0;
        uint32_t wpar = 0, apar = 1;
#ifdef QMV_PHASE_STAMPS
        int jd = 0;   // ring rounds published (trace only)
#endif
        for (int c = 0; ok && c < nC; ++c) {
            if (!warp_wait_or_abort(&wfull[slot], wpar, abort_flag, p.status)) {
                ok = false;
                break;
            }
#ifdef QMV_PHASE_STAMPS
            if (warp == 0 && lane == 0) QMV_TRACE(jd, 6);
#endif
            const uint32_t *row = reinterpret_cast<const uint32_t *>(w_tiles + slot * w_slot_bytes + r * kRowB);
            uint32_t v[2][kBW];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int b = part + 4 * k;   // block of the chunk
                // Q4_0: 18-byte blocks, block b from word 9 (b / 2) + 4 (b mod 2);
                // Q8_0: 34-byte blocks, from word 17 (b / 2) + 8 (b mod 2)
                const uint32_t *w = row + (FMT == kPfQ8_0 ? 17 * (b >> 1) + 8 * (b & 1) : 9 * (b >> 1) + 4 * (b & 1));
#pragma unroll
                for (int i = 0; i < kBW; ++i) v[k][i] = w[i];
            }
            // Hand the slot back once this thread's reads of it are done (the
            // words consumed into a register; fence.proxy.async orders the
            // generic-proxy reads before the producer's next copy).
            {
                uint32_t x = 0u;
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int i = 0; i < kBW; ++i) x ^= v[k][i];
                asm volatile("" ::"r"(x) : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[slot]);
            if (++slot == NW) {
                slot = 0;
                wpar ^= 1u;
            }
            uint32_t f2[2][16];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if constexpr (FMT == kPfQ8_0) {
                    if ((part & 1) == 0)
                        dequant_block_q8_f16<true>(v[k], f2[k]);
                    else
                        dequant_block_q8_f16<false>(v[k], f2[k]);
                } else {
                    uint32_t q[4], dbits;
                    if ((part & 1) == 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = __byte_perm(v[k][i], v[k][i + 1], 0x5432);
                        dbits = v[k][0] & 0xffffu;
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = v[k][i + 1];
                        dbits = v[k][0] >> 16;
                    }
                    dequant_block_f16(dbits, q, f2[k]);
                }
            }
#ifdef QMV_PHASE_STAMPS
            if (warp == 0 && lane == 0) QMV_TRACE(jd, 7);
#endif
            if (!warp_wait_or_abort(&aempty[sa], apar, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
#ifdef QMV_PHASE_STAMPS
            if (warp == 0 && lane == 0) QMV_TRACE(jd, 4);
#endif
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int b = part + 4 * k;
                tmem_st_16cols(tmem_a0 + lane_base + static_cast<uint32_t>((sa * 4 + (b >> 1)) * kAtomCols + 16 * (b & 1)),
                               f2[k]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[sa]);
#ifdef QMV_PHASE_STAMPS
            if (warp == 0 && lane == 0) QMV_TRACE(jd, 5);
            ++jd;
#endif
            if (++sa == NSA) {
                sa = 0;
                apar ^= 1u;
            }
        }
    } else if constexpr (FMT == kPfQ8_0) {
        // ---------------- dequantising warps 0..7, Q8_0 ----------------
        // The same split as for Q4_0 (warp w: lane quarter w mod 4, block
        // parity w / 4 of every 64-K atom); a thread loads the nine words of
        // each of its four blocks of the chunk (words 17 * sub + 8 * hsel + i).
        const int quarter = warp & 3;
        const int hsel = warp >> 2;
        const int r = 32 * quarter + lane;         // weight row within each tile
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
        int slot = 0, sa = 0, atom = 0;
        uint32_t wpar = 0, apar = 1;
        for (int c = 0; ok && c < nC; ++c) {
            if (!warp_wait_or_abort(&wfull[slot], wpar, abort_flag, p.status)) {
                ok = false;
                break;
            }
            uint32_t w[WT][36];
#pragma unroll
            for (int t = 0; t < WT; ++t) {
                const uint32_t *row =
                    reinterpret_cast<const uint32_t *>(w_tiles + slot * w_slot_bytes + t * kTileB + r * kRowB);
#pragma unroll
                for (int sub = 0; sub < 4; ++sub)
#pragma unroll
                    for (int i = 0; i < 9; ++i) w[t][9 * sub + i] = row[17 * sub + 8 * hsel + i];
            }
            // Hand the slot back once this thread's reads of it are done (the
            // words consumed into a register; fence.proxy.async orders the
            // generic-proxy reads before the producer's next copy).
            {
                uint32_t x4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int t = 0; t < WT; ++t)
#pragma unroll
                    for (int i = 0; i < 36; ++i) x4[i & 3] ^= w[t][i];
                asm volatile("" ::"r"(x4[0] ^ x4[1] ^ x4[2] ^ x4[3]) : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[slot]);
            if (++slot == NW) {
                slot = 0;
                wpar ^= 1u;
            }
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) {
                // dequantise first, then wait for the tensor-memory slot
                uint32_t f[WT][16];
#pragma unroll
                for (int t = 0; t < WT; ++t) {
                    if (hsel == 0)
                        dequant_block_q8_f16<true>(&w[t][9 * sub], f[t]);
                    else
                        dequant_block_q8_f16<false>(&w[t][9 * sub], f[t]);
                }
                if (atom == 0) {
                    if (!warp_wait_or_abort(&aempty[sa], apar, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
#pragma unroll
                for (int t = 0; t < WT; ++t)
                    tmem_st_16cols(tmem_a0 + lane_base +
                                       static_cast<uint32_t>(((sa * KSUB + atom) * WT + t) * kAtomCols + 16 * hsel),
                                   f[t]);
                if (++atom == KSUB) {
                    atom = 0;
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&afull[sa]);
                    if (++sa == NSA) {
                        sa = 0;
                        apar ^= 1u;
                    }
                }
            }
        }
    } else {
        // ---------------- dequantising warps 0..7 ----------------
        // Warp w writes lanes 32 * (w mod 4) .. + 31 (weight rows r of each of
        // the WT tiles) of tensor memory, the even (w < 4) or odd (w >= 4)
        // block of each 64-K atom.
        const int quarter = warp & 3;
        const int hsel = warp >> 2;
        const int r = 32 * quarter + lane;         // weight row within each tile
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
        int slot = 0, sa = 0, atom = 0;
        uint32_t wpar = 0, apar = 1;
#ifdef QMV_PHASE_STAMPS
        int jd = 0;   // ring rounds published (trace only)
#endif
        for (int c = 0; ok && c < nC; ++c) {
            if (!warp_wait_or_abort(&wfull[slot], wpar, abort_flag, p.status)) {
                ok = false;
                break;
            }
#ifdef QMV_PHASE_STAMPS
            if (warp == 0 && lane == 0) QMV_TRACE(jd, 6);
#endif
            // this thread's row of each weight tile: 36 words (a 256-K chunk)
            uint32_t w[WT][36];
#pragma unroll
            for (int t = 0; t < WT; ++t) {
                const uint8_t *src = w_tiles + slot * w_slot_bytes + t * kPackedTileBytes + r * kPackedRowBytes;
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src + 16 * i);
                    w[t][4 * i] = v.x;
                    w[t][4 * i + 1] = v.y;
                    w[t][4 * i + 2] = v.z;
                    w[t][4 * i + 3] = v.w;
                }
            }
            // Hand the slot back only once this thread's reads of it are done:
            // the words are consumed (into a register, or by the dequantising
            // arithmetic), and fence.proxy.async orders the reads (generic
            // proxy) before the producer's next copy into the slot (async
            // proxy).
            int wslot = slot;
            auto release_w = [&](bool consumed) {
                if (!consumed) {
                    uint32_t x4[4] = {0u, 0u, 0u, 0u};   // four short XOR chains
#pragma unroll
                    for (int t = 0; t < WT; ++t)
#pragma unroll
                        for (int i = 0; i < 36; ++i) x4[i & 3] ^= w[t][i];
                    asm volatile("" ::"r"(x4[0] ^ x4[1] ^ x4[2] ^ x4[3]) : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&wempty[wslot]);
            };
            if (++slot == NW) {
                slot = 0;
                wpar ^= 1u;
            }
            if (WT == 1 && KSUB == 4) {
                // One slot is the whole 256-K chunk (64-token tiles): all four
                // blocks are dequantised before the slot wait, four independent
                // chains the scheduler can interleave.
                uint32_t f4[4][16];
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    const int h = 9 * sub;
                    uint32_t q[4], dbits;
                    if (hsel == 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = __byte_perm(w[0][h + i], w[0][h + i + 1], 0x5432);
                        dbits = w[0][h] & 0xffffu;
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = w[0][h + 5 + i];
                        dbits = w[0][h + 4] >> 16;
                    }
                    dequant_block_f16(dbits, q, f4[sub]);
                }
                // Every word this thread loaded has fed the arithmetic above
                // (values 0, 2, 4, 6 of a block depend on all its code words
                // and its scale), so the loads are complete.
#pragma unroll
                for (int sub = 0; sub < 4; ++sub)
                    asm volatile("" ::"r"(f4[sub][0]), "r"(f4[sub][2]), "r"(f4[sub][4]), "r"(f4[sub][6]) : "memory");
                release_w(true);
#ifdef QMV_PHASE_STAMPS
                if (warp == 0 && lane == 0) QMV_TRACE(jd, 7);
#endif
                if (!warp_wait_or_abort(&aempty[sa], apar, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#ifdef QMV_PHASE_STAMPS
                if (warp == 0 && lane == 0) QMV_TRACE(jd, 4);
#endif
#pragma unroll
                for (int sub = 0; sub < 4; ++sub)
                    tmem_st_16cols(tmem_a0 + lane_base + static_cast<uint32_t>((sa * 4 + sub) * kAtomCols + 16 * hsel),
                                   f4[sub]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[sa]);
#ifdef QMV_PHASE_STAMPS
                if (warp == 0 && lane == 0) QMV_TRACE(jd, 5);
                ++jd;
#endif
                if (++sa == NSA) {
                    sa = 0;
                    apar ^= 1u;
                }
                continue;
            }
            release_w(false);
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) {
                // Dequantise block 2*sub + hsel of each weight tile into
                // registers first (even blocks start 2 bytes into word 9*sub):
                // the arithmetic overlaps the wait for the tensor-memory slot,
                // and only the stores remain once the slot is free.
                const int h = 9 * sub;
                uint32_t f[WT][16];
#pragma unroll
                for (int t = 0; t < WT; ++t) {
                    uint32_t q[4], dbits;
                    if (hsel == 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = __byte_perm(w[t][h + i], w[t][h + i + 1], 0x5432);
                        dbits = w[t][h] & 0xffffu;
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) q[i] = w[t][h + 5 + i];
                        dbits = w[t][h + 4] >> 16;
                    }
                    dequant_block_f16(dbits, q, f[t]);
                }
                if (atom == 0) {
                    // the slot's previous atoms have been read by their MMAs
                    if (!warp_wait_or_abort(&aempty[sa], apar, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#ifdef QMV_PHASE_STAMPS
                    if (warp == 0 && lane == 0) QMV_TRACE(jd, 4);
#endif
                }
                // elements 2j, 2j+1 of the block -> column 16 * hsel + j of the atom
#pragma unroll
                for (int t = 0; t < WT; ++t)
                    tmem_st_16cols(tmem_a0 + lane_base +
                                       static_cast<uint32_t>(((sa * KSUB + atom) * WT + t) * kAtomCols + 16 * hsel),
                                   f[t]);
                if (++atom == KSUB) {
                    atom = 0;
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&afull[sa]);
#ifdef QMV_PHASE_STAMPS
                    if (warp == 0 && lane == 0) QMV_TRACE(jd, 5);
                    ++jd;
#endif
                    if (++sa == NSA) {
                        sa = 0;
                        apar ^= 1u;
                    }
                }
            }
        }
    }

    // ---------------- epilogue: every warp ----------------
    // Warp w reads TMEM lane quarter w mod 4; the warps of a quarter take the
    // 32-column chunks of the WT accumulators round-robin.  A role that gave
    // up skips it.
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (lane == 0) ok = ok && wait_or_abort(accfull, 0, abort_flag, p.status);
    ok = __shfl_sync(0xffffffffu, (ok && !*abort_flag) ? 1 : 0, 0) != 0;
    if (ok) {
        while (!mbar_try_wait_sleep(accfull, 0, kSuspendHintNs)) {
        }
        tc_fence_after();
#ifdef QMV_PHASE_STAMPS
        if (threadIdx.x == 0) phs[4] = global_timer_ns();
#endif
        const int quarter = warp & 3;
        const int nq = (kWarps - quarter + 3) / 4;   // warps in this quarter
        const int rank = warp >> 2;
        if constexpr (SMALL) {
            // 16-token tiles: the first warp of each lane quarter reads its 16
            // columns; with split K the partial tile goes to this CTA's shared
            // memory (the rings are idle now), row-major [128][TN].
            if (rank == 0) {
                uint32_t v[16];
                tmem_ld_16cols(tmem_base + (static_cast<uint32_t>(32 * quarter) << 16), v);
                const int rl = 32 * quarter + lane;
                const int64_t row = n0 + rl;
                if (gridDim.z > 1) {
                    // split K: store this partial row into its owner's receive
                    // buffer, slot of this CTA's rank
                    const int sk = static_cast<int>(gridDim.z);
                    const int owner = ((rl + 1) * sk - 1) / kBM;
                    const int rmax = (kBM + sk - 1) / sk;
                    const float *dst = red_buf + (static_cast<int>(blockIdx.z) * rmax + (rl - kBM * owner / sk)) * 16;
                    st_cluster_f32x16(dst, static_cast<uint32_t>(owner), v);
                } else if (row < p.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t m = m0 + i;
                        if (m < p.M) p.y[m * p.N + row] = __uint_as_float(v[i]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < WT; ++t) {
                const int64_t row = n0 + t * kBM + 32 * quarter + lane;
                for (int c0 = 32 * rank; c0 < TN; c0 += 32 * nq) {
                    uint32_t v[32];
                    tmem_ld_32cols(tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + t * TN + c0, v);
                    if (row < p.N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int64_t m = m0 + c0 + i;
                            if (m < p.M) p.y[m * p.N + row] = __uint_as_float(v[i]);
                        }
                    }
                }
            }
        }
    }
    if (SMALL && gridDim.z > 1) {
        // Split K (16-token tiles, one cluster along z): every CTA has stored
        // its partial rows into their owners' receive buffers (rows [128 z /
        // SK, 128 (z + 1) / SK) belong to CTA z); after the cluster barrier
        // CTA z adds its rows' partials in rank order (the same order on every
        // call) from its own shared memory and stores y.  Nothing reads another
        // CTA's shared memory after the barrier, so one barrier suffices.
        cluster_sync();
        const int sk = static_cast<int>(gridDim.z), z = static_cast<int>(blockIdx.z);
        const int r0 = kBM * z / sk, nr = kBM * (z + 1) / sk - r0;
        const int rmax = (kBM + sk - 1) / sk;
        for (int i = threadIdx.x; i < nr * 16; i += blockDim.x) {
            const int col = i / nr, rr = i - col * nr;
            float acc = 0.0f;
            for (int q = 0; q < sk; ++q) acc += red_buf[(q * rmax + rr) * 16 + col];
            const int64_t row = n0 + r0 + rr, m = m0 + col;
            if (ok && row < p.N && m < p.M) p.y[m * p.N + row] = acc;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    // No CTA leaves while a peer may still multicast into its shared memory or
    // arrive on its barriers.
    if constexpr (CL > 1) cluster_sync();
#ifdef QMV_PHASE_STAMPS
    if (threadIdx.x == 0 && p.phase) {
        // the end stamp is taken before the record's slot is claimed: the
        // atomic's round trip (every CTA on one counter) is not the kernel's
        const unsigned long long t_end = global_timer_ns();
        const unsigned long long i = atomicAdd(p.phase, 1ull);
        if (i < kPrefillPhaseCap) {
            unsigned long long *rec = p.phase + 1 + i * kPrefillPhaseWords;
            rec[0] = (static_cast<unsigned long long>(p.phase_seq) << 32) | (blockIdx.y * gridDim.x + blockIdx.x);
            rec[1] = phs[0];
            rec[2] = phs[1];
            rec[3] = phs[2];
            rec[4] = phs[3];
            rec[5] = phs[4];
            rec[6] = t_end;
            rec[7] = phs[6] - phs[5];
        }
    }
#endif
}

// ---- host side -------------------------------------------------------------------

#ifdef QMV_PHASE_STAMPS
__device__ unsigned long long g_prefill_phase[1 + static_cast<size_t>(kPrefillPhaseWords) * kPrefillPhaseCap];

std::atomic<unsigned> g_prefill_phase_seq{0};
#endif

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Ring depths, cluster size and tile forced for tests and sweeps:
// QMV_PREFILL_RING="NW,NS[,CL[,TN[,WT[,KSUB[,SK]]]]]" (packed-weight slots,
// activation slots, CTAs per cluster, token tile, weight tiles per CTA, atoms
// per slot, CTAs along K; NW below 1, NS below 2, CL other than 1 or 2, TN,
// WT, KSUB or SK of 0 keep the rule).
int ring_override(int which)
{
    static int v[7] = {0, 0, 0, 0, 0, 0, 0};
    static std::once_flag once;
    std::call_once(once, [] {
        const char *e = std::getenv("QMV_PREFILL_RING");
        if (!e) return;
        for (int i = 0; i < 7 && e; ++i) {
            v[i] = std::atoi(e);
            e = std::strchr(e, ',');
            if (e) ++e;
        }
    });
    return v[which];
}

}  // namespace

namespace {

// Clusters of `sk` CTAs along z (16-token tiles of format `fmt`, `smem` bytes
// each) the device can hold at once: a cluster's CTAs must share one GPC, so
// sizes that do not pack its SMs leave some idle (measured: 20 tiles split 7
// ways, 140 CTAs, ran as two waves).  Cached per (format, size, bytes).
int max_active_clusters(int fmt, int sk, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(fmt, sk, smem, dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const void *k = fmt == kPfQ8_0 ? reinterpret_cast<const void *>(prefill_kernel<1, 1, kPfQ8_0, true>)
                                   : reinterpret_cast<const void *>(prefill_kernel<1, 1, kPfQ4_0, true>);
    int n = 0;
    if (ensure_smem_optin(k, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, static_cast<unsigned>(sk));
        cfg.blockDim = dim3(kThreadsSmall);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = static_cast<unsigned>(sk);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

}  // namespace

PrefillPlan prefill_plan(int64_t N, int64_t K, int64_t M, int sms, int fmt, int splitk)
{
    const int sk_force = ring_override(6);
    auto plan = [&](int sk) {
        return plan_prefill(N, K, M, sms, ring_override(0), ring_override(1), ring_override(2), ring_override(3),
                            ring_override(4), ring_override(5), fmt, sk);
    };
    PrefillPlan pl = plan(sk_force > 0 ? sk_force : splitk);
    // An automatic split keeps every cluster of the grid resident at once.
    if (sk_force <= 0 && splitk < 0)
        while (pl.ok && pl.splitk > 1 && pl.grid_x * pl.grid_y > max_active_clusters(fmt, pl.splitk, pl.smem))
            pl = plan(pl.splitk - 1);
    if (encode_fn() == nullptr) pl.ok = false;
    return pl;
}

cudaError_t launch_prefill(const PrefillPlan &pl, const void *W, const void *x, float *y, int64_t N, int64_t K,
                           int64_t M, int *status, cudaStream_t s, bool pdl, bool test_skip_copy)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc || !pl.ok) return cudaErrorNotSupported;
    const bool q8 = pl.fmt == kPfQ8_0;
    const int64_t row_bytes = (K / 32) * (q8 ? 34 : 18);
    CUtensorMap wmap, xmap;
    {
        // Q8_0: 16-bit elements, so that one 272-byte chunk row fits a box
        // (at most 256 elements per box dimension).
        const int esz = q8 ? 2 : 1;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / esz), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(prefill_row_bytes(pl.fmt) / esz), kBM};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&wmap, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W),
                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
        const cuuint32_t box[2] = {kKB, static_cast<cuuint32_t>(pl.TN / pl.cluster)};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    PrefillParams p = {};
    p.y = y;
    p.status = status;
    p.N = N;
    p.K = K;
    p.M = M;
    p.TN = pl.TN;
    p.WT = pl.WT;
    p.NW = pl.NW;
    p.NSA = pl.NSA;
    p.NSB = pl.NSB;
    p.KSUB = pl.KSUB;
    p.cluster = pl.cluster;
    p.tmem_cols = pl.tmem_cols;
    p.test_skip_copy = test_skip_copy ? 1 : 0;
#ifdef QMV_PHASE_STAMPS
    {
        void *ph = nullptr;
        if (cudaGetSymbolAddress(&ph, g_prefill_phase) == cudaSuccess)
            p.phase = static_cast<unsigned long long *>(ph);
        p.phase_seq = g_prefill_phase_seq.fetch_add(1);
    }
#endif
    // Q8_0 takes no multicast pairs (the plan never sets them for it).
    if (q8 && pl.cluster > 1) return cudaErrorInvalidValue;
    if (pl.splitk > 1 && (pl.cluster > 1 || pl.TN != 16)) return cudaErrorInvalidValue;
    if (pl.TN == 16 && (pl.WT != 1 || pl.cluster != 1)) return cudaErrorInvalidValue;
    auto kernel =
        pl.TN == 16 ? (q8 ? prefill_kernel<1, 1, kPfQ8_0, true> : prefill_kernel<1, 1, kPfQ4_0, true>)
        : q8 ? (pl.WT == 2 ? prefill_kernel<2, 1, kPfQ8_0, false> : prefill_kernel<1, 1, kPfQ8_0, false>)
        : pl.WT == 2 ? (pl.cluster > 1 ? prefill_kernel<2, 2, kPfQ4_0, false> : prefill_kernel<2, 1, kPfQ4_0, false>)
                     : (pl.cluster > 1 ? prefill_kernel<1, 2, kPfQ4_0, false> : prefill_kernel<1, 1, kPfQ4_0, false>);
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void *>(kernel), pl.smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(pl.grid_x), static_cast<unsigned>(pl.grid_y),
                    static_cast<unsigned>(pl.splitk));
    const dim3 cluster(static_cast<unsigned>(pl.cluster), 1, static_cast<unsigned>(pl.splitk));
    return launch_ex_cluster_dims(kernel, grid, dim3(pl.TN == 16 ? kThreadsSmall : kThreads), pl.smem, s, pdl,
                                  cluster, wmap, xmap, p);
}

}  // namespace qmv

#ifdef QMV_PHASE_STAMPS
// Phase-timeline builds only (not declared in include/qmv.h): copies up to
// max_records prefill records to host memory and resets them; returns the
// count or -1 on a CUDA error.
// The slot-level trace of CTA (0, 0) of the last prefill launch: 128 rounds x 8 stamps.
extern "C" QMV_API int qmv_prefill_trace(unsigned long long *host)
{
    using namespace qmv;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    return cudaMemcpyFromSymbol(host, g_prefill_trace_dev, sizeof(unsigned long long) * kTraceSlotsDev * kTraceCols) ==
                   cudaSuccess
               ? 0
               : -1;
}

extern "C" QMV_API int64_t qmv_prefill_phase_stamps(unsigned long long *host, int64_t max_records)
{
    using namespace qmv;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    unsigned long long n = 0;
    if (cudaMemcpyFromSymbol(&n, g_prefill_phase, sizeof(n)) != cudaSuccess) return -1;
    if (n > static_cast<unsigned long long>(kPrefillPhaseCap)) n = kPrefillPhaseCap;
    if (static_cast<int64_t>(n) > max_records) n = static_cast<unsigned long long>(max_records);
    if (n && cudaMemcpyFromSymbol(host, g_prefill_phase, n * kPrefillPhaseWords * sizeof(unsigned long long),
                                  sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(g_prefill_phase, &zero, sizeof(zero)) != cudaSuccess) return -1;
    g_prefill_phase_seq.store(0);
    return static_cast<int64_t>(n);
}
#endif
