// qmv_prefill_plan.h -- launch plan of the tensor-core prefill kernel for one
// call: token tile width, accumulators, ring depths, shared memory and grid.
// Host-only arithmetic with no CUDA calls, so that the bounds checker can
// replay every plan on a machine without a GPU.
#pragma once

#include <cstddef>
#include <cstdint>

namespace qmv {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kKB = 64;                  // K per atom: one 128-byte swizzle row of fp16 activations
constexpr int kKChunk = 256;             // K per packed weight tile (8 Q4_0 blocks = 144 bytes per row)
constexpr int kPackedRowBytes = 144;
constexpr int kPackedTileBytes = kBM * kPackedRowBytes;    // 18432
constexpr int kAtomCols = kKB / 2;       // tensor-memory columns of one dequantised 64-K atom (2 fp16 per column)
constexpr int kTmemCols = 512;           // every CTA allocates all of tensor memory
constexpr int kPrefillThreads = 352;     // 11 warps: 8 dequantising, MMA issue, 2 copy producers
// Alignment slack for the 1024-byte-aligned activation tiles, then the
// barriers (2*NW + 4*NS + 1 of 8 bytes), the tensor-memory address slot and
// the abort flag.
constexpr size_t kPrefillFixedSmem = 1024 + 512;
constexpr size_t kPrefillSmemCap = 225 * 1024;
constexpr int64_t kMaxGridY = 65535;     // CUDA's limit on gridDim.y

struct PrefillPlan {
    bool ok;           // false: the tensor-core kernel does not take this shape
    int TN;            // token columns per tile = the MMA's N (multiple of 64, <= 256)
    int KSUB;          // 64-K atoms per ring slot (1, 2 or 4): MMAs per barrier round = 4 * KSUB
    int NW;            // packed-weight ring slots (256-K tiles)
    int NS;            // operand ring slots (activation atoms in shared memory, weight atoms in tensor memory)
    int cluster;       // CTAs per cluster along the weight tiles (1 or 2): each loads 1/cluster of every
                       // activation tile and multicasts it to the others
    uint32_t tmem_cols;   // allocated: the accumulator [0, TN), then NS * KSUB atoms of A
    size_t smem;       // dynamic shared memory per CTA
    int64_t grid_x;    // 128-row weight tiles
    int64_t grid_y;    // token tiles
};

inline int prefill_pick_tn(int64_t M)
{
    // Multiples of 64 so that the epilogue warps read whole 32-column chunks.
    if (M >= 256) return 256;
    int tn = static_cast<int>((M + 63) / 64) * 64;
    return tn < 64 ? 64 : tn;
}

// nw_force / ns_force: ring depths forced for tests and sweeps (a packed-weight
// depth below 1 or an operand depth below 2 keeps the rule; shared memory and
// tensor memory still cap them).  One packed-weight slot is correct (each
// dequantising thread copies its 144-byte row into registers before releasing
// the slot) but slow: the four atoms held in registers do not cover the next
// tile's DRAM latency.
// cluster_force: 1 or 2 forces the cluster size (0 keeps the rule).
inline PrefillPlan plan_prefill(int64_t N, int64_t K, int64_t M, int sms, int nw_force, int ns_force,
                                int cluster_force = 0)
{
    (void)sms;
    PrefillPlan pl = {};
    if (!(K % kKChunk == 0 && K > 0 && N > 0 && M > 0 && N < (int64_t(1) << 31) && M < (int64_t(1) << 31) &&
          K < (int64_t(1) << 30)))
        return pl;
    const int TN = prefill_pick_tn(M);
    // Narrow token tiles take several 64-K atoms per barrier round, so the
    // MMA-issuing thread's fixed cost per round (two barrier waits and a
    // commit) is paid once per 8 or 16 MMAs.
    const int KSUB = TN <= 64 ? 4 : (TN <= 128 ? 2 : 1);
    const size_t b_atom = static_cast<size_t>(TN) * kKB * 2;
    // Activation tiles take 1.5-2 us to land (measured), so the operand ring
    // is as deep as tensor memory (TN + NS * KSUB * 32 columns) and shared
    // memory allow; three packed-weight slots cover DRAM latency at these rates.
    int NW = 3, NS = TN <= 64 ? 3 : 5;
    auto total = [&] {
        return kPrefillFixedSmem + static_cast<size_t>(NW) * kPackedTileBytes +
               static_cast<size_t>(NS) * KSUB * b_atom;
    };
    auto tmem = [&] { return static_cast<int64_t>(TN) + static_cast<int64_t>(NS) * KSUB * kAtomCols; };
    if (nw_force >= 1) NW = nw_force;
    if (ns_force >= 2) NS = ns_force;
    while ((total() > kPrefillSmemCap || tmem() > kTmemCols) && NS > 2) --NS;
    while (total() > kPrefillSmemCap && NW > 2) --NW;
    pl.TN = TN;
    pl.KSUB = KSUB;
    pl.NW = NW;
    pl.NS = NS;
    pl.tmem_cols = kTmemCols;
    pl.smem = total();
    pl.grid_x = (N + kBM - 1) / kBM;
    // Pairs of CTAs on neighbouring weight tiles can share every activation
    // tile (cluster = 2): each brings in half of its token rows and multicasts
    // them to both.  It halves the L2 reads and each SM's tensor-copy requests
    // but measured slower (prefill workload 564 -> 509 TFLOP/s on the same
    // GB300; the 512-token slice period 544 -> 608 ns), so the rule keeps one
    // CTA per cluster; QMV_PREFILL_RING=",,2" forces pairs.  An odd tile count
    // then gets one extra CTA whose rows lie past N (it loads zeros for its
    // weights and stores nothing).
    pl.cluster = 1;
    if (cluster_force == 1 || cluster_force == 2) pl.cluster = cluster_force;
    pl.grid_x = (pl.grid_x + pl.cluster - 1) / pl.cluster * pl.cluster;
    pl.grid_y = (M + TN - 1) / TN;
    // More token tiles than gridDim.y allows (M above 65535 * 256) take the
    // generic kernel rather than a launch the runtime would refuse.
    pl.ok = pl.grid_y <= kMaxGridY && pl.smem <= kPrefillSmemCap && tmem() <= kTmemCols;
    return pl;
}

}  // namespace qmv
