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
constexpr int kKChunk = 256;             // K per packed weight tile (8 blocks of 32 weights per row)
// Packed weight formats the kernel takes, and one row's 256-K chunk in bytes:
// eight 18-byte Q4_0 blocks or eight 34-byte Q8_0 blocks.
constexpr int kPfQ4_0 = 0, kPfQ8_0 = 1;
constexpr int prefill_row_bytes(int fmt) { return fmt == kPfQ8_0 ? 272 : 144; }
constexpr int kPackedRowBytes = 144;     // Q4_0
constexpr int kPackedTileBytes = kBM * kPackedRowBytes;    // 18432
constexpr int kAtomCols = kKB / 2;       // tensor-memory columns of one dequantised 64-K atom (2 fp16 per column)
constexpr int kTmemCols = 512;           // every CTA allocates all of tensor memory
// Threads of a CTA: 8 dequantising warps (16 in 16-token tiles), the MMA warp
// and the two copy producers.
constexpr int prefill_threads(bool small) { return ((small ? 16 : 8) + 3) * 32; }
constexpr int kPrefillThreads = prefill_threads(false);
// Alignment slack for the 1024-byte-aligned activation tiles, then the
// barriers (2*NW + 2*NSA + 2*NSB + 1 of 8 bytes), the tensor-memory address
// slot and the abort flag.
constexpr size_t kPrefillFixedSmem = 1024 + 512;
// Split K: each CTA receives the other CTAs' partial rows of its share in a
// buffer after the barriers' 512 bytes, [SK][ceil(128 / SK)][16] fp32 (16-token
// tiles): at most 135 rows of 64 bytes.
constexpr size_t kPrefillSplitSmem = 135 * 64;
constexpr size_t kPrefillSmemCap = 225 * 1024;
constexpr int64_t kMaxGridY = 65535;     // CUDA's limit on gridDim.y

struct PrefillPlan {
    bool ok;           // false: the tensor-core kernel does not take this shape
    int fmt;           // kPfQ4_0 or kPfQ8_0
    int TN;            // token columns per tile = the MMA's N (16, or a multiple of 64 up to 256)
    int WT;            // 128-row weight tiles per CTA (1 or 2): each activation atom feeds WT MMAs
    int KSUB;          // 64-K atoms per ring slot (1, 2 or 4): MMAs per barrier round = 4 * KSUB * WT
    int NW;            // packed-weight ring slots (256-K chunks of WT tiles)
    int NSA;           // weight-atom ring slots in tensor memory
    int NSB;           // activation ring slots in shared memory
    int cluster;       // CTAs per cluster along the weight tiles (1 or 2): each loads 1/cluster of every
                       // activation tile and multicasts it to the others
    uint32_t tmem_cols;   // allocated: WT accumulators [t * TN, (t + 1) * TN), then the weight atoms
    size_t smem;       // dynamic shared memory per CTA
    int64_t grid_x;    // CTAs along the weight rows (WT * 128 rows each)
    int64_t grid_y;    // token tiles
    int splitk;        // CTAs along K (gridDim.z, one cluster): each takes a contiguous share of the
                       // 256-K chunks, and the cluster adds the partial tiles through distributed
                       // shared memory in rank order
};

// Atoms per ring slot: a barrier round carries at least 8 MMAs when it can.
inline int prefill_ksub(int TN, int WT)
{
    const int k = TN <= 64 ? 4 : (TN <= 128 ? 2 : 1);
    return k / WT > 0 ? k / WT : 1;
}

// Accumulators (WT * TN columns, rounded up to 32), then NSA slots of weight atoms.
inline int64_t prefill_tmem_cols(int TN, int WT, int KSUB, int NSA)
{
    return (static_cast<int64_t>(WT) * TN + 31) / 32 * 32 + static_cast<int64_t>(NSA) * KSUB * WT * kAtomCols;
}

// Estimated SM cycles of a call with token tiles of TN and WT weight tiles per
// CTA, fitted to slot-level timelines on the GB300: a CTA sustains about 4000
// flop per cycle in its main loop whatever the tile (7.7-7.9 TFLOP/s per SM
// for 128 x 256 and 2 x 128 x 192 tiles), and no 64-K slice takes less than
// ~130 cycles per MMA to issue (64-token tiles); plus ~6000 cycles of ramp and
// epilogue per wave of CTAs.  Two weight tiles per CTA are only tried with
// 192-token tiles, where they were measured to pay (a 2 x 128 x 128 tile ran
// at 4.9 TFLOP/s per SM).
inline int64_t prefill_cost(int64_t N, int64_t K, int64_t M, int sms, int TN, int WT)
{
    const int64_t grid = (N + 128 * WT - 1) / (128 * WT) * ((M + TN - 1) / TN);
    const int64_t waves = (grid + sms - 1) / (sms > 0 ? sms : 1);
    const int64_t flops = 2LL * 128 * WT * TN * kKB;
    const int64_t tensor = flops / 4000;
    const int64_t issue = 4LL * WT * 130;
    return waves * ((K / kKB) * (tensor > issue ? tensor : issue) + 6000);
}

// nw_force / ns_force: ring depths forced for tests and sweeps (a packed-weight
// depth below 1 or an activation-ring depth below 2 keeps the rule; shared
// memory and tensor memory still cap them).  One packed-weight slot is correct
// (each dequantising thread copies its rows into registers before releasing
// the slot) but slow.  cluster_force: 1 or 2 forces the cluster size;
// tn_force (64..256, a multiple of 64) and wt_force (1 or 2) force the tile,
// ksub_force (1, 2 or 4) the atoms per ring slot where tensor memory still
// holds two weight-atom slots (0 keeps the rule).
//
// fmt: the packed weight format.  splitk: 0 = one CTA per tile along K;
// -1 = as many CTAs along K (at most 8, at most one per 256-K chunk) as keep
// the grid within one wave of `sms`; n > 0 forces n (tests and sweeps; kept
// within the same limits).  Split K is taken with 16-token tiles only.
inline PrefillPlan plan_prefill(int64_t N, int64_t K, int64_t M, int sms, int nw_force, int ns_force,
                                int cluster_force = 0, int tn_force = 0, int wt_force = 0, int ksub_force = 0,
                                int fmt = kPfQ4_0, int splitk = 0)
{
    PrefillPlan pl = {};
    pl.fmt = fmt;
    pl.splitk = 1;
    if (!(K % kKChunk == 0 && K > 0 && N > 0 && M > 0 && N < (int64_t(1) << 31) && M < (int64_t(1) << 31) &&
          K < (int64_t(1) << 30) && (fmt == kPfQ4_0 || fmt == kPfQ8_0)))
        return pl;
    // Tile choice: the (token tile, weight tiles per CTA) of least estimated
    // time among those tensor memory holds with two weight-atom slots; ties
    // go to the larger grid.  Token tiles wider than the call are not tried.
    const int64_t m_cover = (M + 63) / 64 * 64;
    int TN = 0, WT = 0;
    int64_t best = 0, best_grid = 0;
    // Up to 16 tokens: 16-token tiles (the MMA's smallest N at M = 128), one
    // weight tile per CTA.
    const bool small = M <= 16 && (tn_force == 0 || tn_force == 16) && (wt_force == 0 || wt_force == 1);
    if (small) {
        TN = 16;
        WT = 1;
    }
    for (int tn = 64; !small && tn <= 256; tn += 64) {
        if (tn > m_cover && tn > 64) break;
        if (tn_force && tn != tn_force) continue;
        for (int wt = 1; wt <= 2; ++wt) {
            if (wt_force && wt != wt_force) continue;
            if (!wt_force && wt == 2 && tn != 192) continue;
            if (prefill_tmem_cols(tn, wt, prefill_ksub(tn, wt), 2) > kTmemCols) continue;
            const int64_t c = prefill_cost(N, K, M, sms, tn, wt);
            const int64_t g = (N + 128 * wt - 1) / (128 * wt) * ((M + tn - 1) / tn);
            if (TN == 0 || c < best || (c == best && g > best_grid)) {
                TN = tn;
                WT = wt;
                best = c;
                best_grid = g;
            }
        }
    }
    if (TN == 0) return pl;
    const size_t b_atom = static_cast<size_t>(TN) * kKB * 2;
    const size_t w_tile = static_cast<size_t>(WT) * kBM * prefill_row_bytes(fmt);
    int KSUB = prefill_ksub(TN, WT);
    if ((ksub_force == 1 || ksub_force == 2 || ksub_force == 4) &&
        prefill_tmem_cols(TN, WT, ksub_force, 2) <= kTmemCols &&
        kPrefillFixedSmem + static_cast<size_t>(nw_force >= 1 && nw_force < 2 ? nw_force : 2) * w_tile +
                2 * static_cast<size_t>(ksub_force) * b_atom <= kPrefillSmemCap)
        KSUB = ksub_force;
    // Activation tiles take 1.5-2 us to land (measured), so their ring is as
    // deep as shared memory allows; the weight atoms only wait for the
    // dequantising warps, and take what tensor memory leaves.
    int NW = 3, NSB = 5, NSA = 6;
    auto total = [&] {
        return kPrefillFixedSmem + static_cast<size_t>(NW) * w_tile + static_cast<size_t>(NSB) * KSUB * b_atom;
    };
    if (nw_force >= 1) NW = nw_force;
    if (ns_force >= 2) NSB = ns_force;
    while (prefill_tmem_cols(TN, WT, KSUB, NSA) > kTmemCols && NSA > 2) --NSA;
    while (total() > kPrefillSmemCap && NSB > 2) --NSB;
    while (total() > kPrefillSmemCap && NW > 2) --NW;
    // One ring for both operands when both can be at least three deep: the
    // MMA thread then releases a slot with one commit instead of two (one
    // 64-token slot of 16 MMAs: 1088 against 1440 ns; 128 x 256 tiles: 21.3
    // against 25.5 us per call on 8192x2048 at 512 tokens).
    if (NSA >= 3 && NSB >= 3 && ns_force < 2) NSA = NSB = (NSA < NSB ? NSA : NSB);
    pl.TN = TN;
    pl.WT = WT;
    pl.KSUB = KSUB;
    pl.NW = NW;
    pl.NSA = NSA;
    pl.NSB = NSB;
    pl.tmem_cols = kTmemCols;
    pl.smem = total();
    pl.grid_x = (N + 128 * WT - 1) / (128 * WT);
    // Pairs of CTAs on neighbouring weight tiles can share every activation
    // tile (cluster = 2): each brings in half of its token rows and multicasts
    // them to both.  It halves the L2 reads and each SM's tensor-copy requests
    // but measured slower (prefill workload 564 -> 509 TFLOP/s on the same
    // GB300; the 512-token slice period 544 -> 608 ns), so the rule keeps one
    // CTA per cluster; QMV_PREFILL_RING=",,2" forces pairs.  An odd tile count
    // then gets one extra CTA whose rows lie past N (it loads zeros for its
    // weights and stores nothing).
    pl.cluster = 1;
    if ((cluster_force == 1 || cluster_force == 2) && fmt == kPfQ4_0) pl.cluster = cluster_force;
    pl.grid_x = (pl.grid_x + pl.cluster - 1) / pl.cluster * pl.cluster;
    pl.grid_y = (M + TN - 1) / TN;
    // Split K: CTA z of the cluster adds rows [128 z / SK, 128 (z + 1) / SK) of
    // every CTA's partial tile, which the others store into its shared memory.
    const int64_t chunks = K / kKChunk;
    if (splitk != 0 && TN == 16 && pl.cluster == 1) {
        int64_t sk = splitk > 0 ? splitk : 8;
        if (splitk < 0)
            while (sk > 1 && pl.grid_x * pl.grid_y * sk > sms) --sk;
        if (sk > 8) sk = 8;
        if (sk > chunks) sk = chunks;
        if (sk < 1) sk = 1;
        pl.splitk = static_cast<int>(sk);
    }
    if (pl.splitk > 1) pl.smem += kPrefillSplitSmem;
    // More token tiles than gridDim.y allows (M above 65535 * 256) take the
    // generic kernel rather than a launch the runtime would refuse.
    pl.ok = pl.grid_y <= kMaxGridY && pl.smem <= kPrefillSmemCap &&
            prefill_tmem_cols(TN, WT, KSUB, NSA) <= kTmemCols;
    return pl;
}

}  // namespace qmv
