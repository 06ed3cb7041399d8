// qmv_prefill_plan.h -- launch plan of the tensor-core prefill kernel for one
// call: token tile width, accumulators, ring depths, shared memory and grid.
// Host-only arithmetic with no CUDA calls, so that the bounds checker can
// replay every plan on a machine without a GPU.
#pragma once

#include <cstddef>
#include <cstdint>

namespace qmv {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kKB = 64;                  // K per MMA slice (one 128-byte swizzle atom of fp16)
constexpr int kKChunk = 256;             // K per packed weight tile (8 Q4_0 blocks = 144 bytes per row)
constexpr int kPackedRowBytes = 144;
constexpr int kPackedTileBytes = kBM * kPackedRowBytes;    // 18432
constexpr int kATileBytes = kBM * kKB * 2;                 // 16384
constexpr int kPrefillThreads = 352;     // 11 warps: 8 dequantising, MMA issue, 2 copy producers
// Alignment slack for the 1024-byte-aligned operand tiles, then the barriers
// (2*NW + 3*NS + 1 of 8 bytes), the TMEM address slot and the abort flag.
constexpr size_t kPrefillFixedSmem = 1024 + 512;
constexpr size_t kPrefillSmemCap = 225 * 1024;
constexpr int64_t kMaxGridY = 65535;     // CUDA's limit on gridDim.y

struct PrefillPlan {
    bool ok;           // false: the tensor-core kernel does not take this shape
    int TN;            // token columns per tile (multiple of 64, <= 512)
    int NH;            // accumulators per tile: TN / NH <= 256 columns each (the MMA's N)
    int KSUB;          // 64-K atoms per operand slot (1 or 2): MMAs per barrier round = 4 * KSUB
    int NW;            // packed-weight ring slots (256-K tiles)
    int NS;            // operand ring slots
    uint32_t tmem_cols;
    size_t smem;       // dynamic shared memory per CTA
    int64_t grid_x;    // 128-row weight tiles
    int64_t grid_y;    // token tiles
};

inline int prefill_pick_tn(int64_t M)
{
    // Multiples of 64 so that each of the two epilogue warps per lane quarter
    // reads whole 32-column chunks.
    if (M >= 256) return 256;
    int tn = static_cast<int>((M + 63) / 64) * 64;
    return tn < 64 ? 64 : tn;
}

// nw_force / ns_force: ring depths forced for tests and sweeps (a packed-weight
// depth below 1 or an operand depth below 2 keeps the rule; shared memory still
// caps them).  One packed-weight slot is correct (each dequantising thread
// copies its 144-byte row into registers before releasing the slot) but slow
// for narrow token tiles: the four 64-K atoms held in registers do not cover
// the next tile's DRAM latency.
inline PrefillPlan plan_prefill(int64_t N, int64_t K, int64_t M, int sms, int nw_force, int ns_force)
{
    PrefillPlan pl = {};
    if (!(K % kKChunk == 0 && K > 0 && N > 0 && M > 0 && N < (int64_t(1) << 31) && M < (int64_t(1) << 31) &&
          K < (int64_t(1) << 30)))
        return pl;
    int TN = prefill_pick_tn(M);
    int NH = 1;
    // When 256-token tiles would need a second wave of CTAs, one CTA takes
    // 512 tokens in two accumulators (512 TMEM columns): one wave, and each
    // weight tile is dequantised once for all of them.
    const int64_t row_tiles = (N + kBM - 1) / kBM;
    if (TN == 256 && row_tiles * ((M + 255) / 256) > sms && row_tiles * ((M + 511) / 512) <= sms) {
        TN = 512;
        NH = 2;
    }
    // Up to 128 token columns a slot holds two 64-K atoms: eight MMAs per
    // barrier round and per commit (the issuing thread's fixed cost per round
    // is then paid half as often); a 256-column slot would not fit twice.
    const int KSUB = TN <= 128 ? 2 : 1;
    const int b_tile = KSUB * TN * kKB * 2;
    const int a_tile = KSUB * kATileBytes;
    // Ring depths: the packed-weight ring must cover DRAM latency, the
    // activation ring L2 latency, at the MMA rate of this tile width.
    int NW = 4, NS = 3;
    if (TN > 256) {
        NW = 3;
        NS = 2;
    } else if (TN <= 64) {
        NW = 4;
        NS = 3;
    } else if (TN <= 128) {
        NW = 4;
        NS = 2;
    }
    auto total = [&] {
        return kPrefillFixedSmem + static_cast<size_t>(NW) * kPackedTileBytes +
               static_cast<size_t>(NS) * static_cast<size_t>(a_tile + b_tile);
    };
    if (nw_force >= 1) NW = nw_force;
    if (ns_force >= 2) NS = ns_force;
    while (total() > kPrefillSmemCap && NS > 2) --NS;
    while (total() > kPrefillSmemCap && NW > 2) --NW;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(TN)) cols <<= 1;
    pl.TN = TN;
    pl.NH = NH;
    pl.KSUB = KSUB;
    pl.NW = NW;
    pl.NS = NS;
    pl.tmem_cols = cols;
    pl.smem = total();
    pl.grid_x = row_tiles;
    pl.grid_y = (M + TN - 1) / TN;
    // More token tiles than gridDim.y allows (M above 65535 * 256) take the
    // generic kernel rather than a launch the runtime would refuse.
    pl.ok = pl.grid_y <= kMaxGridY && pl.smem <= kPrefillSmemCap;
    return pl;
}

}  // namespace qmv
