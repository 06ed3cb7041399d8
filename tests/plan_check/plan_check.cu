// plan_check.cu -- host-only check of the decode kernels' index arithmetic for
// every launch plan the library's planner produces over a grid of table
// shapes, token counts, formats and call forms.  No GPU is needed and no kernel
// runs: for each plan the program replays, per CTA, warp, stage and lane, the
// kernel's row ranges, bulk-copy sizes and shared-memory destinations, the
// units each lane consumes, the activation offsets it reads and the staging
// writes, and checks every one against the buffer it addresses.  It also
// checks that a call whose activations do not fit in shared memory can be
// split into token subsets that do.  The tensor-core prefill kernel's plans
// are replayed the same way (tensor-copy coordinates, shared-memory layout,
// tensor-memory columns, epilogue coverage).
//
// Built and run by tests/test_plan_bounds.py: the planner's translation unit
// is compiled into this program, with stubs for the launch functions.
#include "../../weight_quantized_decode_gb300/csrc/qmv_api.cu"

#include <algorithm>
#include <cstdio>

using namespace qmv;

namespace {

long g_bad = 0;
long g_checked = 0;

#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            if (g_bad < 20) {                              \
                std::printf("FAIL %s: ", #cond);           \
                std::printf(__VA_ARGS__);                  \
                std::printf("\n");                         \
            }                                              \
            ++g_bad;                                       \
        }                                                  \
    } while (0)

constexpr int kSms = 152;          // GB300
constexpr int kOptin = 232448;     // shared memory a CTA may opt into (227 KB)

int unit_bytes_of(int fmt) { return fmt == kQ4_0 ? 144 : (fmt == kQ2W ? 80 : 272); }
int block_bytes_of(int fmt) { return fmt == kQ4_0 ? 18 : (fmt == kQ2W ? 10 : 34); }

GemvParams params(int fmt, int64_t N, int64_t K, int n_problems, bool xq8, bool swiglu)
{
    GemvParams p = {};
    p.N = N;
    p.K = K;
    p.n_experts = 2 * n_problems;
    p.row_bytes = (K / 32) * block_bytes_of(fmt);
    p.n_problems = n_problems;
    p.max_local_problems = n_problems;
    p.rows_total = swiglu ? 2 * N : N * n_problems;
    p.x = reinterpret_cast<const __half *>(0x1000);     // 16-byte aligned, never dereferenced
    p.W2 = swiglu ? reinterpret_cast<const uint8_t *>(0x2000) : nullptr;
    p.xq8 = xq8 ? 1 : 0;
    return p;
}

// The plain, multi-expert and Q8_1 forms: copies, consumption, activations.
void check_plan(int fmt, int64_t N, int64_t K, int M, int n_problems, bool xq8)
{
    GemvParams p = params(fmt, N, K, n_problems, xq8, false);
    const Plan pl = plan_gemv(fmt, p, M, kSms, kOptin);
    if (!pl.streaming) {
        // A plain call that does not fit must split into token subsets that do.
        if (M > 1 && n_problems == 1 && K % 256 == 0) {
            bool split = false;
            for (int parts = 2; parts <= M && !split; ++parts) {
                const int mc = (M + parts - 1) / parts;
                GemvParams probe = params(fmt, N, K, 1, xq8, false);
                if (!plan_gemv(fmt, probe, mc, kSms, kOptin).streaming) continue;
                split = true;
                for (int mm = 1; mm <= mc; ++mm) {
                    GemvParams part = params(fmt, N, K, 1, xq8, false);
                    CHECK(plan_gemv(fmt, part, mm, kSms, kOptin).streaming, "part of %d tokens of %lldx%lld", mm,
                          (long long)N, (long long)K);
                }
            }
            CHECK(split || K > 65536, "no token split for fmt %d %lldx%lld M=%d", fmt, (long long)N, (long long)K, M);
        }
        return;
    }
    ++g_checked;
    const int XUB = xq8 ? kXQ8UnitBytes : kXUnitBytes;
    const int unit = unit_bytes_of(fmt);
    CHECK(pl.smem <= static_cast<size_t>(kOptin), "smem %zu", pl.smem);
    CHECK(pl.warps >= 1 && pl.warps <= (M <= 2 ? 16 : 12), "warps %d", pl.warps);
    const int U = p.U, G = p.G, SP = p.SP, RG = 32 / G, warps = pl.warps;
    CHECK(G >= 1 && G <= 32 && p.S >= 2, "G %d S %d", G, p.S);
    const size_t xbytes = static_cast<size_t>(p.max_local_problems) * M * U * XUB;
    const int slot_bytes = 32 * SP * unit;
    const int ups = SP * G;                              // units per stage and row
    const uint32_t lane_chunk = static_cast<uint32_t>(ups * unit);
    const int T_stages = (U + ups - 1) / ups;
    const uint32_t R = static_cast<uint32_t>(p.rows_total);
    for (int b = 0; b < pl.grid; ++b) {
        const uint32_t row0 = static_cast<uint32_t>(static_cast<uint64_t>(R) * b / pl.grid);
        const uint32_t row1 = static_cast<uint32_t>(static_cast<uint64_t>(R) * (b + 1) / pl.grid);
        const int nrows = static_cast<int>(row1 - row0);
        const int prob_lo = (n_problems > 1 && nrows > 0) ? static_cast<int>(row0 / N) : 0;
        const int prob_hi = n_problems > 1 ? (nrows > 0 ? static_cast<int>((row1 - 1) / N) : -1) : 0;
        CHECK(prob_hi - prob_lo + 1 <= p.max_local_problems, "problems %d > %d", prob_hi - prob_lo + 1,
              p.max_local_problems);
        // staging writes of this CTA (token tok, 16-byte chunk c of a 32-block)
        const int ntok = (prob_hi - prob_lo + 1) * M;
        for (int tok = 0; tok < ntok; tok += std::max(1, ntok - 1)) {
            for (int64_t blk = 0; blk < K / 32; blk += std::max<int64_t>(1, K / 32 - 1)) {
                const size_t base = static_cast<size_t>(tok) * U * XUB + static_cast<size_t>(blk >> 3) * XUB;
                if (xq8) {
                    CHECK(base + (blk & 7) * 32 + 3 * 8 + 8 <= xbytes, "q8_1 codes");
                    CHECK(base + 256 + (blk & 7) * 8 + 8 <= xbytes && 256 + 8 * 8 <= XUB, "q8_1 block data");
                } else {
                    CHECK(base + (blk & 7) * 64 + 3 * 16 + 16 <= xbytes, "fp16 chunk");
                }
            }
        }
        const int ngroups = (nrows + RG - 1) / RG;
        for (int w = 0; w < warps; ++w) {
            // row groups are dealt to the CTA's warps round-robin; each takes T_stages stages
            for (int grp = w; grp < ngroups; grp += warps) {
                for (int t = 0; t < T_stages; ++t) {
                    const int u0 = t * ups, u1 = std::min(U, u0 + ups);
                    for (int lane = 0; lane < 32; ++lane) {      // copy issue: lane = row of the group
                        const int lr = grp * RG + lane;
                        if (lane >= RG || lr >= nrows || u1 <= u0) continue;
                        const uint32_t bytes = static_cast<uint32_t>(u1 - u0) * unit;
                        CHECK(bytes % 16 == 0 && bytes <= lane_chunk, "copy bytes %u", bytes);
                        CHECK(lane * lane_chunk + bytes <= static_cast<uint32_t>(slot_bytes), "copy destination");
                        CHECK(u1 <= U, "source units %d..%d of %d", u0, u1, U);
                    }
                    for (int lane = 0; lane < 32; ++lane) {      // consumption: lane (r, q)
                        const int r = lane / G, q = lane - r * G;
                        if (r >= RG) continue;                  // idle lanes when G does not divide 32
                        const int lr = grp * RG + r;
                        if (lr >= nrows) continue;
                        CHECK(r * G + G - 1 < 32, "reduction lanes");
                        for (int pass = 0; pass < SP; ++pass) {
                            const int u = u0 + q + pass * G;
                            if (u >= U) continue;
                            const int off = pass * G + q;       // unit within the lane's chunk
                            CHECK(u < u1, "unit %d read but not copied (%d..%d)", u, u0, u1);
                            CHECK(static_cast<size_t>(r) * lane_chunk + static_cast<size_t>(off + 1) * unit <=
                                      static_cast<size_t>(slot_bytes),
                                  "shared read");
                            const uint32_t row = row0 + lr;
                            const int prob = n_problems > 1 ? static_cast<int>(row / N) : 0;
                            const size_t xo = static_cast<size_t>(prob - prob_lo) * M * U * XUB +
                                              static_cast<size_t>(M - 1) * U * XUB + static_cast<size_t>(u + 1) * XUB;
                            CHECK(xo <= xbytes, "activations %zu > %zu", xo, xbytes);
                        }
                    }
                }
            }
        }
    }
}

// The fused SwiGLU: CTAs own whole gate/up pairs, a row group holds whole pairs
// and the up partner sits G lanes above its gate lane.
void check_swiglu(int64_t N, int64_t K, int M)
{
    GemvParams p = params(kQ4_0, N, K, 1, false, true);
    const Plan pl = plan_gemv(kQ4_0, p, M, kSms, kOptin);
    if (!pl.streaming) return;
    ++g_checked;
    const int G = p.G, RG = 32 / G;
    CHECK((G & (G - 1)) == 0 && G <= 16 && RG % 2 == 0, "G %d", G);
    CHECK(pl.smem <= static_cast<size_t>(kOptin), "smem");
    const uint32_t R = static_cast<uint32_t>(p.rows_total);
    for (int b = 0; b < pl.grid; ++b) {
        const uint32_t row0 = 2u * static_cast<uint32_t>((static_cast<uint64_t>(R / 2) * b) / pl.grid);
        const uint32_t row1 = 2u * static_cast<uint32_t>((static_cast<uint64_t>(R / 2) * (b + 1)) / pl.grid);
        const int nrows = static_cast<int>(row1 - row0);
        CHECK(row0 % 2 == 0 && nrows % 2 == 0 && row1 <= R, "pairs");
        const int ngroups = (nrows + RG - 1) / RG;
        for (int gi = 0; gi < ngroups; ++gi) {
            for (int lane = 0; lane < 32; ++lane) {
                const int r = lane / G, q = lane - r * G;
                if (r >= RG) continue;
                const int lr = gi * RG + r;
                if (lr >= nrows) continue;
                const uint32_t row = row0 + lr;
                CHECK((row >> 1) < static_cast<uint32_t>(N), "table row");
                if ((lr & 1) == 0 && q == 0) CHECK(lane + G < 32 && r + 1 < RG && lr + 1 < nrows, "partner lane");
            }
        }
    }
}

// The tensor-core prefill kernel: tile and ring choices, the shared-memory
// layout and its alignment, tensor-copy boxes and coordinates, tensor-memory
// columns (WT accumulators and the dequantised weight atoms), the
// dequantising threads' reads of the packed slot and writes of tensor memory
// (each lane and column of every weight atom written exactly once, by a warp
// whose lane quarter holds it), the MMAs' operand addresses, and the
// epilogue's coverage of every (lane quarter, column chunk) of the
// accumulators.
void check_prefill(int64_t N, int64_t K, int64_t M, int sms, int nw_force, int ns_force, int cl_force,
                   int tn_force, int wt_force, int ksub_force = 0, int fmt = kPfQ4_0, int splitk = 0)
{
    const PrefillPlan pl =
        plan_prefill(N, K, M, sms, nw_force, ns_force, cl_force, tn_force, wt_force, ksub_force, fmt, splitk);
    const bool shape_ok = K % kKChunk == 0 && K > 0 && N > 0 && M > 0 && N < (int64_t(1) << 31) &&
                          M < (int64_t(1) << 31) && K < (int64_t(1) << 30);
    if (!pl.ok) {
        // a shape of the kernel's form is refused only where the grid would exceed gridDim.y, or where a
        // forced tile is not available
        CHECK(!shape_ok || pl.grid_y > kMaxGridY || tn_force || wt_force, "prefill refused %lldx%lld M=%lld",
              (long long)N, (long long)K, (long long)M);
        return;
    }
    ++g_checked;
    CHECK(shape_ok, "prefill took %lldx%lld M=%lld", (long long)N, (long long)K, (long long)M);
    const int TN = pl.TN, WT = pl.WT, KSUB = pl.KSUB, NW = pl.NW, NSA = pl.NSA, NSB = pl.NSB;
    // kind::f16, M = 128: N a multiple of 16 up to 256; 16-token tiles for calls of up to 16 tokens
    CHECK((TN % 64 == 0 && TN >= 64 && TN <= 256) || (TN == 16 && M <= 16 && WT == 1), "TN %d", TN);
    CHECK(pl.fmt == fmt, "format");
    const int SK = pl.splitk;
    const int64_t chunks_all = K / kKChunk;
    CHECK(SK >= 1 && SK <= 8 && SK <= chunks_all, "split K %d", SK);
    CHECK(SK == 1 || (TN == 16 && pl.cluster == 1), "split K needs 16-token tiles without multicast");
    CHECK(splitk != 0 || SK == 1, "split K unasked");
    if (splitk < 0 && SK > 1) CHECK(pl.grid_x * pl.grid_y * SK <= sms, "split K beyond one wave");
    CHECK(WT == 1 || WT == 2, "WT %d", WT);
    CHECK(KSUB == 1 || KSUB == 2 || KSUB == 4, "KSUB %d", KSUB);              // a slot never straddles a W chunk
    CHECK(NW >= 1 && NSA >= 2 && NSB >= 2, "rings %d %d %d", NW, NSA, NSB);
    CHECK(pl.smem <= static_cast<size_t>(kOptin), "prefill smem %zu", pl.smem);
    const uint32_t cols = pl.tmem_cols;
    CHECK(cols == 512, "TMEM %u", cols);
    const int64_t a0 = (static_cast<int64_t>(WT) * TN + 31) / 32 * 32;   // first weight-atom column
    const int64_t a_end = a0 + static_cast<int64_t>(NSA) * KSUB * WT * kAtomCols;
    CHECK(a_end <= cols, "TMEM columns %lld > %u", (long long)a_end, cols);
    const int CL = pl.cluster;
    CHECK(CL == 1 || CL == 2, "cluster %d", CL);
    CHECK(pl.grid_x >= 1 && pl.grid_x <= INT32_MAX && pl.grid_y >= 1 && pl.grid_y <= kMaxGridY, "grid");
    CHECK(pl.grid_x % CL == 0, "grid x %lld not a multiple of the cluster", (long long)pl.grid_x);
    const int64_t rows_per_cta = static_cast<int64_t>(kBM) * WT;
    CHECK(pl.grid_x * rows_per_cta >= N && (pl.grid_x - CL) * rows_per_cta < N, "row tiles");
    CHECK(pl.grid_y * TN >= M && (pl.grid_y - 1) * TN < M, "token tiles");
    // each CTA along K: chunks [c_first, c_first + nC), nK slots
    int64_t covered = 0;
    for (int z = 0; z < SK; ++z) {
        const int64_t c_first = chunks_all * z / SK, nCz = chunks_all * (z + 1) / SK - c_first;
        CHECK(c_first == covered && nCz >= 1 && (nCz * 4) % KSUB == 0, "split K chunks %d", z);
        covered += nCz;
    }
    CHECK(covered == chunks_all, "split K cover");
    const int64_t nK = K / (kKB * KSUB), nC = K / kKChunk;
    CHECK(nK * KSUB * kKB == K && nC * 4 == nK * KSUB && nK < INT32_MAX, "K loop");
    const int row_b = prefill_row_bytes(fmt), esz = fmt == kPfQ8_0 ? 2 : 1;
    CHECK(row_b % 16 == 0 && row_b / esz <= 256, "W box row");

    // shared memory, as offsets from the 1024-byte-aligned base
    const size_t b_atom = static_cast<size_t>(TN) * kKB * 2;
    const size_t b_slot = KSUB * b_atom;
    const size_t w_slot = static_cast<size_t>(WT) * kBM * row_b;
    const size_t w_off = NSB * b_slot;
    const size_t bar_off = w_off + static_cast<size_t>(NW) * w_slot;
    const size_t bar_end = bar_off + static_cast<size_t>(2 * NW + 2 * NSA + 2 * NSB + 1) * 8 + 4 + 4;
    CHECK(1023 + bar_end <= pl.smem, "layout %zu + slack > %zu", bar_end, pl.smem);
    CHECK(bar_end <= bar_off + 512, "barriers within their 512 bytes");
    if (pl.splitk > 1) {
        // the split-K receive buffer after the barriers: [SK][ceil(128/SK)][16] fp32, 16-byte rows
        const size_t red_end = bar_off + 512 + static_cast<size_t>(pl.splitk) * ((kBM + pl.splitk - 1) / pl.splitk) * 64;
        CHECK(1023 + red_end <= pl.smem && (bar_off + 512) % 16 == 0, "split-K buffer %zu > %zu", red_end, pl.smem);
    }
    CHECK((bar_off + 1024) >> 4 < (size_t(1) << 14), "descriptor address field");
    for (int s = 0; s < NSB; ++s)
        for (int a = 0; a < KSUB; ++a)
            for (int r = 0; r < CL; ++r) {
                // each cluster CTA's share of the token rows lands at its own 1024-byte-aligned offset
                const size_t off = s * b_slot + a * b_atom + static_cast<size_t>(r) * (TN / CL) * 128;
                CHECK(off % 1024 == 0 && off + static_cast<size_t>(TN / CL) * 128 <= s * b_slot + (a + 1) * b_atom,
                      "B tile share alignment");
            }
    for (int w = 0; w < NW; ++w)
        for (int t = 0; t < WT; ++t)
            CHECK((w_off + static_cast<size_t>(w) * w_slot + static_cast<size_t>(t) * kBM * row_b) % 128 == 0,
                  "W slot");

    // tensor-copy boxes: within the box limits; bytes landed = the barrier's expected count
    CHECK(kBM <= 256 && TN / CL <= 256 && TN % CL == 0 && kKB * 2 <= 128, "boxes");
    CHECK(static_cast<size_t>(row_b) * kBM * WT == w_slot, "W box bytes");
    // the slot's barrier expects the bytes of every CTA's multicast share
    CHECK(static_cast<size_t>(KSUB) * CL * kKB * (TN / CL) * 2 == b_slot, "x box bytes");
    // coordinates: innermost x times the element size on 16 bytes and inside the row
    const int64_t row_bytes = (K / 32) * (fmt == kPfQ8_0 ? 34 : 18);
    CHECK(row_bytes % 16 == 0, "W row stride");
    for (int64_t c = 0; c < nC; c += (c < 4 || c + 4 >= nC) ? 1 : std::max<int64_t>(1, nC / 64)) {
        const int64_t x = c * (row_b / esz);   // in the map's elements
        CHECK((x * esz) % 16 == 0 && (x * esz) + row_b <= row_bytes && x < INT32_MAX, "W x %lld", (long long)x);
    }
    if (fmt == kPfQ8_0)   // a thread's nine words of block 2 * sub + hsel lie inside its 272-byte row
        for (int sub = 0; sub < 4; ++sub)
            for (int hsel = 0; hsel < 2; ++hsel) CHECK(4 * (17 * sub + 8 * hsel + 9) <= row_b, "Q8_0 block words");
    for (int64_t j = 0; j < nK; j += (j < 4 || j + 4 >= nK) ? 1 : std::max<int64_t>(1, nK / 64))
        for (int a = 0; a < KSUB; ++a) {
            const int64_t x = (j * KSUB + a) * kKB;
            CHECK((x * 2) % 16 == 0 && x + kKB <= K, "x x %lld", (long long)x);
        }
    for (int64_t by = 0; by < pl.grid_y; ++by)
        for (int r = 0; r < CL; ++r) {
            const int64_t yc = by * TN + static_cast<int64_t>(r) * (TN / CL);   // rows past M read the fill value
            CHECK(yc >= 0 && yc + TN / CL <= INT32_MAX, "x y %lld", (long long)yc);
        }
    // W rows of the last CTA's tiles (rows past N read zeros)
    CHECK((pl.grid_x - 1) * rows_per_cta + (WT - 1) * kBM <= INT32_MAX, "W y");

    // dequantising warps: reads of the packed slot; tensor-memory writes.  With
    // 8 warps (the rule's tiles), warp w writes block half w / 4 of every atom;
    // with 16 (16-token tiles: one slot per 256-K chunk of one weight tile),
    // warp w writes blocks w / 4 and w / 4 + 4 of the chunk (atom b / 2, half
    // b mod 2), reading only those blocks' words.
    const bool small = TN == 16;
    CHECK(!small || (KSUB == 4 && WT == 1), "16-token tiles: one slot per chunk of one tile");
    const int dq = small ? 16 : 8;
    static unsigned char cover[4][kBM][kAtomCols];
    for (int s = 0; s < NSA; ++s)
        for (int t = 0; t < WT; ++t) {
            std::fill(&cover[0][0][0], &cover[0][0][0] + 4 * kBM * kAtomCols, 0);
            auto mark = [&](int w, int a, int half) {
                const int quarter = w & 3;
                const int64_t base = a0 + static_cast<int64_t>((s * KSUB + a) * WT + t) * kAtomCols;
                for (int lane = 0; lane < 32; ++lane) {
                    const int r = 32 * quarter + lane;
                    CHECK(r / 32 == (w & 3), "lane quarter of warp %d", w);
                    CHECK(static_cast<size_t>(NW - 1) * w_slot + static_cast<size_t>(t) * kBM * row_b +
                                  static_cast<size_t>(r) * row_b + row_b <=
                              static_cast<size_t>(NW) * w_slot,
                          "packed read");
                    const int64_t c0 = base + 16 * half;
                    CHECK(c0 >= a0 && c0 % 16 == 0 && base % 32 == 0 && c0 + 16 <= a_end, "A columns");
                    for (int j = 0; j < 16; ++j) ++cover[a][r][16 * half + j];
                }
            };
            if (!small) {
                for (int w = 0; w < dq; ++w)
                    for (int a = 0; a < KSUB; ++a) mark(w, a, w >> 2);
            } else {
                for (int w = 0; w < dq; ++w)
                    for (int k = 0; k < 2; ++k) {
                        const int b = (w >> 2) + 4 * k;
                        const int words = fmt == kPfQ8_0 ? 17 * (b >> 1) + 8 * (b & 1) + 9 : 9 * (b >> 1) + 4 * (b & 1) + 5;
                        CHECK(4 * words <= row_b, "block %d words", b);
                        mark(w, b >> 1, b & 1);
                    }
            }
            for (int a = 0; a < KSUB; ++a) {
                for (int r = 0; r < kBM; ++r)
                    for (int c = 0; c < kAtomCols; ++c)
                        CHECK(cover[a][r][c] == 1, "A cell %d,%d written %d times", r, c, cover[a][r][c]);
                // the MMAs of this atom read columns [base, base + 32) in four K = 16 steps of 8 columns
                const int64_t base = a0 + static_cast<int64_t>((s * KSUB + a) * WT + t) * kAtomCols;
                for (int k = 0; k < 4; ++k) CHECK(base + 8 * k + 8 <= a_end, "MMA A columns");
            }
        }
    for (int t = 0; t < WT; ++t) CHECK(static_cast<int64_t>(t + 1) * TN <= a0, "accumulator %d", t);
    if (fmt == kPfQ4_0)
        for (int sub = 0; sub < 4; ++sub) CHECK(4 * (9 * sub + 8) + 4 <= kPackedRowBytes, "block words");

    // epilogue: each (lane quarter, 32-column chunk) read by exactly one warp, inside the accumulators
    static unsigned char ecover[4][16];
    std::fill(&ecover[0][0], &ecover[0][0] + 64, 0);
    const int warps = prefill_threads(TN == 16) / 32;
    if (TN < 32) {
        // 16-token tiles: the first warp of each lane quarter reads its 16 columns
        for (int w = 0; w < warps; ++w)
            if ((w >> 2) == 0) ++ecover[w & 3][0];
        for (int q = 0; q < 4; ++q) CHECK(ecover[q][0] == 1, "epilogue quarter %d read %d times", q, ecover[q][0]);
        // split K: the CTAs' row shares cover the 128 rows once, and every row's
        // owner (as the kernel computes it) holds it
        int rows = 0;
        const int rmax = (kBM + SK - 1) / SK;
        for (int z = 0; z < SK; ++z) {
            const int r0 = kBM * z / SK, r1 = kBM * (z + 1) / SK;
            CHECK(r0 == rows && r1 >= r0 && r1 - r0 <= rmax, "split-K rows %d", z);
            for (int rl = r0; rl < r1; ++rl) CHECK(((rl + 1) * SK - 1) / kBM == z, "split-K owner of row %d", rl);
            rows = r1;
        }
        CHECK(rows == kBM, "split-K row cover");
    } else {
        for (int w = 0; w < warps; ++w) {
            const int quarter = w & 3, nq = (warps - quarter + 3) / 4, rank = w >> 2;
            for (int c0 = 32 * rank; c0 < WT * TN; c0 += 32 * nq) {
                CHECK(c0 + 32 <= WT * TN && (c0 % TN) + 32 <= TN, "epilogue columns");
                ++ecover[quarter][c0 / 32];
            }
        }
        for (int q = 0; q < 4; ++q)
            for (int c = 0; c < WT * TN / 32; ++c)
                CHECK(ecover[q][c] == 1, "epilogue chunk %d,%d read %d times", q, c, ecover[q][c]);
    }
}

}  // namespace

int main()
{
    const int64_t Ns[] = {1,   2,   7,    9,    16,   20,   33,   40,   64,    77,    96,    100,   130,   300,
                          333, 515, 600,  640,  1000, 2560, 4096, 4133, 6144,  8192,  12288, 14336, 28672, 128256};
    const int64_t Ks[] = {256,  512,  768,  1024, 2048, 2304, 2560, 2816, 3072,
                          3328, 3584, 3840, 4096, 5632, 6144, 6912, 8192, 14336};
    for (int fmt : {kQ4_0, kQ8_0, kQ2W})
        for (int64_t N : Ns)
            for (int64_t K : Ks)
                for (int M = 1; M <= 8; ++M) check_plan(fmt, N, K, M, 1, false);
    for (int64_t N : Ns)
        for (int64_t K : Ks)
            for (int slots : {2, 3, 5, 8, 10, 64})
                if (N * slots < 200000) check_plan(kQ4_0, N, K, 1, slots, false);
    for (int64_t N : Ns)
        for (int64_t K : Ks)
            for (int M = 1; M <= 8; ++M) {
                check_swiglu(N, K, M);
                check_plan(kQ4_0, N, K, M, 1, true);
                check_plan(kQ8_0, N, K, M, 1, true);
            }
    // every shape of the measured launch table, in each call form that can look it up
    for (const TuneEntry &e : kTuneTable) {
        const int f = e.fmt == 3 ? kQ4_0 : (e.fmt == 4 ? kQ8_0 : e.fmt);
        check_plan(f, e.N, e.K, e.M, 1, e.fmt >= 3);
        if (e.fmt == kQ4_0) {
            for (int slots : {8, 10}) check_plan(kQ4_0, e.N, e.K, 1, slots, false);
            check_swiglu(e.N, e.K, e.M);
            if (e.N % 2 == 0) check_swiglu(e.N / 2, e.K, e.M);
        }
    }
    const int64_t pN[] = {1, 127, 128, 129, 640, 4096, 14336, 128256, (int64_t(1) << 31) - 1};
    const int64_t pK[] = {32, 256, 512, 2560, 4096, 14336, (int64_t(1) << 30) - 256, int64_t(1) << 30};
    const int64_t pM[] = {1,   2,   63,   64,    65,    127,    128,           129,               192,
                          255, 256, 257,  511,   512,   513,    1024,          4096,              16384,
                          65535LL * 256,  65535LL * 256 + 1,    int64_t(1) << 24, (int64_t(1) << 31) - 1};
    for (int64_t N : pN)
        for (int64_t K : pK)
            for (int64_t M : pM)
                for (int sms : {152, 148, 132, 1})
                    for (int nw : {0, 1, 2, 3, 5, 8})
                        for (int ns : {0, 2, 3, 4, 6})
                            for (int cl : {0, 1, 2}) check_prefill(N, K, M, sms, nw, ns, cl, 0, 0);
    // every token tile and weight-tile count forced, over the same shapes
    for (int64_t N : pN)
        for (int64_t K : pK)
            for (int64_t M : pM)
                for (int tn : {64, 128, 192, 256})
                    for (int wt : {1, 2})
                        for (int cl : {1, 2})
                            for (int ks : {0, 1, 2, 4}) check_prefill(N, K, M, 152, 0, 0, cl, tn, wt, ks);
    // Q8_0 weights, and split K over up to 8 CTAs (automatic and forced), over the same shapes
    for (int64_t N : pN)
        for (int64_t K : pK)
            for (int64_t M : pM)
                for (int sms : {152, 132, 1}) {
                    for (int sk : {0, -1, 2, 3, 8}) check_prefill(N, K, M, sms, 0, 0, 0, 0, 0, 0, kPfQ8_0, sk);
                    for (int sk : {-1, 2, 5, 8}) check_prefill(N, K, M, sms, 0, 0, 0, 0, 0, 0, kPfQ4_0, sk);
                    check_prefill(N, K, M, sms, 1, 0, 2, 0, 0, 0, kPfQ8_0, 0);
                }
    std::printf("checked %ld plans, %ld failures\n", g_checked, g_bad);
    return g_bad ? 1 : 0;
}
