// qmv_api.cu -- the C ABI (include/qmv.h): argument validation, the per-shape
// launch configuration, the device status word, and the generic kernel's
// instantiations.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/qmv.h"
#include "qmv_gemv.cuh"
#include "qmv_launch.h"
#include "qmv_prefill.h"
#include "qmv_tune_table.h"

namespace qmv {

// One status word per device; kernels receive its address.
__device__ int g_device_status;

// Where qmv_device_status leaves the word it fetched and cleared: one slot per
// concurrent reader (a host-side ticket picks the slot).
constexpr int kFetchSlots = 64;
__device__ int g_status_fetched[kFetchSlots];

__global__ void status_fetch_clear_kernel(int *status, int *slot) { *slot = atomicExch(status, 0); }

#ifdef QMV_PHASE_STAMPS
// Phase-timeline builds only: [record count, records of kPhaseWords words].
__device__ unsigned long long g_phase_buf[1 + static_cast<size_t>(kPhaseWords) * kPhaseCap];
std::atomic<unsigned> g_phase_seq{0};
#endif

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int *> g_status_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];
std::atomic<int> g_pdl{1};
std::atomic<unsigned> g_fetch_ticket{0};

// Failure detection is tested without a GPU fault: QMV_TEST_SKIP_COPY=
// "decode:N" or "prefill:N" makes the N-th launch (counted from 1) of the
// streaming decode kernel or of the prefill kernel in this process skip one
// bulk copy whose bytes a barrier still expects.  The wait on that barrier
// then runs out, the kernel records QMV_DEV_TIMEOUT, waits (bounded) for its
// other copies and returns; nothing else of the call changes.  Unset in every
// normal run.
constexpr int kArmDecode = 0, kArmPrefill = 1;
std::atomic<long long> g_launches_seen[2];

bool test_skip_this_launch(int kind)
{
    static int armed_kind = -1;
    static long long armed_n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        const char *e = std::getenv("QMV_TEST_SKIP_COPY");
        if (!e) return;
        const char *c = std::strchr(e, ':');
        if (!c) return;
        if (!std::strncmp(e, "decode", static_cast<size_t>(c - e))) armed_kind = kArmDecode;
        else if (!std::strncmp(e, "prefill", static_cast<size_t>(c - e))) armed_kind = kArmPrefill;
        armed_n = std::atoll(c + 1);
    });
    if (armed_kind != kind) return false;
    return g_launches_seen[kind].fetch_add(1) + 1 == armed_n;
}

cudaError_t current_device(int *dev)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
    return cudaSuccess;
}

cudaError_t device_info(int dev, int **status, int *sms, int *smem_optin)
{
    int *sp = g_status_ptr[dev].load(std::memory_order_acquire);
    if (!sp) {
        void *addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_device_status);
        if (e != cudaSuccess) return e;
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev].store(v, std::memory_order_relaxed);
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        g_smem_optin[dev].store(v, std::memory_order_relaxed);
        sp = static_cast<int *>(addr);
        g_status_ptr[dev].store(sp, std::memory_order_release);
    }
    *status = sp;
    *sms = g_sm_count[dev].load(std::memory_order_relaxed);
    *smem_optin = g_smem_optin[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int lanes_per_row(int U, int M, int64_t N, int sms)
{
    // G lanes share a row, each taking every G-th 256-weight unit.
    if (M <= 2) {
        // One or two tokens: bound by the weight stream.  Rows of 9..15 units
        // get one unit per lane (e.g. K = 2560: G = 10, three rows per warp).
        if (U > 8 && U <= 16 && U % 8 != 0) return U;
        // Otherwise the largest power of two up to 16 that divides the row, at
        // least 8 for rows of 8 or more units (short rows otherwise leave most
        // warps without work), never more lanes than units.
        int G = 1;
        while (G * 2 <= 16 && U % (G * 2) == 0) G *= 2;
        if (G < 8 && U >= 8) G = 8;
        while (G > 1 && G > U) G >>= 1;
        return G;
    }
    // Several tokens: bound by arithmetic per row, so rows are spread over as
    // few lanes as still give every SM about four row groups (measured on
    // Q4_0 tables of 512..28672 rows at 8 tokens), at most 16 lanes and no more
    // than the smallest power of two that covers the row.
    int G = 1;
    while (G < 16 && N * G < int64_t(4) * 32 * (sms > 0 ? sms : 1)) G *= 2;
    int cover = 1;
    while (cover < U) cover *= 2;
    return G < cover ? G : cover;
}

struct Plan {
    bool streaming;
    int grid, warps;
    size_t smem;
};

// Launch-shape overrides for tuning sweeps: QMV_GEMV_TUNE="warps=16,stages=3,
// G=8,SP=1,ctas=2,share=2,early=1" (any subset; 0 or absent = the built-in
// rule; early = stages requested before the previous grid completes).
// ctas = CTAs per SM in the grid; share = the fraction 1/share of an SM's
// shared memory one CTA may use (share=2 leaves room for the next call's CTA
// to become resident early under programmatic dependent launch).  N=, K= and
// M= restrict the override to one table shape (N the planned rows: 2N for the
// fused SwiGLU, the expert's rows for the multi-expert call).
struct Tune {
    int warps = 0, stages = 0, G = 0, SP = 0, ctas = 0, share = 0, early = -1;
    // optional: apply only to the table shape N x K at M tokens (0 = every shape)
    long long N = 0, K = 0;
    int M = 0;
};

const Tune &tune_overrides()
{
    static Tune t;
    static std::once_flag once;
    std::call_once(once, [] {
        const char *env = std::getenv("QMV_GEMV_TUNE");
        if (!env) return;
        const char *c = env;
        while (*c) {
            char key[16] = {0};
            int k = 0;
            while (*c && *c != '=' && k < 15) key[k++] = *c++;
            if (*c != '=') break;
            ++c;
            const long long vl = std::atoll(c);
            const int v = static_cast<int>(vl);
            while (*c && *c != ',') ++c;
            if (*c == ',') ++c;
            if (!std::strcmp(key, "N")) t.N = vl;
            else if (!std::strcmp(key, "K")) t.K = vl;
            else if (!std::strcmp(key, "M")) t.M = v;
            else if (!std::strcmp(key, "warps")) t.warps = v;
            else if (!std::strcmp(key, "stages")) t.stages = v;
            else if (!std::strcmp(key, "G")) t.G = v;
            else if (!std::strcmp(key, "SP")) t.SP = v;
            else if (!std::strcmp(key, "ctas")) t.ctas = v;
            else if (!std::strcmp(key, "share")) t.share = v;
            else if (!std::strcmp(key, "early")) t.early = v;
        }
    });
    return t;
}

const TuneEntry *tune_lookup(int fmt, int64_t N, int64_t K, int M)
{
    for (const TuneEntry &e : kTuneTable)
        if (e.fmt == fmt && e.M == M && e.N == N && e.K == K) return &e;
    return nullptr;
}

// Choose the launch of the streaming kernel (or fall back to the generic one).
// Order of precedence: QMV_GEMV_TUNE overrides (sweeps), the measured table
// (qmv_tune_table.h), then a rule by weight bytes per SM.  Lanes-per-row (G)
// fixes the summation order, so it depends only on (format, N, K, M) -- the
// multi-expert call looks up its per-expert shape and matches a single call
// bit for bit.
Plan plan_gemv(int fmt, GemvParams &p, int M, int sms, int smem_optin)
{
    Plan pl{false, 0, 8, 0};
    if (p.K % 256 != 0 || p.K == 0) return pl;
    // staged with 4-byte (fp16 pairs), 8-byte (fp32 pairs) or 16-byte (codes) loads of 16-byte-aligned rows
    const uintptr_t xaddr = p.xq ? reinterpret_cast<uintptr_t>(p.xq)
                                 : (p.xf ? reinterpret_cast<uintptr_t>(p.xf) : reinterpret_cast<uintptr_t>(p.x));
    if (xaddr % 16 != 0) return pl;
    if (p.rows_total >= (int64_t(1) << 31)) return pl;             // 32-bit row indices
    const int64_t U = p.K / 256;
    if (U > (1 << 20)) return pl;
    p.U = static_cast<int>(U);
    const int unit_bytes = fmt == kQ4_0 ? 144 : (fmt == kQ2W ? 80 : 272);
    const Tune &tu_all = tune_overrides();
    // One problem (a plain call, or the fused SwiGLU's gate and up tables
    // stacked row by row) is planned as one table of rows_total rows; the
    // multi-expert call by its per-expert shape.
    const int64_t Nplan = p.n_problems == 1 ? p.rows_total : p.N;
    // Q4_0 and Q8_0 against Q8_1 activations have their own entries (table
    // formats 3 and 4): their per-unit arithmetic differs from the fp16 path's.
    const TuneEntry *te = tune_lookup(p.xq8 ? (fmt == kQ8_0 ? 4 : 3) : fmt, Nplan, p.K, M);
    const Tune none{};
    const bool tu_applies = (tu_all.N == 0 || tu_all.N == Nplan) && (tu_all.K == 0 || tu_all.K == p.K) &&
                            (tu_all.M == 0 || tu_all.M == M);
    const Tune &tu = tu_applies ? tu_all : none;

    // defaults by rule
    const int64_t wbytes_per_sm = Nplan * (p.K / 256) * unit_bytes / (sms > 0 ? sms : 1);
    const bool big = wbytes_per_sm > 128 * 1024 && M <= 2;
    int G = lanes_per_row(p.U, M, Nplan, sms);
    // 12 warps for large tables at one or two tokens, and for three or more
    // tokens (one CTA per SM: its warps are the latency hiding; measured on the
    // Llama-3-8B and Q8_0 tables at 4 and 8 tokens)
    int warps = (big || M > 2) ? 12 : 8;
    int stages = 2;
    int SP = 1;
    int share = 1;
    if (big && p.U % 8 == 0) {
        G = 8;
        if (p.U % 16 == 0) SP = 2;
    }
    if (p.n_problems > 1) {
        // The multi-expert call cannot request weights before the previous
        // kernel (which may have written the expert indices) completes, so it
        // keeps more warps and stages in flight from the start (measured on
        // 10 x 640x2560 and 8 x 512x2048 expert calls).
        warps = 12;
        stages = 3;
    }
    if (te) {
        if (te->G) G = te->G;
        warps = te->warps;
        stages = te->stages;
        SP = te->SP;
        share = te->share;
    }
    if (tu.G >= 1 && tu.G <= 32) G = tu.G;
    if (tu.warps >= 1) warps = tu.warps;
    if (tu.stages >= 1) stages = tu.stages;
    if (tu.SP >= 1) SP = tu.SP;
    if (tu.share >= 1) share = tu.share;
    const int ctas_per_sm = (tu.ctas >= 1 && tu.ctas <= 4) ? tu.ctas : 1;

    if (p.W2) {
        // fused SwiGLU: a gate row and its up row share a row group, so the
        // group holds an even number of rows: G a power of two, at most 16.
        int g2 = 1;
        while (g2 * 2 <= G && g2 * 2 <= 16) g2 *= 2;
        G = g2;
    }
    p.G = G;
    // Passes per stage: odd for G < 8 keeps the lanes of a quarter warp in
    // distinct banks; any value works for G >= 8.
    p.SP = (SP >= 1 && SP <= 8 && ((SP & 1) || p.G >= 8)) ? SP : 1;
    if (share < 1 || share > 4) share = 1;
    const int max_warps = (M <= 2) ? 16 : 12;
    if (warps < 1 || warps > max_warps) warps = 8;

    const int RG = 32 / p.G;
    const int64_t groups = (p.rows_total + RG - 1) / RG;
    const int64_t max_grid = static_cast<int64_t>(sms) * ctas_per_sm;
    int grid = static_cast<int>(groups < max_grid ? groups : max_grid);
    if (grid < 1) grid = 1;
    const int64_t rows_per_cta = (p.rows_total + grid - 1) / grid;
    int64_t pmax = (rows_per_cta + p.N - 1) / p.N + 1;
    if (pmax > p.n_problems) pmax = p.n_problems;
    p.max_local_problems = static_cast<int>(pmax);
    const size_t xbytes = static_cast<size_t>(pmax) * M * p.U * (p.xq8 ? kXQ8UnitBytes : kXUnitBytes);
    const size_t budget = static_cast<size_t>(smem_optin) / (ctas_per_sm > share ? ctas_per_sm : share) - 1024;
    if (xbytes + 8 * 1024 > budget) return pl;
    // Fit the ring: fewer stages, then fewer passes, then fewer warps.
    for (int attempt = 0; attempt < 8; ++attempt) {
        const size_t per_stage = static_cast<size_t>(warps) * (32 * p.SP * unit_bytes + 8);
        int S = static_cast<int>((budget - xbytes) / per_stage);
        if (S > stages) S = stages;
        if (S >= 2) {
            p.S = S;
            // stages requested before the activation loads: one for a plain
            // call (before the previous grid completes); none for the
            // multi-expert call, whose stages follow its first activation
            // loads (requesting them all right after the indices measured
            // 1467 against 1503 GB/s on its workload)
            p.early = tu.early >= 0 ? tu.early : (p.n_problems > 1 ? 0 : 1);
            pl.streaming = true;
            pl.grid = grid;
            pl.warps = warps;
            pl.smem = gemv_smem_bytes(fmt, M, static_cast<int>(pmax), p.U, warps, S, p.SP, p.xq8 != 0);
            return pl;
        }
        if (p.SP > 1) p.SP = 1;
        else if (warps > 4) warps -= 4;
        else break;
    }
    return pl;
}

cudaError_t launch_streaming(int fmt, const GemvParams &p0, int M, const Plan &pl, cudaStream_t stream, bool pdl)
{
    GemvParams p = p0;
    p.test_skip_copy = test_skip_this_launch(kArmDecode) ? 1 : 0;
#ifdef QMV_PHASE_STAMPS
    void *ph = nullptr;
    if (cudaGetSymbolAddress(&ph, g_phase_buf) == cudaSuccess) p.phase = static_cast<unsigned long long *>(ph);
    p.phase_seq = g_phase_seq.fetch_add(1);
#endif
    if (fmt == kQ4_0 && p.xq8) return launch_gemv_stream_q4_0_q8_1(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
    if (fmt == kQ8_0 && p.xq8) return launch_gemv_stream_q8_0_q8_1(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
    if (fmt == kQ4_0 && p.W2) return launch_gemv_stream_q4_0_swiglu(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
    if (fmt == kQ4_0)
        return p.xf ? launch_gemv_stream_q4_0_f32(M, p, pl.grid, pl.warps, pl.smem, stream, pdl)
                    : launch_gemv_stream_q4_0(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
    if (fmt == kQ2W) return launch_gemv_stream_q2w(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
    return launch_gemv_stream_q8_0(M, p, pl.grid, pl.warps, pl.smem, stream, pdl);
}

// Whether a plain Q4_0 / Q8_0 decode call of M tokens goes to the tensor
// cores.  Measured on the GB300 (us per call back to back, streaming kernel
// against tensor cores): eight tokens, the tensor cores win on every table
// (Q8_0 12288x2560 21.9 -> 13.0, 2560x6144 24.0 -> 9.1, 8192x2048 12.6 -> 9.3;
// Q4_0 4096x14336 43.4 -> 15.3, 128256x4096 193 -> 107); four tokens they win
// from K = 2560 up (Q8_0 12288x2560 14.3 -> 13.0, 2560x6144 10.5 -> 9.1;
// Q4_0 4096x14336 21.7 -> 15.3) and lose below (Q8_0 8192x2048 8.0 against
// 9.3); two tokens the streaming kernel wins.  QMV_TC_MIN_TOKENS=n replaces
// the rule by "n tokens or more" for sweeps (0 or above 8: never).
bool tc_route(int64_t K, int M)
{
    static const int forced = [] {
        const char *e = std::getenv("QMV_TC_MIN_TOKENS");
        if (!e) return -1;
        const int n = std::atoi(e);
        return (n >= 1 && n <= 8) ? n : 1 << 20;
    }();
    if (forced >= 0) return M >= forced;
    return M >= 8 || (M >= 4 && K >= 2560);
}

qmv_status run_gemv(int fmt, const void *W, const int32_t *idx, int64_t n_experts, const void *x, float *y,
                    int64_t N, int64_t K, int64_t M, int n_problems, cudaStream_t stream, const void *W2 = nullptr,
                    const float *xf = nullptr, bool xq8 = false, const int8_t *xq = nullptr,
                    const uint16_t *xq_d = nullptr, const int32_t *xq_s = nullptr)
{
    if (xf && fmt != kQ4_0) return QMV_ERR_SHAPE;   // fp32 activations: Q4_0 kernels only
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    int *status = nullptr;
    int sms = 0, optin = 0;
    if (device_info(dev, &status, &sms, &optin) != cudaSuccess) return QMV_ERR_CUDA;

    GemvParams p = {};
    p.W = static_cast<const uint8_t *>(W);
    p.x = static_cast<const __half *>(x);
    p.xf = xf;
    p.xq8 = xq8 ? 1 : 0;
    p.xq = xq;
    p.xq_d = xq_d;
    p.xq_s = xq_s;
    p.y = y;
    p.expert_idx = idx;
    p.N = N;
    p.K = K;
    p.n_experts = n_experts;
    p.row_bytes = (K / 32) * (fmt == kQ4_0 ? 18 : (fmt == kQ2W ? 10 : 34));
    p.n_problems = n_problems;
    p.max_local_problems = n_problems;
    p.rows_total = N * n_problems;
    p.W2 = static_cast<const uint8_t *>(W2);
    if (W2) p.rows_total = 2 * N;     // gate and up rows interleaved
    p.status = status;
    const int Mk = static_cast<int>(M);
    const bool pdl = g_pdl.load(std::memory_order_relaxed) != 0;

    cudaError_t e;
    // Several tokens of a plain Q4_0 / Q8_0 GEMV on the tensor cores (the
    // prefill kernel's 16-token tiles, split along K over a cluster where the
    // weight tiles alone leave SMs idle) where tc_route() says they win.
    if (n_problems == 1 && !W2 && !xf && !xq8 && (fmt == kQ4_0 || fmt == kQ8_0) && tc_route(K, Mk) &&
        K % 256 == 0 && aligned(W, 16) && aligned(x, 16)) {
        const PrefillPlan pp = prefill_plan(N, K, M, sms, fmt == kQ8_0 ? kPfQ8_0 : kPfQ4_0, -1);
        if (pp.ok && pp.TN == 16) {
            e = launch_prefill(pp, W, x, y, N, K, M, status, stream, pdl, test_skip_this_launch(kArmDecode));
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                return QMV_ERR_LAUNCH;
            }
            return QMV_OK;
        }
    }
    GemvParams p0 = p;
    Plan pl = plan_gemv(fmt, p, Mk, sms, optin);
    if (!pl.streaming && Mk > 1 && n_problems == 1) {
        // The activations of all the tokens do not fit in shared memory beside
        // a weight ring (e.g. 8 tokens of K = 14336 in fp16): split the tokens
        // into the fewest launches whose activations fit.  Each launch streams
        // the weights again, which is far cheaper than the generic kernel.
        for (int parts = 2; parts <= Mk; ++parts) {
            const int mc = (Mk + parts - 1) / parts;
            GemvParams probe = p0;
            if (!plan_gemv(fmt, probe, mc, sms, optin).streaming) continue;
            for (int m0 = 0; m0 < Mk; m0 += mc) {
                const int mm = Mk - m0 < mc ? Mk - m0 : mc;
                GemvParams ps = p0;
                if (ps.x) ps.x += static_cast<int64_t>(m0) * K;
                if (ps.xf) ps.xf += static_cast<int64_t>(m0) * K;
                if (ps.xq) {
                    ps.xq += static_cast<int64_t>(m0) * K;
                    ps.xq_d += static_cast<int64_t>(m0) * (K / 32);
                    ps.xq_s += static_cast<int64_t>(m0) * (K / 32);
                }
                ps.y += static_cast<int64_t>(m0) * N;
                Plan pp = plan_gemv(fmt, ps, mm, sms, optin);
                if (pp.streaming) {
                    e = launch_streaming(fmt, ps, mm, pp, stream, pdl);
                } else {   // not expected (fewer tokens than a part that fits), but correct
                    int64_t grid = ((W2 ? N : ps.rows_total) + 7) / 8;
                    if (grid > 32LL * sms) grid = 32LL * sms;
                    e = launch_gemv_generic(fmt, ps, mm, static_cast<int>(grid < 1 ? 1 : grid), stream, pdl);
                }
                if (e != cudaSuccess) {
                    (void)cudaGetLastError();
                    return QMV_ERR_LAUNCH;
                }
            }
            return QMV_OK;
        }
    }
    if (pl.streaming) {
        e = launch_streaming(fmt, p, Mk, pl, stream, pdl);
    } else {
        const int64_t warps_needed = W2 ? N : p.rows_total;
        int64_t grid = (warps_needed + 7) / 8;
        if (grid > 32LL * sms) grid = 32LL * sms;
        if (grid < 1) grid = 1;
        e = launch_gemv_generic(fmt, p, Mk, static_cast<int>(grid), stream, pdl);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QMV_ERR_LAUNCH;
    }
    return QMV_OK;
}

qmv_status check_common(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M, int64_t max_m)
{
    if (N < 0 || K < 0 || M < 0 || M > max_m) return QMV_ERR_SHAPE;
    if (K % 32 != 0) return QMV_ERR_SHAPE;
    if (N > (int64_t(1) << 40) || K > (int64_t(1) << 31)) return QMV_ERR_SHAPE;
    if (N == 0 || M == 0) return QMV_OK;
    if (!y) return QMV_ERR_NULL;
    if (K > 0 && (!W || !x)) return QMV_ERR_NULL;
    if (W && !aligned(W, 16)) return QMV_ERR_ALIGN;
    if (x && !aligned(x, 2)) return QMV_ERR_ALIGN;
    if (!aligned(y, 4)) return QMV_ERR_ALIGN;
    return QMV_OK;
}

}  // namespace

cudaError_t ensure_smem_optin(const void *func, size_t smem)
{
    if (smem <= 48 * 1024) return cudaSuccess;
    // Setting the attribute is cheap but not free; do it for the maximum once
    // per (kernel, device) pair and remember it.
    static std::mutex mu;
    static const void *seen_func[256];
    static int seen_dev[256];
    static int nseen = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < nseen; ++i)
        if (seen_func[i] == func && seen_dev[i] == dev) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    // The opt-in limit covers static and dynamic shared memory together.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess) return e;
    if (nseen < 256) {
        seen_func[nseen] = func;
        seen_dev[nseen] = dev;
        ++nseen;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv_generic(int fmt, const GemvParams &p, int M, int grid, cudaStream_t s, bool pdl)
{
    if (fmt == kQ4_0) return launch_ex(qmv_generic_kernel<kQ4_0>, dim3(grid), dim3(256), 0, s, pdl, p, M);
    if (fmt == kQ2W) return launch_ex(qmv_generic_kernel<kQ2W>, dim3(grid), dim3(256), 0, s, pdl, p, M);
    return launch_ex(qmv_generic_kernel<kQ8_0>, dim3(grid), dim3(256), 0, s, pdl, p, M);
}

}  // namespace qmv

using namespace qmv;

extern "C" {

qmv_status qmv_q4_0(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    return run_gemv(kQ4_0, W, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status qmv_q8_0(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    return run_gemv(kQ8_0, W, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status qmv_q4_0_q8_1(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                         qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    return run_gemv(kQ4_0, W, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    nullptr, true);
}

qmv_status qmv_q4_0_q8_1_pre(const void *W, const int8_t *q, const uint16_t *d_bits, const int32_t *sumq, float *y,
                             int64_t N, int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W, q, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    if (K > 0 && (!d_bits || !sumq)) return QMV_ERR_NULL;
    if ((d_bits && !aligned(d_bits, 2)) || (sumq && !aligned(sumq, 4))) return QMV_ERR_ALIGN;
    return run_gemv(kQ4_0, W, nullptr, 1, nullptr, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    nullptr, true, q, d_bits, sumq);
}

qmv_status qmv_q8_0_q8_1(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                         qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    return run_gemv(kQ8_0, W, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    nullptr, true);
}

qmv_status qmv_q8_0_q8_1_pre(const void *W, const int8_t *q, const uint16_t *d_bits, float *y, int64_t N,
                             int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W, q, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    if (K > 0 && !d_bits) return QMV_ERR_NULL;
    if (d_bits && !aligned(d_bits, 2)) return QMV_ERR_ALIGN;
    return run_gemv(kQ8_0, W, nullptr, 1, nullptr, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    nullptr, true, q, d_bits, nullptr);
}

qmv_status qmv_quantize_q8_1(const void *x, int8_t *q, uint16_t *d_bits, int32_t *sumq, int64_t M, int64_t K,
                             qmv_stream_t stream)
{
    if (M < 0 || K < 0 || K % 32 != 0 || K > (int64_t(1) << 31) || M > (int64_t(1) << 31)) return QMV_ERR_SHAPE;
    if (M == 0 || K == 0) return QMV_OK;
    if (!x || !q || !d_bits || !sumq) return QMV_ERR_NULL;
    if (!aligned(x, 16) || !aligned(q, 8) || !aligned(d_bits, 2) || !aligned(sumq, 4)) return QMV_ERR_ALIGN;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    if (launch_quantize_q8_1(x, q, d_bits, sumq, M, K, reinterpret_cast<cudaStream_t>(stream),
                             g_pdl.load(std::memory_order_relaxed) != 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return QMV_ERR_LAUNCH;
    }
    return QMV_OK;
}

qmv_status qmv_q2w(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    return run_gemv(kQ2W, W, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream));
}

qmv_status qmv_q4_0_swiglu(const void *W_gate, const void *W_up, const void *x, float *y, int64_t N, int64_t K,
                           int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W_gate, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    if (K > 0 && !W_up) return QMV_ERR_NULL;
    if (W_up && !aligned(W_up, 16)) return QMV_ERR_ALIGN;
    if (N > (int64_t(1) << 39)) return QMV_ERR_SHAPE;     // 2N interleaved rows
    // K == 0 (W_up may then be null): y = silu(0) * 0 = 0, as the plain call gives.
    return run_gemv(kQ4_0, W_gate, nullptr, 1, x, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), W_up);
}

qmv_status qmv_q4_0_f32(const void *W, const float *x, float *y, int64_t N, int64_t K, int64_t M,
                        qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    if (x && !aligned(x, 4)) return QMV_ERR_ALIGN;
    return run_gemv(kQ4_0, W, nullptr, 1, nullptr, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    x);
}

qmv_status qmv_q4_0_swiglu_f32(const void *W_gate, const void *W_up, const float *x, float *y, int64_t N,
                               int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W_gate, x, y, N, K, M, 8);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    if (x && !aligned(x, 4)) return QMV_ERR_ALIGN;
    if (K > 0 && !W_up) return QMV_ERR_NULL;
    if (W_up && !aligned(W_up, 16)) return QMV_ERR_ALIGN;
    if (N > (int64_t(1) << 39)) return QMV_ERR_SHAPE;     // 2N interleaved rows
    return run_gemv(kQ4_0, W_gate, nullptr, 1, nullptr, y, N, K, M, 1, reinterpret_cast<cudaStream_t>(stream),
                    W_up, x);
}

qmv_status qmv_moe(const void *W_pool, const int32_t *expert_idx, int64_t n_experts, const void *x, float *y,
                   int64_t N, int64_t K, int64_t M, qmv_stream_t stream)
{
    qmv_status st = check_common(W_pool, x, y, N, K, M, 64);
    if (st != QMV_OK) return st;
    if (n_experts < 1) return QMV_ERR_SHAPE;
    if (N == 0 || M == 0) return QMV_OK;
    if (!expert_idx) return QMV_ERR_NULL;
    if (!aligned(expert_idx, 4)) return QMV_ERR_ALIGN;
    if (n_experts > (int64_t(1) << 31)) return QMV_ERR_SHAPE;
    // Each token is one problem of one row-set: M slots with 1 token each.
    return run_gemv(kQ4_0, W_pool, expert_idx, n_experts, x, y, N, K, 1, static_cast<int>(M),
                    reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The many-token GEMM on the tensor cores for Q4_0 (fmt kPfQ4_0) or Q8_0
// weights; shapes the tensor-core kernel does not take run on the generic
// kernel.
qmv_status run_prefill(int fmt, const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                       qmv_stream_t stream)
{
    qmv_status st = check_common(W, x, y, N, K, M, int64_t(1) << 24);
    if (st != QMV_OK || N == 0 || M == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (x && !aligned(x, 16)) return QMV_ERR_ALIGN;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    int *status = nullptr;
    int sms = 0, optin = 0;
    if (device_info(dev, &status, &sms, &optin) != cudaSuccess) return QMV_ERR_CUDA;
    const PrefillPlan pl = prefill_plan(N, K, M, sms, fmt, -1);
    if (pl.ok) {
        cudaError_t e = launch_prefill(pl, W, x, y, N, K, M, status, s, g_pdl.load(std::memory_order_relaxed) != 0,
                                       test_skip_this_launch(kArmPrefill));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return QMV_ERR_LAUNCH;
        }
        return QMV_OK;
    }
    // Other shapes: the generic kernel, eight tokens at a time per warp pass.
    GemvParams p = {};
    p.W = static_cast<const uint8_t *>(W);
    p.x = static_cast<const __half *>(x);
    p.y = y;
    p.N = N;
    p.K = K;
    p.n_experts = 1;
    p.row_bytes = (K / 32) * (fmt == kPfQ8_0 ? 34 : 18);
    p.n_problems = 1;
    p.max_local_problems = 1;
    p.rows_total = N;
    p.status = status;
    int64_t grid = (N + 7) / 8;
    if (grid > 32LL * sms) grid = 32LL * sms;
    if (grid < 1) grid = 1;
    cudaError_t e = launch_gemv_generic(fmt == kPfQ8_0 ? kQ8_0 : kQ4_0, p, static_cast<int>(M),
                                        static_cast<int>(grid), s, g_pdl.load() != 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QMV_ERR_LAUNCH;
    }
    return QMV_OK;
}

}  // namespace

qmv_status qmm_q4_0_prefill(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                            qmv_stream_t stream)
{
    return run_prefill(kPfQ4_0, W, x, y, N, K, M, stream);
}

qmv_status qmm_q8_0_prefill(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                            qmv_stream_t stream)
{
    return run_prefill(kPfQ8_0, W, x, y, N, K, M, stream);
}

qmv_status qmv_device_status(qmv_stream_t stream, int32_t *out)
{
    if (!out) return QMV_ERR_NULL;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    int *status = nullptr;
    int sms = 0, optin = 0;
    if (device_info(dev, &status, &sms, &optin) != cudaSuccess) return QMV_ERR_CUDA;
    // Fetch and clear in one atomic step, in `stream` order: a kernel on
    // another stream that sets a bit in between is never lost (it stays for
    // the next read).  Concurrent readers take different result slots.
    void *slots = nullptr;
    if (cudaGetSymbolAddress(&slots, g_status_fetched) != cudaSuccess) return QMV_ERR_CUDA;
    int *slot = static_cast<int *>(slots) + (g_fetch_ticket.fetch_add(1) % kFetchSlots);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    status_fetch_clear_kernel<<<1, 1, 0, s>>>(status, slot);
    if (cudaGetLastError() != cudaSuccess) return QMV_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpyAsync(&v, slot, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return QMV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QMV_ERR_CUDA;
    *out = v;
    return QMV_OK;
}

qmv_status qmv_read_probe(const void *buf, int64_t bytes, uint32_t *out, qmv_stream_t stream)
{
    if (bytes < 0 || bytes % 256 != 0 || bytes > (int64_t(1) << 46)) return QMV_ERR_SHAPE;
    if (!out || (bytes > 0 && !buf)) return QMV_ERR_NULL;
    if (!aligned(buf, 16) || !aligned(out, 4)) return QMV_ERR_ALIGN;
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    int *status = nullptr;
    int sms = 0, optin = 0;
    if (device_info(dev, &status, &sms, &optin) != cudaSuccess) return QMV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bytes == 0) return cudaMemsetAsync(out, 0, sizeof(uint32_t), s) == cudaSuccess ? QMV_OK : QMV_ERR_CUDA;
    if (launch_read_probe(buf, bytes, out, status, sms, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return QMV_ERR_LAUNCH;
    }
    return QMV_OK;
}

void qmv_set_pdl(int enable) { g_pdl.store(enable ? 1 : 0); }

const char *qmv_status_str(qmv_status s)
{
    switch (s) {
    case QMV_OK: return "ok";
    case QMV_ERR_NULL: return "null pointer";
    case QMV_ERR_ALIGN: return "misaligned pointer";
    case QMV_ERR_SHAPE: return "shape out of range";
    case QMV_ERR_LAUNCH: return "kernel launch failed";
    case QMV_ERR_DEVICE: return "device-side error";
    case QMV_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}

const char *qmv_version(void) { return "qmv 0.1.0 sm_103a"; }

#ifdef QMV_PHASE_STAMPS
// Phase-timeline builds only (not declared in include/qmv.h): copies up to
// max_records records of the streaming decode kernel's phase stamps to host
// memory, then resets the record count and the launch sequence.  Returns the
// number of records copied, or -1 on a CUDA error.
QMV_API int64_t qmv_phase_stamps(unsigned long long *host, int64_t max_records)
{
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    unsigned long long n = 0;
    if (cudaMemcpyFromSymbol(&n, g_phase_buf, sizeof(n)) != cudaSuccess) return -1;
    if (n > static_cast<unsigned long long>(kPhaseCap)) n = kPhaseCap;
    if (static_cast<int64_t>(n) > max_records) n = static_cast<unsigned long long>(max_records);
    if (n && cudaMemcpyFromSymbol(host, g_phase_buf, n * kPhaseWords * sizeof(unsigned long long),
                                  sizeof(unsigned long long)) != cudaSuccess)
        return -1;
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(g_phase_buf, &zero, sizeof(zero)) != cudaSuccess) return -1;
    g_phase_seq.store(0);
    return static_cast<int64_t>(n);
}
#endif

}  // extern "C"
