// qmv_probe.cu -- read-only bandwidth probe: streams a device buffer through
// per-warp shared-memory rings filled by bulk (TMA) copies, as the decode
// kernel streams its weights, with no arithmetic on the bytes.  Its rate is
// the measured read roofline the decode kernels are compared with, beside the
// copy (read + write) bandwidth (sm8x-bench reports its kernels against a
// measured bandwidth probe as well as the spec figure -- sm8x-bench,
// methodology bullets).
#include <cstdint>

#include "../../include/qmv.h"
#include "qmv_common.cuh"
#include "qmv_launch.h"

namespace qmv {

namespace {

constexpr int kProbeWarps = 8;
constexpr int kProbeStages = 3;
constexpr int kProbeLaneBytes = 256;                     // bytes one lane copies per stage
constexpr int kProbeSlotBytes = 32 * kProbeLaneBytes;    // one warp's stage
constexpr size_t kProbeSmem = static_cast<size_t>(kProbeWarps) * kProbeStages * (kProbeSlotBytes + 8);

// CTA b reads 256-byte chunks [c0, c1) of the buffer; warp w takes stage
// chunks w, w + warps, ... of 32 lanes x 256 bytes each.  After a stage lands
// every lane XORs the first 16 bytes of its piece into a checksum (the bytes
// are consumed, so nothing can skip the copy), then the slot is refilled.
__global__ void __launch_bounds__(kProbeWarps * 32, 1)
    read_probe_kernel(const uint8_t *buf, int64_t chunks, uint32_t *out, int *status)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t *ring = smem + static_cast<size_t>(warp) * kProbeStages * kProbeSlotBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(kProbeWarps) * kProbeStages *
                                                               kProbeSlotBytes) + warp * kProbeStages;
    const int64_t c0 = chunks * blockIdx.x / gridDim.x;
    const int64_t c1 = chunks * (blockIdx.x + 1) / gridDim.x;
    const int64_t n_stages_cta = (c1 - c0 + 31) / 32;                 // 32 chunks per stage
    const int64_t my_stages = n_stages_cta > warp ? (n_stages_cta - warp + kProbeWarps - 1) / kProbeWarps : 0;

    if (lane == 0) {
        for (int s = 0; s < kProbeStages; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    __syncwarp();
    const uint64_t policy = l2_evict_first_policy();
    int64_t issued = 0;
    auto issue = [&](int64_t t) {
        const int slot = static_cast<int>(t % kProbeStages);
        const int64_t chunk = c0 + (warp + t * kProbeWarps) * 32 + lane;
        const uint32_t bytes = chunk < c1 ? static_cast<uint32_t>(kProbeLaneBytes) : 0u;
        const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
        if (lane == 0) mbar_arrive_expect_tx(&bars[slot], total);
        __syncwarp();
        if (bytes)
            bulk_g2s_hint(ring + slot * kProbeSlotBytes + lane * kProbeLaneBytes, buf + chunk * kProbeLaneBytes,
                          bytes, &bars[slot], policy);
    };
    for (; issued < my_stages && issued < kProbeStages; ++issued) issue(issued);

    uint32_t acc = 0;
    int64_t consumed = 0;
    bool alive = true;
    for (int64_t t = 0; t < my_stages; ++t) {
        const int slot = static_cast<int>(t % kProbeStages);
        const uint32_t parity = static_cast<uint32_t>((t / kProbeStages) & 1);
        if (!__all_sync(0xffffffffu, mbar_try_wait(&bars[slot], parity)) &&
            !mbar_wait_warp(&bars[slot], parity, status)) {
            alive = false;
            break;
        }
        consumed = t + 1;
        const int64_t chunk = c0 + (warp + t * kProbeWarps) * 32 + lane;
        if (chunk < c1) {
            const uint4 v = *reinterpret_cast<const uint4 *>(ring + slot * kProbeSlotBytes + lane * kProbeLaneBytes);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (issued < my_stages) issue(issued++);
    }
    if (!alive && lane == 0)
        for (int64_t j = consumed; j < issued; ++j)
            mbar_wait_bounded(&bars[j % kProbeStages], static_cast<uint32_t>((j / kProbeStages) & 1), nullptr);
    __syncwarp();
    acc = __reduce_xor_sync(0xffffffffu, acc);
    if (lane == 0 && acc) atomicXor(out, acc);
}

}  // namespace

cudaError_t launch_read_probe(const void *buf, int64_t bytes, uint32_t *out, int *status, int sms, cudaStream_t s)
{
    const void *k = reinterpret_cast<const void *>(read_probe_kernel);
    cudaError_t e = ensure_smem_optin(k, kProbeSmem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(out, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    read_probe_kernel<<<sms, kProbeWarps * 32, kProbeSmem, s>>>(static_cast<const uint8_t *>(buf),
                                                                bytes / kProbeLaneBytes, out, status);
    return cudaGetLastError();
}

}  // namespace qmv
