// qmv_gemv_q4_0_q81.cu -- the streaming decode kernel for Q4_0 weights against
// activations quantised to Q8_1 (8-bit codes per block of 32) while each CTA
// stages them, with integer dots; and the standalone Q8_1 quantisation.
#include "qmv_gemv.cuh"
#include "qmv_launch.h"

namespace qmv {

template <int M, int MAXT>
static cudaError_t launch_q81_t(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    auto kernel = qmv_stream_kernel<kQ4_0, M, MAXT, false, false, false, true>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void *>(kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_ex(kernel, dim3(grid), dim3(warps * 32), smem, s, pdl, p);
}

// Up to 8 warps per CTA for every token count; up to 16 for one or two tokens.
template <int M>
static cudaError_t launch_q81_one(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    if (p.expert_idx || p.W2 || p.xf || !p.xq8) return cudaErrorInvalidValue;
    if (warps <= 8) return launch_q81_t<M, 256>(p, grid, warps, smem, s, pdl);
    if constexpr (M <= 2) {
        if (warps <= 16) return launch_q81_t<M, 512>(p, grid, warps, smem, s, pdl);
    } else {
        if (warps <= 12) return launch_q81_t<M, 384>(p, grid, warps, smem, s, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemv_stream_q4_0_q8_1(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                         cudaStream_t s, bool pdl)
{
    switch (M) {
    case 1: return launch_q81_one<1>(p, grid, warps, smem, s, pdl);
    case 2: return launch_q81_one<2>(p, grid, warps, smem, s, pdl);
    case 3: return launch_q81_one<3>(p, grid, warps, smem, s, pdl);
    case 4: return launch_q81_one<4>(p, grid, warps, smem, s, pdl);
    case 5: return launch_q81_one<5>(p, grid, warps, smem, s, pdl);
    case 6: return launch_q81_one<6>(p, grid, warps, smem, s, pdl);
    case 7: return launch_q81_one<7>(p, grid, warps, smem, s, pdl);
    case 8: return launch_q81_one<8>(p, grid, warps, smem, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

// One thread per 16-byte chunk of 8 activations; the four chunks of a block
// are adjacent lanes (the chunk count is a multiple of 4 and so is every
// warp's first chunk).  Lanes past the end take part in the shuffles only.
// Programmatic dependent launch: the next kernel (a product on these codes)
// may start streaming its weights at once, and waits for this grid before it
// reads the codes; this grid waits for the previous one before it reads x.
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const uint4 *x, int8_t *q, uint16_t *d_bits,
                                                           int32_t *sumq, int64_t nchunks)
{
    pdl_allow_next_grid();
    pdl_wait_prior_grid();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool ok = c < nchunks;
    const uint4 v = ok ? __ldg(x + c) : make_uint4(0u, 0u, 0u, 0u);
    float dq;
    int s;
    const uint2 codes = q8_1_chunk(v, dq, s);
    if (ok) {
        *reinterpret_cast<uint2 *>(q + 8 * c) = codes;
        if ((c & 3) == 0) {
            d_bits[c >> 2] = __half_as_ushort(__float2half_rn(dq));
            sumq[c >> 2] = s;
        }
    }
}

cudaError_t launch_quantize_q8_1(const void *x, int8_t *q, uint16_t *d_bits, int32_t *sumq, int64_t M, int64_t K,
                                 cudaStream_t s, bool pdl)
{
    const int64_t nchunks = M * (K / 8);
    const int64_t grid = (nchunks + 255) / 256;
    if (grid > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
    return launch_ex(quantize_q8_1_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, pdl,
                     static_cast<const uint4 *>(x), q, d_bits, sumq, nchunks);
}

}  // namespace qmv
