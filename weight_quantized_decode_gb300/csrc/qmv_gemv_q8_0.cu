// qmv_gemv_q8_0.cu -- instantiations of the streaming decode kernel for Q8_0.
#include "qmv_gemv.cuh"
#include "qmv_launch.h"

namespace qmv {

template <int M, int MAXT, bool MOE>
static cudaError_t launch_t(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    auto kernel = qmv_stream_kernel<kQ8_0, M, MAXT, MOE>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void *>(kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_ex(kernel, dim3(grid), dim3(warps * 32), smem, s, pdl, p);
}

// Up to 8 warps per CTA for every token count; up to 16 (at most 128
// registers a thread) for one or two tokens.
template <int M>
static cudaError_t launch_one(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    if (p.expert_idx) {
        if constexpr (M == 1) {
            if (warps <= 8) return launch_t<1, 256, true>(p, grid, warps, smem, s, pdl);
            if (warps <= 16) return launch_t<1, 512, true>(p, grid, warps, smem, s, pdl);
        }
        return cudaErrorInvalidConfiguration;
    }
    if (warps <= 8) return launch_t<M, 256, false>(p, grid, warps, smem, s, pdl);
    if constexpr (M <= 2) {
        if (warps <= 16) return launch_t<M, 512, false>(p, grid, warps, smem, s, pdl);
    } else {
        if (warps <= 12) return launch_t<M, 384, false>(p, grid, warps, smem, s, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemv_stream_q8_0(int M, const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s,
                                  bool pdl)
{
    switch (M) {
    case 1: return launch_one<1>(p, grid, warps, smem, s, pdl);
    case 2: return launch_one<2>(p, grid, warps, smem, s, pdl);
    case 3: return launch_one<3>(p, grid, warps, smem, s, pdl);
    case 4: return launch_one<4>(p, grid, warps, smem, s, pdl);
    case 5: return launch_one<5>(p, grid, warps, smem, s, pdl);
    case 6: return launch_one<6>(p, grid, warps, smem, s, pdl);
    case 7: return launch_one<7>(p, grid, warps, smem, s, pdl);
    case 8: return launch_one<8>(p, grid, warps, smem, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
