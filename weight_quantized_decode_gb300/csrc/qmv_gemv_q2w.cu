// qmv_gemv_q2w.cu -- instantiations of the streaming decode kernel for the
// plain 2-bit format (codes from -2 to 1 with an fp16 scale for every 32 weights).
#include "qmv_gemv.cuh"
#include "qmv_launch.h"

namespace qmv {

template <int M, int MAXT>
static cudaError_t launch_q2w_t(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    auto kernel = qmv_stream_kernel<kQ2W, M, MAXT, false>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void *>(kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_ex(kernel, dim3(grid), dim3(warps * 32), smem, s, pdl, p);
}

// Up to 8 warps per CTA for every token count; up to 16 for one or two tokens.
template <int M>
static cudaError_t launch_q2w_one(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    if (p.expert_idx || p.W2 || p.xf) return cudaErrorInvalidValue;
    if (warps <= 8) return launch_q2w_t<M, 256>(p, grid, warps, smem, s, pdl);
    if constexpr (M <= 2) {
        if (warps <= 16) return launch_q2w_t<M, 512>(p, grid, warps, smem, s, pdl);
    } else {
        if (warps <= 12) return launch_q2w_t<M, 384>(p, grid, warps, smem, s, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemv_stream_q2w(int M, const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s,
                                   bool pdl)
{
    switch (M) {
    case 1: return launch_q2w_one<1>(p, grid, warps, smem, s, pdl);
    case 2: return launch_q2w_one<2>(p, grid, warps, smem, s, pdl);
    case 3: return launch_q2w_one<3>(p, grid, warps, smem, s, pdl);
    case 4: return launch_q2w_one<4>(p, grid, warps, smem, s, pdl);
    case 5: return launch_q2w_one<5>(p, grid, warps, smem, s, pdl);
    case 6: return launch_q2w_one<6>(p, grid, warps, smem, s, pdl);
    case 7: return launch_q2w_one<7>(p, grid, warps, smem, s, pdl);
    case 8: return launch_q2w_one<8>(p, grid, warps, smem, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
