// qmv_gemv_q4_0_launch.cuh -- launch shapes of the Q4_0 streaming decode
// kernel, shared by the translation unit for fp16 activations and the one for
// fp32 activations (XF32: rounded to fp16 as they are staged).
#pragma once

#include "qmv_gemv.cuh"
#include "qmv_launch.h"

namespace qmv {

template <int M, int MAXT, bool MOE, bool SWIGLU, bool XF32>
static cudaError_t launch_q4_t(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    auto kernel = qmv_stream_kernel<kQ4_0, M, MAXT, MOE, SWIGLU, XF32>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void *>(kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_ex(kernel, dim3(grid), dim3(warps * 32), smem, s, pdl, p);
}

// Up to 8 warps per CTA for every token count; up to 16 (at most 128
// registers a thread) for one or two tokens, up to 12 (at most 168) for three
// or more: with eight tokens the staged activations leave room for one CTA per
// SM, and its warps are all the latency hiding there is.
// SW selects the instantiations of one translation unit: the fused SwiGLU
// form, or the plain and multi-expert forms.
template <int M, bool XF32, bool SW>
static cudaError_t launch_q4_one(const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s, bool pdl)
{
    if ((p.W2 != nullptr) != SW) return cudaErrorInvalidValue;
    if constexpr (!SW) {
        if (p.expert_idx) {
            if constexpr (M == 1 && !XF32) {
                if (warps <= 8) return launch_q4_t<1, 256, true, false, false>(p, grid, warps, smem, s, pdl);
                if (warps <= 16) return launch_q4_t<1, 512, true, false, false>(p, grid, warps, smem, s, pdl);
            }
            return cudaErrorInvalidConfiguration;
        }
    }
    if (warps <= 8) return launch_q4_t<M, 256, false, SW, XF32>(p, grid, warps, smem, s, pdl);
    if constexpr (M <= 2) {
        if (warps <= 16) return launch_q4_t<M, 512, false, SW, XF32>(p, grid, warps, smem, s, pdl);
    } else {
        if (warps <= 12) return launch_q4_t<M, 384, false, SW, XF32>(p, grid, warps, smem, s, pdl);
    }
    return cudaErrorInvalidConfiguration;
}

template <bool XF32, bool SW>
static cudaError_t launch_q4_by_m(int M, const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s,
                                  bool pdl)
{
    switch (M) {
    case 1: return launch_q4_one<1, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 2: return launch_q4_one<2, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 3: return launch_q4_one<3, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 4: return launch_q4_one<4, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 5: return launch_q4_one<5, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 6: return launch_q4_one<6, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 7: return launch_q4_one<7, XF32, SW>(p, grid, warps, smem, s, pdl);
    case 8: return launch_q4_one<8, XF32, SW>(p, grid, warps, smem, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
