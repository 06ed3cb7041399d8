// qmv_gemv_q4_0_swiglu_f32.cu -- instantiations of the streaming decode kernel
// for the fused gate + up + SwiGLU form over two Q4_0 tables with fp32
// activations (rounded to fp16 while each CTA stages them).
#include "qmv_gemv_q4_0_launch.cuh"

namespace qmv {

cudaError_t launch_gemv_stream_q4_0_swiglu_f32(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                               cudaStream_t s, bool pdl)
{
    return launch_q4_by_m<true, true>(M, p, grid, warps, smem, s, pdl);
}

}  // namespace qmv
