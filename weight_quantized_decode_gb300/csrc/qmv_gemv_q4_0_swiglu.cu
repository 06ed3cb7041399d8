// qmv_gemv_q4_0_swiglu.cu -- instantiations of the streaming decode kernel for
// the fused gate + up + SwiGLU form over two Q4_0 tables with fp16 activations
// (units of their own so the build compiles them beside the plain forms).
#include "qmv_gemv_q4_0_launch.cuh"

namespace qmv {

cudaError_t launch_gemv_stream_q4_0_swiglu(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                           cudaStream_t s, bool pdl)
{
    if (p.xf) return launch_gemv_stream_q4_0_swiglu_f32(M, p, grid, warps, smem, s, pdl);
    return launch_q4_by_m<false, true>(M, p, grid, warps, smem, s, pdl);
}

}  // namespace qmv
