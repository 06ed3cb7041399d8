// qmv_gemv_q4_0.cu -- instantiations of the streaming decode kernel for Q4_0
// with fp16 activations (plain and multi-expert forms).
#include "qmv_gemv_q4_0_launch.cuh"

namespace qmv {

cudaError_t launch_gemv_stream_q4_0(int M, const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s,
                                    bool pdl)
{
    return launch_q4_by_m<false, false>(M, p, grid, warps, smem, s, pdl);
}

}  // namespace qmv
