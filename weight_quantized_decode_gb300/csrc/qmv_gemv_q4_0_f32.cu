// qmv_gemv_q4_0_f32.cu -- instantiations of the streaming decode kernel for
// Q4_0 with fp32 activations (plain form).  The activations
// are rounded to fp16 while each CTA stages them into shared memory, so no
// separate conversion pass runs before the product.
#include "qmv_gemv_q4_0_launch.cuh"

namespace qmv {

cudaError_t launch_gemv_stream_q4_0_f32(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                        cudaStream_t s, bool pdl)
{
    if (p.expert_idx) return cudaErrorInvalidValue;
    return launch_q4_by_m<true, false>(M, p, grid, warps, smem, s, pdl);
}

}  // namespace qmv
