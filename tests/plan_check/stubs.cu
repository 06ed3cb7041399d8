// stubs.cu -- the launch functions the planner's translation unit refers to,
// as no-ops: plan_check.cu only plans, it never launches.
#include "../../weight_quantized_decode_gb300/csrc/qmv_gemv.cuh"
#include "../../weight_quantized_decode_gb300/csrc/qmv_launch.h"
#include "../../weight_quantized_decode_gb300/csrc/qmv_prefill.h"

namespace qmv {

#define QMV_STUB_GEMV(name) \
    cudaError_t name(int, const GemvParams &, int, int, size_t, cudaStream_t, bool) { return cudaSuccess; }
QMV_STUB_GEMV(launch_gemv_stream_q4_0)
QMV_STUB_GEMV(launch_gemv_stream_q8_0)
QMV_STUB_GEMV(launch_gemv_stream_q4_0_f32)
QMV_STUB_GEMV(launch_gemv_stream_q2w)
QMV_STUB_GEMV(launch_gemv_stream_q4_0_swiglu)
QMV_STUB_GEMV(launch_gemv_stream_q4_0_swiglu_f32)
QMV_STUB_GEMV(launch_gemv_stream_q4_0_q8_1)
QMV_STUB_GEMV(launch_gemv_stream_q8_0_q8_1)
#undef QMV_STUB_GEMV

cudaError_t launch_quantize_q8_1(const void *, int8_t *, uint16_t *, int32_t *, int64_t, int64_t, cudaStream_t, bool)
{
    return cudaSuccess;
}

cudaError_t launch_read_probe(const void *, int64_t, uint32_t *, int *, int, cudaStream_t) { return cudaSuccess; }

PrefillPlan prefill_plan(int64_t, int64_t, int64_t, int, int, int) { return PrefillPlan{}; }

cudaError_t launch_prefill(const PrefillPlan &, const void *, const void *, float *, int64_t, int64_t, int64_t, int *,
                           cudaStream_t, bool, bool)
{
    return cudaSuccess;
}

}  // namespace qmv
