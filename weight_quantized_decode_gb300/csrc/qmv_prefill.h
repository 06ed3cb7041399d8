// qmv_prefill.h -- host hooks of the tensor-core prefill kernel (internal).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmv {

// True when the tensor-core kernel handles this shape.
bool prefill_supported(int64_t N, int64_t K, int64_t M);

cudaError_t launch_prefill(const void *W, const void *x, float *y, int64_t N, int64_t K, int64_t M, int sms,
                           int *status, cudaStream_t s, bool pdl);

}  // namespace qmv
