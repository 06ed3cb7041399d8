// qmv_prefill.cu -- Q4_0 prefill GEMM on the 5th-generation tensor cores.
#include "qmv_prefill.h"

namespace qmv {

bool prefill_supported(int64_t, int64_t, int64_t) { return false; }

cudaError_t launch_prefill(const void *, const void *, float *, int64_t, int64_t, int64_t, int, int *,
                           cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace qmv
