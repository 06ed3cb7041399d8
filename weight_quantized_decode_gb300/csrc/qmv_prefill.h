// qmv_prefill.h -- host hooks of the tensor-core prefill kernel (internal).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qmv_prefill_plan.h"

namespace qmv {

// The tensor-core kernel's plan for this call on a device of `sms` SMs, with
// the ring depths forced through QMV_PREFILL_RING applied; ok is false when
// that kernel does not take the shape (or the tensor-map encoder is missing).
// fmt: kPfQ4_0 or kPfQ8_0; splitk as in plan_prefill (0: none, -1: fill the
// GPU with CTAs along K where 16-token tiles leave SMs idle).
PrefillPlan prefill_plan(int64_t N, int64_t K, int64_t M, int sms, int fmt = kPfQ4_0, int splitk = 0);

// test_skip_copy: failure-detection tests only (one tile of CTA (0, 0) is never
// requested, so its bounded waits run out); false in every normal call.
cudaError_t launch_prefill(const PrefillPlan &pl, const void *W, const void *x, float *y, int64_t N, int64_t K,
                           int64_t M, int *status, cudaStream_t s, bool pdl, bool test_skip_copy);

}  // namespace qmv
