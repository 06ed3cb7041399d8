// qmv_launch.h -- host-side launch hooks shared by the translation units of
// the library (internal; the public interface is include/qmv.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qmv {

struct GemvParams;

// Streaming decode kernel for one format and token count M (1..8).
cudaError_t launch_gemv_stream_q4_0(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                    cudaStream_t s, bool pdl);
// Q4_0 fused gate + up + SwiGLU (p.W2 set; fp16, or fp32 activations with p.xf).
cudaError_t launch_gemv_stream_q4_0_swiglu(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                           cudaStream_t s, bool pdl);
cudaError_t launch_gemv_stream_q4_0_swiglu_f32(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                               cudaStream_t s, bool pdl);
// Q4_0 with fp32 activations (plain form; p.xf set).
cudaError_t launch_gemv_stream_q4_0_f32(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                        cudaStream_t s, bool pdl);
// Q4_0 against Q8_1-quantised activations (plain form only; p.xq8 set).
cudaError_t launch_gemv_stream_q4_0_q8_1(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                         cudaStream_t s, bool pdl);
// Q8_0 against Q8_1-quantised activations (plain form only; p.xq8 set).
cudaError_t launch_gemv_stream_q8_0_q8_1(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                         cudaStream_t s, bool pdl);
// Q8_1 quantisation of fp16 activations [M][K] (K % 32 == 0, x 16-byte aligned).
cudaError_t launch_quantize_q8_1(const void *x, int8_t *q, uint16_t *d_bits, int32_t *sumq, int64_t M, int64_t K,
                                 cudaStream_t s, bool pdl);
// Plain 2-bit (plain form only).
cudaError_t launch_gemv_stream_q2w(int M, const GemvParams &p, int grid, int warps, size_t smem, cudaStream_t s,
                                   bool pdl);
cudaError_t launch_gemv_stream_q8_0(int M, const GemvParams &p, int grid, int warps, size_t smem,
                                    cudaStream_t s, bool pdl);
// Read-only bandwidth probe over `bytes` (a multiple of 256) of device memory;
// *out (device) receives an XOR checksum of the bytes it consumed.
cudaError_t launch_read_probe(const void *buf, int64_t bytes, uint32_t *out, int *status, int sms, cudaStream_t s);
// Generic kernel (any K % 32 == 0, activations read from global memory).
cudaError_t launch_gemv_generic(int fmt, const GemvParams &p, int M, int grid, cudaStream_t s, bool pdl);

// Opt a kernel into more than 48 KB of dynamic shared memory on the current
// device (once per device).
cudaError_t ensure_smem_optin(const void *func, size_t smem);

// Launch `kernel` with optional programmatic dependent launch.
template <typename Kernel, typename... Args>
cudaError_t launch_ex(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_ex with thread-block clusters of cluster.x * cluster.y * cluster.z
// CTAs (all ones = none).
template <typename Kernel, typename... Args>
cudaError_t launch_ex_cluster_dims(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                   dim3 cluster, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster.x * cluster.y * cluster.z > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster.x;
        attr[n].val.clusterDim.y = cluster.y;
        attr[n].val.clusterDim.z = cluster.z;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_ex with thread-block clusters of `cluster` CTAs along x (1 = none).
template <typename Kernel, typename... Args>
cudaError_t launch_ex_cluster(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                              int cluster, Args... args)
{
    return launch_ex_cluster_dims(kernel, grid, block, smem, s, pdl, dim3(static_cast<unsigned>(cluster), 1, 1),
                                  args...);
}

}  // namespace qmv
