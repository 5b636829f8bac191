// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hsa.h"

#if defined(__CUDACC__)
#define HSA_HOST_DEVICE __host__ __device__ inline
#else
#define HSA_HOST_DEVICE inline
#endif

namespace hsa {

struct Spans;

// Streaming multiprocessors of the current device (cached per device).
int device_sms();

cudaError_t launch_compress(const void* kv, const void* z, const float* b, int64_t S, int64_t T,
                            int64_t C, int64_t r, void* out, int out_dtype, cudaStream_t stream);

size_t topk_workspace_bytes(int64_t B, int64_t total_rows, int64_t k);
cudaError_t launch_topk(const float* scores, Spans sp, int B, int64_t total_rows, int k,
                        int32_t* idx, float* vals, void* ws, cudaStream_t stream);

}  // namespace hsa
