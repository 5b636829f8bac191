// Per-row E4M3 quantization of fp32 rows: the storage format of the E4M3
// indexer-key pool (one binary32 scale per row, 8-bit codes).
//
// The pages speak of FP8 rollout and of a 1M-token KV cache held under 10 GB
// ([LH] "DeepSeek-V4: SGLang và Miles ...", §Hỗ trợ Học tăng cường; [WK]
// "与 SGLang 团队聊 DeepSeek V4", §DeepSeek V4 的新架构) without fixing a
// format; the library's reading: amax = max |x|, scale = amax / 448,
// code = e4m3(x * (448 / amax)) rounded to nearest even and saturated at
// +-448 (the hardware conversion), every step rounded to binary32; a row of
// zeros gets scale 0 and zero codes.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

__global__ void __launch_bounds__(32 * kRowsPerBlock) quantize_e4m3_kernel(const float4* __restrict__ x,
                                                                          int64_t rows, int C4,
                                                                          uint32_t* __restrict__ codes,
                                                                          float* __restrict__ scales) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4* xr = x + row * C4;
  float am = 0.f;
  for (int c = lane; c < C4; c += 32) {
    const float4 v = __ldg(xr + c);
    am = fmaxf(am, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const float inv = am > 0.f ? __fdiv_rn(448.f, am) : 0.f;
  for (int c = lane; c < C4; c += 32) {
    const float4 v = __ldg(xr + c);
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(v.z, inv), __fmul_rn(v.w, inv)), __NV_SATFINITE, __NV_E4M3);
    codes[row * C4 + c] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  if (lane == 0) scales[row] = __fdiv_rn(am, 448.f);
}

}  // namespace

cudaError_t launch_quantize_e4m3(const float* x, int64_t rows, int64_t C, uint8_t* codes,
                                 float* scales, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  return launch_k(quantize_e4m3_kernel, dim3(static_cast<unsigned>(blocks)), dim3(32 * kRowsPerBlock), 0,
                  stream, false, reinterpret_cast<const float4*>(x), rows, static_cast<int>(C / 4),
                  reinterpret_cast<uint32_t*>(codes), scales);
}

}  // namespace hsa
