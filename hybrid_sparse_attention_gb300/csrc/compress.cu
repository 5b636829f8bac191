// Flash Compressor: one pass over each complete block of r tokens.
//
// [KD] "DeepSeek-V4: optimización de inferencia y RL ...", §Arquitectura del
// Sistema: the 5-stage compression chain is fused into a single on-chip pass
// to cut HBM round trips.  [WK] "与 SGLang 团队聊 DeepSeek V4", §推理侧优化,
// Kernel fusion: read -> add -> softmax -> dot -> write.
//
// out[s, n, ch] = sum_i softmax_i(z[s, n*r+i, ch] + b[i, ch]) * kv[s, n*r+i, ch]
//
// Layout of the work: one thread owns one 16-byte chunk (8 channels) of one
// block and streams the block's r rows of kv and z through registers, so each
// input byte crosses HBM exactly once and the only write is the compressed
// row.  Consecutive threads own consecutive chunks of the same row (a warp
// reads 512 contiguous bytes per load).  The softmax is evaluated online in
// groups of 4 rows: one max per group, one rescale per group (the shared
// arithmetic lives in compress_core.cuh).
//
// C4 overlap transform ([WK] §RL 训练侧 ①: neighbouring compressed entries
// share tokens; the library's reading): entry n runs over the 2r-token window
// of blocks n-1 and n with a bias per window position (entry 0 over block 0
// alone), the same one pass per entry; the rows two windows share are read
// twice, the second time from L2.
#include "common.cuh"
#include "compress_core.cuh"
#include "internal.h"

namespace hsa {
namespace {

template <bool kBf16Out, bool kOverlap>
__global__ void __launch_bounds__(256) compress_kernel(const uint4* __restrict__ kv,
                                                       const uint4* __restrict__ z,
                                                       const float* __restrict__ b, int64_t S,
                                                       int64_t T, int64_t C, int r,
                                                       void* __restrict__ out) {
  const int64_t chunks = C / 8;
  const int64_t nblk = T / r;
  const int64_t total = S * nblk * chunks;
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t c8 = w % chunks;
    const int64_t sn = w / chunks;  // s * nblk + n
    const int64_t s = sn / nblk, n = sn - s * nblk;
    // window positions [i0, i1) (the overlap window starts a block early)
    const int i0 = kOverlap && n == 0 ? r : 0, i1 = kOverlap ? 2 * r : r;
    const int64_t row0 = n * r - (kOverlap ? r : 0) + i0;  // the first row read
    const int64_t first = (s * T + row0) * chunks + c8;
    auto bias = [&](int i, float4* lo, float4* hi) {
      const float4* p = reinterpret_cast<const float4*>(b + (i + i0) * C + c8 * 8);
      *lo = __ldg(p);
      *hi = __ldg(p + 1);
    };
    GatePartial part;
    partial_init(part);
    partial_rows<kOverlap>(kv + first, z + first, chunks, 0, i1 - i0, bias, part);
    float o[8];
    partial_result(part, o);
    if (kBf16Out) {
      reinterpret_cast<uint4*>(out)[sn * chunks + c8] = f32x8_to_bf16(o);
    } else {
      float4* dst = reinterpret_cast<float4*>(out) + (sn * chunks + c8) * 2;
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace

cudaError_t launch_compress(const void* kv, const void* z, const float* b, int64_t S, int64_t T,
                            int64_t C, int64_t r, void* out, int out_dtype, cudaStream_t stream,
                            bool overlap) {
  const int64_t total = S * (T / r) * (C / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = static_cast<int>(want < device_sms() * 16 ? want : device_sms() * 16);
  auto kernel = out_dtype == HSA_BF16 ? (overlap ? compress_kernel<true, true> : compress_kernel<true, false>)
                                      : (overlap ? compress_kernel<false, true> : compress_kernel<false, false>);
  kernel<<<grid, threads, 0, stream>>>(static_cast<const uint4*>(kv), static_cast<const uint4*>(z),
                                       b, S, T, C, static_cast<int>(r), out);
  return cudaGetLastError();
}

}  // namespace hsa
