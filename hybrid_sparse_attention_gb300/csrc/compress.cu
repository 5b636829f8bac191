// Flash Compressor: one pass over each complete block of r tokens.
//
// [KD] "DeepSeek-V4: optimización de inferencia y RL ...", §Arquitectura del
// Sistema: the 5-stage compression chain is fused into a single on-chip pass
// to cut HBM round trips.  [WK] "与 SGLang 团队聊 DeepSeek V4", §推理侧优化,
// Kernel fusion: read -> add -> softmax -> dot -> write.
//
// out[s, n, ch] = sum_i softmax_i(z[s, n*r+i, ch] + b[i, ch]) * kv[s, n*r+i, ch]
//
// Layout of the work.  Blocks of r <= 16 tokens (compress_stream_kernel, the
// plain transform, C <= 768): the input of every sequence is one contiguous
// run of rows, so a producer warp copies it, unchanged, into a shared-memory
// ring with bulk copies (a stage holds floor(16 / r) whole blocks: at most 16
// rows of kv and 16 of z), and eight warps evaluate the gated softmax out of
// shared memory, a thread per 16-byte chunk (8 channels) of one block.  The
// ring keeps the bytes in flight independent of the registers a thread
// needs: the per-thread layout below, every thread loading its block's rows
// into registers in groups of 4, held one 256-thread CTA per SM (213
// registers a thread), which kept too few short blocks in flight (r = 4:
// 1.59 ms against 0.90 ms over 32 x 65,536 x 512).
//
// Longer blocks (and the overlap variant, and C > 768): one thread owns one
// chunk of one block and streams the block's r rows of kv and z through
// registers, one row at a time (few registers: two CTAs per SM keep enough
// loads in flight).  Consecutive
// threads own consecutive chunks of the same row (a warp reads 512 contiguous
// bytes per load).  The staged layout with 16-row slices of long blocks cut
// across lanes was slower there (r = 128: 1.60 ms against 1.07 ms).
//
// Each input byte crosses HBM once and the only write is the compressed row.
// The softmax is evaluated online in groups of 4 rows (one max and one rescale
// per group; compress_core.cuh), or in two passes over a staged block.
//
#include "common.cuh"
#include "compress_core.cuh"
#include "internal.h"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kSliceRows = 16;       // rows of kv (and of z) per ring stage
constexpr int kStreamStages = 2;     // ring stages per CTA
constexpr int kStreamCtasPerSm = 2;
constexpr int kStreamWarps = 8;      // softmax warps; one more warp issues the copies
constexpr int kStreamThreads = 32 * (kStreamWarps + 1);
constexpr int64_t kStreamMaxC = 768;

struct StreamParams {
  const uint8_t* kv;
  const uint8_t* z;
  const float* b;
  int64_t T, nblk, nk;  // tokens per sequence, blocks per sequence, blocks in all
  int64_t units;        // stages (of bps blocks each)
  int C, chunks, r;
  int bps;              // whole blocks per stage
  void* out;
};

// Rows 0..n-1 of one chunk, read from a shared-memory stage (rows(i, &kv,
// &z)), into the partial p: the maximum logit over the n rows, one rescale
// of p, then the weighted sum, reading each row twice (shared memory is cheap
// to re-read; registers are what bound the threads per SM).  bias(i) points
// at row i's 8 fp32 biases (L1-resident: r <= 16 rows of them).  With p fresh
// and the whole block in the n rows this is the two-pass softmax: one
// exponential per (row, channel).
template <typename RowFn, typename BiasFn>
HSA_DEVINL void partial_rows_staged(RowFn rows, int n, BiasFn bias, GatePartial& p) {
  float gm[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) gm[c] = -INFINITY;
  for (int i = 0; i < n; ++i) {
    const uint4 *kp, *zp;
    rows(i, &kp, &zp);
    float x[8];
    bf16x8_to_f32(*zp, x);
    const float4* bp = bias(i);
    const float4 b0 = __ldg(bp), b1 = __ldg(bp + 1);
    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) gm[c] = fmaxf(gm[c], x[c] + bb[c]);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float mn = fmaxf(p.m[c], gm[c]);
    const float alpha = __expf(p.m[c] - mn);  // 0 while p is empty (m = -inf)
    p.l[c] *= alpha;
    p.acc[c] *= alpha;
    p.m[c] = mn;
  }
  for (int i = 0; i < n; ++i) {
    const uint4 *kp, *zp;
    rows(i, &kp, &zp);
    float x[8], v[8];
    bf16x8_to_f32(*zp, x);
    bf16x8_to_f32(*kp, v);
    const float4* bp = bias(i);
    const float4 b0 = __ldg(bp), b1 = __ldg(bp + 1);
    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float e = __expf(x[c] + bb[c] - p.m[c]);
      p.l[c] += e;
      p.acc[c] = fmaf(e, v[c], p.acc[c]);
    }
  }
}

template <bool kBf16Out>
HSA_DEVINL void store_row_chunk(void* out, int64_t at, const float (&o)[8]) {
  if (kBf16Out) {
    reinterpret_cast<uint4*>(out)[at] = f32x8_to_bf16(o);
  } else {
    float4* dst = reinterpret_cast<float4*>(out) + at * 2;
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
}

template <bool kBf16Out>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm) compress_stream_kernel(StreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kStreamStages], empty[kStreamStages];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const uint32_t row_bytes = static_cast<uint32_t>(p.C) * 2;
  const uint32_t half = kSliceRows * row_bytes;  // the stage's kv rows; its z rows follow
  const uint32_t stage_bytes = 2 * half;
  // a contiguous range of stages
  const int64_t u0 = p.units * blockIdx.x / gridDim.x, u1 = p.units * (blockIdx.x + 1) / gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kStreamWarps);
    }
    tc::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kStreamWarps) {
    // ------------------------------------------------------------ copies
    if (lane == 0) {
      int64_t i = 0;  // stages issued
      for (int64_t u = u0; u < u1; ++u, ++i) {
        const int s = static_cast<int>(i % kStreamStages);
        if (i >= kStreamStages &&
            !tc::mbar_wait(&empty[s], static_cast<uint32_t>((i / kStreamStages) & 1) ^ 1u, nullptr))
          break;
        uint8_t* st = ring + s * stage_bytes;
        const int64_t k0 = u * p.bps;
        const int nb = static_cast<int>(p.nk - k0 < p.bps ? p.nk - k0 : p.bps);
        const uint32_t bytes = static_cast<uint32_t>(p.r) * row_bytes;
        tc::mbar_arrive_expect_tx(&full[s], 2u * nb * bytes);
        int64_t sq = k0 / p.nblk, n = k0 - sq * p.nblk;
        for (int j = 0; j < nb; ++j) {  // (a stage may hold the end of one sequence and the start of the next)
          const int64_t row = sq * p.T + n * p.r;
          tc::bulk_load(st + j * bytes, p.kv + row * row_bytes, bytes, &full[s]);
          tc::bulk_load(st + half + j * bytes, p.z + row * row_bytes, bytes, &full[s]);
          if (++n == p.nblk) {
            n = 0;
            ++sq;
          }
        }
      }
      // every issued copy lands before the CTA exits (only the last stages
      // can be outstanding: after a wait that ran out the softmax warps may
      // not have consumed them)
      for (int64_t j = i > kStreamStages ? i - kStreamStages : 0; j < i; ++j)
        tc::mbar_wait(&full[j % kStreamStages], static_cast<uint32_t>((j / kStreamStages) & 1), nullptr);
    }
    return;
  }
  // -------------------------------------------------------------- softmax
  const int t = threadIdx.x;
  auto bias_at = [&](int row, int c8) {
    return reinterpret_cast<const float4*>(p.b + static_cast<int64_t>(row) * p.C + c8 * 8);
  };
  int64_t i = 0;
  for (int64_t u = u0; u < u1; ++u, ++i) {
    const int s = static_cast<int>(i % kStreamStages);
    if (!__all_sync(0xffffffffu, tc::mbar_wait(&full[s], static_cast<uint32_t>((i / kStreamStages) & 1), nullptr)))
      return;
    const uint8_t* st = ring + s * stage_bytes;
    const int64_t k0 = u * p.bps;
    const int nb = static_cast<int>(p.nk - k0 < p.bps ? p.nk - k0 : p.bps);
    const int items = nb * p.chunks;
    for (int it = t; it < items; it += kStreamWarps * 32) {
      const int j = it / p.chunks, c8 = it - j * p.chunks;
      const uint4* kvs = reinterpret_cast<const uint4*>(st + j * p.r * row_bytes) + c8;
      const uint4* zs = reinterpret_cast<const uint4*>(st + half + j * p.r * row_bytes) + c8;
      GatePartial part;
      partial_init(part);
      auto rows = [&](int r, const uint4** kp, const uint4** zp) {
        *kp = kvs + r * p.chunks;
        *zp = zs + r * p.chunks;
      };
      auto bias = [&](int r) { return bias_at(r, c8); };
      // the C4 ratio with its row loops unrolled (every row's loads issued
      // together): 1.03 -> 0.90 ms over 32 x 65,536 x 512
      if (p.r == 4)
        partial_rows_staged(rows, 4, bias, part);
      else
        partial_rows_staged(rows, p.r, bias, part);
      float o[8];
      partial_result(part, o);
      store_row_chunk<kBf16Out>(p.out, (k0 + j) * p.chunks + c8, o);
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[s]);
  }
}

template <bool kBf16Out, bool kOverlap>
__global__ void __launch_bounds__(256, 2) compress_kernel(const uint4* __restrict__ kv,
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
    // one row at a time: ~70 registers, two CTAs per SM (groups of 4 rows took
    // 213 registers and one CTA per SM: r = 128 1.07 -> 0.91 ms)
    partial_rows<kOverlap, 1>(kv + first, z + first, chunks, 0, i1 - i0, bias, part);
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
  if (!overlap && C <= kStreamMaxC && r <= kSliceRows) {
    StreamParams p{};
    p.kv = static_cast<const uint8_t*>(kv);
    p.z = static_cast<const uint8_t*>(z);
    p.b = b;
    p.T = T;
    p.nblk = T / r;
    p.nk = S * p.nblk;
    p.C = static_cast<int>(C);
    p.chunks = static_cast<int>(C / 8);
    p.r = static_cast<int>(r);
    p.out = out;
    p.bps = kSliceRows / p.r;
    p.units = (p.nk + p.bps - 1) / p.bps;
    const size_t smem = static_cast<size_t>(kStreamStages) * 2 * kSliceRows * C * 2 + 128;
    auto kernel = out_dtype == HSA_BF16 ? compress_stream_kernel<true> : compress_stream_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t nres = static_cast<int64_t>(kStreamCtasPerSm) * device_sms();
    const int grid = static_cast<int>(p.units < nres ? p.units : nres);
    kernel<<<grid, kStreamThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
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
