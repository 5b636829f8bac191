// Indexer scores on the tcgen05 tensor cores.
//
// [KD] "DeepSeek-V4: optimización de inferencia y RL ...", §Flujo de
// Inferencia step 6 (top-k selection over the compressed attention
// candidates) and §Arquitectura del Sistema (the DSA indexer); [WK] "与 SGLang
// 团队聊 DeepSeek V4", §RL 训练侧 (the attention indexer acts like an MoE
// router).  The library fixes the score of compressed entry j of sequence b as
//     s[b, j] = sum_h w[b, h] * max(0, q[b, h, :] . k[j, :]).
//
// Mapping: the C4 keys are the M = 128 operand (one TMEM lane per key) and
// the sequence's Hi <= 16 indexer heads the N = 16 operand, so one
// tcgen05.mma chain of Di/16 instructions produces the 128 x Hi dot products
// of a tile in TMEM; the ReLU-weighted head sum runs in the epilogue straight
// out of TMEM, one thread per key.  Keys and queries arrive by TMA into
// 128-byte (Di >= 64) or 64-byte (Di = 32) swizzled shared memory, exactly
// the K-major layout the MMA descriptors describe.  Each CTA owns one tile of
// 128 keys of one sequence; several CTAs per SM keep enough TMA loads in
// flight to stream the keys at HBM rate (the kernel is bound by the key
// bytes: 2*Di bytes per entry against 4*Hi*Di flops).
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kTileRows = 128;  // M
constexpr int kQRows = 16;      // N (heads, padded)
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 32;

struct IndexerParams {
  const float* w;  // [B, Hi]
  Spans sp;
  int B, Hi, Di;
  float* scores;
  uint32_t* status;
};

struct TilePieces {
  Spans sp;
  HSA_DEVINL int64_t operator()(int b) const {
    return (sp.count(b) + kTileRows - 1) / kTileRows;
  }
};

__global__ void __launch_bounds__(kThreads) indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                                                          const __grid_constant__ CUtensorMap qmap,
                                                          IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ok;
  __shared__ float s_w[kQRows];

  int seq;
  int64_t piece, npieces;
  if (!locate_piece(p.B, blockIdx.x, TilePieces{p.sp}, &seq, &piece, &npieces)) return;
  const int64_t n = p.sp.count(seq);
  const int64_t row_lo = p.sp.start(seq) + piece * kTileRows;
  const int64_t left = n - piece * kTileRows;
  const int rows = static_cast<int>(left < kTileRows ? left : kTileRows);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb_elems = p.Di >= 64 ? 64 : p.Di;  // elements of one swizzle row
  const int nkb = p.Di / kb_elems;
  const uint32_t a_kb_bytes = kTileRows * kb_elems * 2;
  const uint32_t b_kb_bytes = kQRows * kb_elems * 2;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + nkb * a_kb_bytes;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_tma, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&kmap);
    tc::tma_prefetch_map(&qmap);
    s_ok = 0;
  }
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  if (threadIdx.x < kQRows)
    s_w[threadIdx.x] = threadIdx.x < p.Hi ? p.w[static_cast<int64_t>(seq) * p.Hi + threadIdx.x] : 0.f;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  bool tma_done = true, mma_issued = false;
  if (threadIdx.x == 0) {
    tc::mbar_arrive_expect_tx(&bar_tma, nkb * (a_kb_bytes + b_kb_bytes));
    for (int kb = 0; kb < nkb; ++kb) {
      tc::tma_load_2d(sA + kb * a_kb_bytes, &kmap, kb * kb_elems, static_cast<int32_t>(row_lo),
                      &bar_tma);
      tc::tma_load_2d(sB + kb * b_kb_bytes, &qmap, kb * kb_elems, seq * p.Hi, &bar_tma);
    }
    tma_done = tc::mbar_wait(&bar_tma, 0, p.status);
    if (tma_done) {
      tc::fence_after_sync();
      const tc::Swizzle sw = kb_elems == 64 ? tc::kSwizzle128B : tc::kSwizzle64B;
      const uint32_t sbo = 8 * kb_elems * 2;  // bytes between 8-row groups
      const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, kQRows);
      for (int kb = 0; kb < nkb; ++kb) {
        for (int ks = 0; ks < kb_elems / 16; ++ks) {
          const uint64_t a = tc::smem_desc(tc::smem_u32(sA + kb * a_kb_bytes + ks * 32), 16, sbo, sw);
          const uint64_t b = tc::smem_desc(tc::smem_u32(sB + kb * b_kb_bytes + ks * 32), 16, sbo, sw);
          tc::mma_bf16(tmem, a, b, idesc, (kb | ks) != 0);
        }
      }
      tc::mma_commit(&bar_mma);
      mma_issued = true;
      s_ok = 1;
    }
  }
  __syncthreads();
  bool ok = s_ok != 0;
  if (ok) ok = tc::mbar_wait(&bar_mma, 0, p.status);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc::fence_after_sync();
    uint32_t acc[16];
    tc::tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16), acc);
    tc::tmem_ld_wait();
    const int r = warp * 32 + lane;
    if (r < rows) {
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < kQRows; ++h)
        if (h < p.Hi) s = fmaf(s_w[h], fmaxf(__uint_as_float(acc[h]), 0.f), s);
      p.scores[row_lo + r] = s;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    // after a timeout, give in-flight copies and MMAs a second bounded chance
    if (!tma_done) tc::mbar_wait(&bar_tma, 0, p.status);
    if (mma_issued && !ok) tc::mbar_wait(&bar_mma, 0, p.status);
  }
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t indexer_smem_bytes(int Di) { return static_cast<size_t>(Di) * 2 * (kTileRows + kQRows) + 1024; }

cudaError_t launch_indexer(const void* iq, const float* w, const void* keys, Spans sp, int B, int Hi,
                           int Di, int64_t total_rows, float* scores, uint32_t* status,
                           cudaStream_t stream) {
  if (total_rows == 0) return cudaSuccess;
  const int kb_elems = Di >= 64 ? 64 : Di;
  const CUtensorMapSwizzle sw = kb_elems == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap kmap, qmap;
  cudaError_t e = make_tmap_2d_bf16(&kmap, keys, Di, total_rows, kb_elems, kTileRows, sw);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&qmap, iq, Di, static_cast<int64_t>(B) * Hi, kb_elems, kQRows, sw);
  if (e != cudaSuccess) return e;
  const size_t smem = indexer_smem_bytes(Di);
  e = cudaFuncSetAttribute(indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(indexer_smem_bytes(128)));
  if (e != cudaSuccess) return e;
  const int64_t grid = (total_rows + kTileRows - 1) / kTileRows + B;
  IndexerParams p{w, sp, B, Hi, Di, scores, status};
  indexer_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(kmap, qmap, p);
  return cudaGetLastError();
}

}  // namespace hsa
