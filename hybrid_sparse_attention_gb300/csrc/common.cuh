// Device helpers shared by the CUDA kernels of the library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hsa.h"
#include "internal.h"

#define HSA_DEVINL __device__ __forceinline__

namespace hsa {

constexpr size_t kWsHeader = 256;  // workspace bytes reserved for the status word

HSA_DEVINL void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Programmatic dependent launch.  pdl_trigger lets the next kernel of the
// stream be scheduled before this one ends; pdl_wait blocks until the previous
// kernel has completed and its writes are visible (a no-op when this kernel
// was launched without the programmatic-serialization attribute).  Kernels
// trigger only after their own wait has returned, so when a kernel starts,
// every kernel older than its immediate predecessor has completed: it may read
// their outputs at once and must wait only before reading its predecessor's.
HSA_DEVINL void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
HSA_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- thread-block clusters (distributed shared memory)

HSA_DEVINL uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Barrier over every thread of the cluster; orders memory at cluster scope.
HSA_DEVINL void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Address of the same shared variable in the cluster's CTA `rank`.
HSA_DEVINL uint32_t map_rank(const void* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

HSA_DEVINL uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

HSA_DEVINL uint64_t ld_cluster_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

HSA_DEVINL void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

HSA_DEVINL float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

HSA_DEVINL void st_cluster_f32x4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Unpack 8 bf16 (one 16-byte chunk) to fp32.
HSA_DEVINL void bf16x8_to_f32(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

HSA_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

HSA_DEVINL uint4 f32x8_to_bf16(const float f[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

HSA_DEVINL uint4 ld_stream_u4(const uint4* p) { return __ldcs(p); }

// Order-preserving key of an fp32 score (its bits): larger key <=> larger
// value; -0.0 is first folded onto +0.0 so the two compare equal.  Shared by
// the top-k and by the indexer, which histograms the keys of the scores it
// writes for the top-k.
HSA_DEVINL uint32_t order_key(uint32_t u) {
  if (u == 0x80000000u) u = 0u;  // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The layer's indexer -> top-k histogram: per sequence, counts of the top
// kRowHistBits bits of every score's order key.
constexpr int kRowHistBits = 13;
constexpr int kRowHistBins = 1 << kRowHistBits;
constexpr int kRowHistShift = 32 - kRowHistBits;

// Rows of a ragged sequence set.  Sequence b starts at offsets[b]; its row
// count is offsets[b+1] - offsets[b] when seq_len is null, otherwise
// (seq_len[b] + add) / ratio (the live prefix of a capacity-laid-out pool).
// `limit` is the number of rows of the underlying buffer: a sequence whose
// offsets are not monotone, reach past it, or whose live count exceeds its
// capacity is invalid, and kernels treat it as empty and flag it.
struct Spans {
  const int64_t* offsets;
  const int32_t* seq_len;
  int32_t add;
  int32_t ratio;
  int64_t limit;
  // Rows of T query tokens per sequence (multi-token queries): row r is token
  // r % T of sequence r / T, whose live count is (seq_len + add + r % T) /
  // ratio; start(r) adds (r % T) * tstride (per-token score arrays, tstride
  // apart), pool_start(r) is the sequence's first pool row.
  int32_t T = 1;
  int64_t tstride = 0;
  HSA_DEVINL int seq(int r) const { return T == 1 ? r : r / T; }
  HSA_DEVINL int tok(int r) const { return T == 1 ? 0 : r % T; }
  HSA_DEVINL int64_t pool_start(int r) const { return offsets[seq(r)]; }
  HSA_DEVINL int64_t start(int r) const { return offsets[seq(r)] + tok(r) * tstride; }
  HSA_DEVINL int64_t raw_count(int r) const {
    const int b = seq(r);
    if (!seq_len) return offsets[b + 1] - offsets[b];
    const int64_t n = (static_cast<int64_t>(seq_len[b]) + add + tok(r)) / ratio;
    return n < 0 ? 0 : n;
  }
  HSA_DEVINL bool valid(int r) const {
    const int b = seq(r);
    const int64_t o0 = offsets[b], o1 = offsets[b + 1];
    return o0 >= 0 && o1 >= o0 && o1 <= limit && raw_count(r) <= o1 - o0;
  }
  HSA_DEVINL int64_t count(int r) const { return valid(r) ? raw_count(r) : 0; }
};

// Arguments of one fused-attention launch (see hsa_decode_attn in hsa.h).
struct AttnArgs {
  const void* q;
  const void* swa;
  const int32_t* seq_len;
  int32_t len_add;    // attended window length is seq_len[b] + len_add (per sequence b)
  int64_t W;          // window rows attended
  // Multi-token queries: tokens b' = b * T + t of sequence b (q, out, lse and
  // idx rows per token); token t attends a window of length seq_len[b] +
  // len_add + t, from a ring of Wr >= W + T - 1 rows (slot = position mod Wr)
  int32_t T = 1;
  int64_t Wr = 0;     // 0: W
  const void* extra;  // compressed pool (null: window only)
  Spans sp;           // its sequences
  const int32_t* idx; // [B, k] row-local indices, or null for dense
  int64_t k;
  int64_t max_rows;   // dense: bound on compressed rows per sequence
  int64_t B, Hq, Dqk, Dv;
  float scale;
  void* out;
  int out_dtype;
  float* lse;
  // The previous kernel of the stream (under programmatic dependent launch)
  // writes only the index lists: the window rows, lengths and q may be read
  // before waiting for it.  False when it may write anything else.
  bool only_idx_pending = false;
  // Dense attention (idx null) right after the append: the lengths come from
  // the step's input (seq_len + len_add, not written by the append), and only
  // the tiles holding rows the append writes (the window's, and the pool rows
  // of a block completed in this step) wait for it.
  bool append_pending = false;
  // Fused selection (idx null): the kernel selects every token's top-k itself
  // from these scores (at the pool's row positions) and the per-row key
  // histograms the indexer built (zeroed again), writing the selection in
  // order to topk_out when it is not null; cand_ws holds heavy-tie
  // candidates (one slot per pool row).  Only the kernels' own reads of their
  // predecessor's outputs wait for it: every read of the append's outputs
  // (window rows) and of the indexer's comes after the wait.
  const float* sel_scores = nullptr;
  uint32_t* row_hist = nullptr;
  uint64_t* cand_ws = nullptr;
  int32_t* topk_out = nullptr;
};

// Launch geometry of the fused attention: HG heads per CTA (N = MMA width),
// G head groups, S key splits of sps attended slots each, TC tiles per chunk
// (S^T accumulators held in TMEM at once), dynamic shared memory.  With cl,
// the S splits of a (token, head group) form one thread-block cluster and
// merge their partial outputs through distributed shared memory (no combine
// kernel, no partials in global memory).
struct AttnPlan {
  int HG, N, G, S, TC;
  int64_t sps;
  size_t smem;
  int cl;
};

AttnPlan attn_plan(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W, int64_t extra_slots);
// Whether a plan can run the fused selection for a top-k of k over rows of at
// most max_row scores.
bool attn_fused_ok(const AttnPlan& pl, int64_t k, int64_t max_row);
size_t attn_workspace_bytes(const AttnPlan& pl, int64_t B, int64_t Hq, int64_t Dv);
// ws: attn_workspace_bytes() of scratch (partials after a kWsHeader gap);
// status: the sticky status word to report into.
cudaError_t launch_attn(const AttnArgs& a, const AttnPlan& pl, void* ws, uint32_t* status,
                        cudaStream_t stream, bool pdl = false);

// Block-wide inclusive sum over one value per thread (blockDim.x <= 1024).
// `scratch` holds 33 elements of shared memory.  Returns the inclusive prefix;
// *total receives the block total.  All threads must call it.
template <typename T>
HSA_DEVINL T block_inclusive_sum(T v, T* scratch, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T s = lane < nwarps ? scratch[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < nwarps) scratch[lane] = s;
    if (lane == nwarps - 1) scratch[32] = s;
  }
  __syncthreads();
  if (warp > 0) v += scratch[warp - 1];
  *total = scratch[32];
  __syncthreads();
  return v;
}

// Maps a flat work-item index to (sequence, piece) when sequence b is cut
// into pieces(b) pieces; pieces() is evaluated per sequence.  Returns false
// when `item` is past the last piece.  All threads of the block must call it
// (blockDim.x <= 1024); the result is uniform across the block.
template <typename PiecesFn>
HSA_DEVINL bool locate_piece(int B, int64_t item, PiecesFn pieces, int* seq, int64_t* piece,
                             int64_t* npieces) {
  __shared__ int64_t s_scratch[33];
  __shared__ int s_seq;
  __shared__ int64_t s_piece, s_np;
  if (threadIdx.x == 0) s_seq = -1;
  int64_t before = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int64_t np = b < B ? pieces(b) : 0;
    int64_t total;
    const int64_t incl = block_inclusive_sum<int64_t>(np, s_scratch, &total);
    const int64_t lo = before + incl - np;
    if (b < B && item >= lo && item < lo + np) {
      s_seq = b;
      s_piece = item - lo;
      s_np = np;
    }
    __syncthreads();
    if (s_seq >= 0) break;
    before += total;
  }
  const bool found = s_seq >= 0;
  if (found) {
    *seq = s_seq;
    *piece = s_piece;
    *npieces = s_np;
  }
  __syncthreads();
  return found;
}

}  // namespace hsa
