// One decode step of one hybrid layer: append -> compress on block
// completion -> (C4) indexer scores -> top-k -> fused attention, all on one
// stream with no host synchronisation.
//
// [WK] "与 SGLang 团队聊 DeepSeek V4", §核心观点: a layer keeps five kinds of
// state — the SWA window, the C4 and C128 pools, and the in-flight C4/C128
// blocks that are compressed once 4 / 128 tokens have accumulated; C4 picks
// its top-k entries, C128 attends all.  [KD] "DeepSeek-V4: optimización de
// inferencia y RL ...", §Arquitectura del Sistema (compression-state ring
// buffers in their own pool) and §Flujo de Inferencia steps 3, 5 and 6.
//
// Step order follows the data dependence (the top-k must pick the C4 entries
// before the attention reads them):
//   a1 append   new kv row -> SWA ring slot (L-1) mod W and in-flight slot
//               (L-1) mod r (kv, gate logits; C4 also the raw indexer key and
//               its gate), L = seq_len_in + 1; seq_len_out = L
//   a2 compress if L mod r == 0: the completed block -> pool row L/r - 1
//   a3 scores   (C4) indexer over the sequence's L/4 entries
//   a4 top-k    (C4) k largest scores
//   a5 attend   window + top-k (C4) or all L/128 entries (C128)
// a1 and a2 run in one small kernel (one CTA per sequence); a3-a5 are the
// standalone kernels reading the live prefix of the capacity-laid-out pools.
#include <cuda_fp8.h>

#include "common.cuh"
#include "compress_core.cuh"
#include "internal.h"

namespace hsa {
namespace {

constexpr int kAppendThreads = 256;
// rows of a block's 8-channel chunk split over this many lanes (one load
// round of at most 4 rows each, up to 32 lanes)
HSA_HOST_DEVICE int block_split(int r) {
  int split = 1;
  while (split < 32 && 8 * split <= r) split <<= 1;
  return split;
}

struct AppendParams {
  int kind, r, B, Dqk, Di, W;
  const int32_t* seq_len_in;
  int32_t* seq_len_out;
  const int64_t* pool_offsets;
  int64_t pool_total_rows;
  const uint4* kv_new;
  const uint4* z_new;
  const float* b_kv;
  const uint4* ik_new;
  const uint4* iz_new;
  const float* b_ik;
  uint4* swa;
  uint4* kv_ring;
  uint4* z_ring;
  uint4* ik_ring;
  uint4* iz_ring;
  uint4* kv_pool;
  uint4* key_pool;
  float* key_scale;  // non-null: key_pool holds E4M3 codes [rows, Di] with these fp32 scales
  uint32_t* status;
  uint32_t* tickets;  // [B] (blocks of more than kShortBlock rows) CTAs done per sequence, zero between steps
  int G;             // (blocks of more than kShortBlock rows) CTAs per sequence
  int T;             // tokens appended per step (rows b * T + t of the new-row inputs)
  int Wr;            // window ring rows (W + T - 1)
};


constexpr int kMaxKeyDi = 128;  // E4M3 key rows (one warp quantizes a row, 4 channels a lane)

// Short blocks (r <= 4, the C4 layer): one thread owns one 8-channel chunk of
// the kv row or of the indexer-key row end to end.  Every load it may need is
// issued up front (the length, the pool offsets, the new rows, the block's
// earlier ring rows and the biases), so the step costs one memory round trip;
// the new row is then written to the rings and, when it completes the block,
// the block is compressed from registers (the ring row it just wrote is the
// block's last row).
constexpr int kShortBlock = 4;

template <int kT>  // tokens appended (p.T == kT)
HSA_DEVINL void append_short(const AppendParams& p, int b) {
  __shared__ float s_key[kMaxKeyDi];  // E4M3 pool: the completed block's fp32 key row
  const int cq = p.Dqk / 8, ci = p.kind == HSA_LAYER_C4 ? p.Di / 8 : 0;
  const int r = p.r;
  constexpr int T = kT;
  const int32_t lin = p.seq_len_in[b];
  const int64_t o0 = p.pool_offsets[b], o1 = p.pool_offsets[b + 1];
  // the step's token whose position completes a block (at most one: T <= r)
  int tcomp = -1;
  for (int t = 0; t < T; ++t)
    if ((static_cast<int64_t>(lin) + t + 1) % r == 0) tcomp = t;
  const int64_t pc = static_cast<int64_t>(lin) + tcomp;  // its position (when tcomp >= 0)
  for (int it = threadIdx.x; it < cq + ci; it += blockDim.x) {
    const bool key = it >= cq;
    const int c = key ? it - cq : it, n8 = key ? ci : cq, C = n8 * 8;
    const uint4* nv_src = key ? p.ik_new : p.kv_new;
    const uint4* nz_src = key ? p.iz_new : p.z_new;
    uint4* ring_v = (key ? p.ik_ring : p.kv_ring) + static_cast<int64_t>(b) * r * n8 + c;
    uint4* ring_z = (key ? p.iz_ring : p.z_ring) + static_cast<int64_t>(b) * r * n8 + c;
    const float* bias = (key ? p.b_ik : p.b_kv) + c * 8;
    uint4 nv[kT], nz[kT];  // the step's new rows (token t: row b * T + t)
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      nv[t] = nv_src[(static_cast<int64_t>(b) * T + t) * n8 + c];
      nz[t] = nz_src[(static_cast<int64_t>(b) * T + t) * n8 + c];
    }
    uint4 rv[kShortBlock], rz[kShortBlock];
    float4 b0[kShortBlock], b1[kShortBlock];
#pragma unroll
    for (int i = 0; i < kShortBlock; ++i) {
      if (i < r) {
        rv[i] = ring_v[static_cast<int64_t>(i) * n8];
        rz[i] = ring_z[static_cast<int64_t>(i) * n8];
        const float4* bp = reinterpret_cast<const float4*>(bias + static_cast<int64_t>(i) * C);
        b0[i] = __ldg(bp);
        b1[i] = __ldg(bp + 1);
      }
    }
    // the new rows into the window ring and the in-flight rings, in order
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      const int64_t pos = static_cast<int64_t>(lin) + t;
      if (!key) p.swa[(static_cast<int64_t>(b) * p.Wr + pos % p.Wr) * cq + c] = nv[t];
      ring_v[(pos % r) * n8] = nv[t];
      ring_z[(pos % r) * n8] = nz[t];
    }
    if (tcomp < 0) continue;
    const int64_t n = (pc + 1) / r - 1;
    if (o0 < 0 || o1 > p.pool_total_rows || o0 + n >= o1) {
      set_status(p.status, HSA_DEV_BOUNDS);
      continue;
    }
    // the completed block: slot i holds position pc - r + 1 + i, a new row of
    // this step when at or past lin (the ring's copy loaded above otherwise)
    float x[kShortBlock][8], v[kShortBlock][8], mx[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) mx[ch] = -INFINITY;
#pragma unroll
    for (int i = 0; i < kShortBlock; ++i) {
      if (i < r) {
        const int64_t tq = pc - r + 1 + i - lin;  // token index of the row, if new
        uint4 zi = rz[i], vi = rv[i];
#pragma unroll
        for (int t = 0; t < kT; ++t)
          if (tq == t) {
            zi = nz[t];
            vi = nv[t];
          }
        bf16x8_to_f32(zi, x[i]);
        bf16x8_to_f32(vi, v[i]);
        const float bb[8] = {b0[i].x, b0[i].y, b0[i].z, b0[i].w, b1[i].x, b1[i].y, b1[i].z, b1[i].w};
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          x[i][ch] += bb[ch];  // add
          mx[ch] = fmaxf(mx[ch], x[i][ch]);
        }
      }
    }
    float o[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      float l = 0.f, acc = 0.f;
#pragma unroll
      for (int i = 0; i < kShortBlock; ++i) {
        if (i < r) {
          const float e = __expf(x[i][ch] - mx[ch]);  // softmax numerator
          l += e;
          acc = fmaf(e, v[i][ch], acc);  // dot
        }
      }
      o[ch] = acc / l;
    }
    if (key && p.key_scale) {  // E4M3 pool: quantized below, once the whole row is here
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) s_key[c * 8 + ch] = o[ch];
      continue;
    }
    uint4* dst = key ? p.key_pool : p.kv_pool;
    dst[(o0 + n) * n8 + c] = f32x8_to_bf16(o);
  }
  __syncthreads();  // every thread has read seq_len_in before it may be overwritten
  if (p.key_scale && threadIdx.x < 32 && tcomp >= 0) {
    // warp 0 quantizes the completed block's key row: amax over the row, then
    // 4 channels a lane
    const int64_t n = (pc + 1) / r - 1;
    if (!(o0 < 0 || o1 > p.pool_total_rows || o0 + n >= o1)) {
      const int lane = threadIdx.x;
      const bool live = 4 * lane < p.Di;
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = live ? s_key[4 * lane + i] : 0.f;
      float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const float inv = am > 0.f ? __fdiv_rn(448.f, am) : 0.f;
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)), __NV_SATFINITE, __NV_E4M3);
      if (live)
        reinterpret_cast<uint32_t*>(p.key_pool)[((o0 + n) * p.Di) / 4 + lane] =
            static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      if (lane == 0) p.key_scale[o0 + n] = __fdiv_rn(am, 448.f);
    }
  }
  if (threadIdx.x == 0) p.seq_len_out[b] = lin + T;
}

template <int kT>  // tokens per step of the short-block path (p.T == kT there)
__global__ void __launch_bounds__(kAppendThreads) layer_append_kernel(AppendParams p) {
  pdl_wait();
  pdl_trigger();
  append_short<kT>(p, blockIdx.x);
}

// Blocks of more than kShortBlock rows (the C128 layer): p.G CTAs per
// sequence, each compressing a slice of the block's 8-channel chunks (each
// chunk's rows split over block_split(r) lanes: one load round per lane, one
// round of the CTA's threads).
// Block row i is ring slot i; the rows this step appends come straight from
// the new-row inputs, so no CTA waits for another's ring writes.  The
// sequence's CTAs take an atomic ticket when done; the last one writes the
// rows of the step's tokens after the completing one (the next block's first
// slots, read by the others until then) and the new length (which may alias
// the one every CTA read), and resets the ticket.
__global__ void __launch_bounds__(kAppendThreads) layer_append_long_kernel(AppendParams p) {
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  const int G = p.G;
  const int b = blockIdx.x / G, g = blockIdx.x % G;
  const int64_t lin = p.seq_len_in[b];
  const int cq = p.Dqk / 8, ci = p.Di / 8;
  const int64_t o0 = p.pool_offsets[b], o1 = p.pool_offsets[b + 1];
  // a1: tokens [t_lo, t_hi)'s rows into the window ring and the in-flight rings
  auto write_rows = [&](int t_lo, int t_hi) {
    for (int t = t_lo; t < t_hi; ++t) {
      const int64_t pos = lin + t;
      const int64_t slot_w = pos % p.Wr, slot_r = pos % p.r;
      const int64_t row = static_cast<int64_t>(b) * p.T + t;
      for (int c = threadIdx.x; c < cq; c += blockDim.x) {
        const uint4 kv = p.kv_new[row * cq + c];
        const uint4 z = p.z_new[row * cq + c];
        p.swa[(static_cast<int64_t>(b) * p.Wr + slot_w) * cq + c] = kv;
        p.kv_ring[(static_cast<int64_t>(b) * p.r + slot_r) * cq + c] = kv;
        p.z_ring[(static_cast<int64_t>(b) * p.r + slot_r) * cq + c] = z;
      }
      if (p.kind == HSA_LAYER_C4) {
        for (int c = threadIdx.x; c < ci; c += blockDim.x) {
          p.ik_ring[(static_cast<int64_t>(b) * p.r + slot_r) * ci + c] = p.ik_new[row * ci + c];
          p.iz_ring[(static_cast<int64_t>(b) * p.r + slot_r) * ci + c] = p.iz_new[row * ci + c];
        }
      }
    }
  };
  // the step's token that completes a block (at most one: T <= r), or -1
  int tcomp = -1;
  for (int t = 0; t < p.T; ++t)
    if ((lin + t + 1) % p.r == 0) tcomp = t;
  if (g == 0) write_rows(0, tcomp >= 0 ? tcomp + 1 : p.T);
  if (tcomp >= 0) {
    // a2: the block is complete -> compress it into pool row (pos + 1)/r - 1
    const int64_t n = (lin + tcomp + 1) / p.r - 1;
    if (o0 < 0 || o1 > p.pool_total_rows || o0 + n >= o1) {
      if (threadIdx.x == 0 && g == 0) set_status(p.status, HSA_DEV_BOUNDS);
    } else {
      // rows [inew, r) are this step's tokens 0..tcomp
      const int inew = p.r - 1 - tcomp;
      const uint4* ring_kv = p.kv_ring + static_cast<int64_t>(b) * p.r * cq;
      const uint4* ring_z = p.z_ring + static_cast<int64_t>(b) * p.r * cq;
      const int64_t new0 = static_cast<int64_t>(b) * p.T;  // row of the step's token 0
      const int c0 = g * cq / G, c1 = (g + 1) * cq / G;
      const int split = block_split(p.r);
      const int items = (c1 - c0) * split;
      uint4* dst = p.kv_pool + (o0 + n) * cq;
      for (int i0 = 0; i0 < items; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        if (split > 1 && i0 + static_cast<int>(threadIdx.x & ~31u) >= items) break;  // whole idle warp
        const bool live = i < items;
        const int c = c0 + (live ? i / split : 0), part = live ? i % split : 0;
        const int per = (p.r + split - 1) / split;
        const int lo = live ? min(p.r, part * per) : 0, hi = live ? min(p.r, lo + per) : 0;
        auto rows = [&](int row, const uint4** kp, const uint4** zp) {
          if (row < inew) {
            *kp = ring_kv + static_cast<int64_t>(row) * cq + c;
            *zp = ring_z + static_cast<int64_t>(row) * cq + c;
          } else {
            *kp = p.kv_new + (new0 + row - inew) * cq + c;
            *zp = p.z_new + (new0 + row - inew) * cq + c;
          }
        };
        auto brow = [&](int row, float4* b0, float4* b1) {
          const float4* bp = reinterpret_cast<const float4*>(p.b_kv + static_cast<int64_t>(row) * p.Dqk + c * 8);
          *b0 = __ldg(bp);
          *b1 = __ldg(bp + 1);
        };
        GatePartial pt;
        partial_init(pt);
        partial_rows_at(rows, lo, hi, brow, pt);
        if (split > 1) partial_merge_lanes(pt, split);
        if (live && part == 0) {
          float o[8];
          partial_result(pt, o);
          dst[c] = f32x8_to_bf16(o);
        }
      }
    }
  }
  // the sequence's last CTA: the later tokens' rows and the new length
  __syncthreads();
  __threadfence();
  if (threadIdx.x == 0) s_last = atomicAdd(p.tickets + b, 1u) == static_cast<uint32_t>(G) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tcomp >= 0) write_rows(tcomp + 1, p.T);
  if (threadIdx.x == 0) {
    p.seq_len_out[b] = static_cast<int32_t>(lin + p.T);
    p.tickets[b] = 0;
  }
}

HSA_HOST_DEVICE size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// Query tokens per sequence in one step (multi-token queries).
int layer_tokens(const hsa_layer_desc& d) { return d.T > 1 ? d.T : 1; }

AttnPlan layer_attn_plan(const hsa_layer_desc& d) {
  const int64_t slots = d.kind == HSA_LAYER_C4 ? d.k : d.max_pool_rows;
  return attn_plan(static_cast<int64_t>(d.B) * layer_tokens(d), d.Hq, d.Dqk, d.Dv, d.W, slots);
}

// A C4 layer whose rows and plan allow it selects its top-k inside the
// attention kernel, from the indexer's scores and the per-row key histograms
// the indexer builds while writing them (no top-k launch, no index list in
// global memory); otherwise the top-k runs as its own kernels.
bool layer_fused(const hsa_layer_desc& d) {
  if (d.kind != HSA_LAYER_C4) return false;
  const int64_t max_row = d.max_pool_rows > 0 ? d.max_pool_rows : d.pool_total_rows;
  return attn_fused_ok(layer_attn_plan(d), d.k, max_row);
}

// With T query tokens the score, top-k and selection areas are per token:
// token t's scores at pool row positions + t * pool_total_rows.
struct LayerWs {
  size_t scores, topk, idx, hist, attn, tickets, total;
  LayerWs(const hsa_layer_desc& d, const AttnPlan& pl) {
    const int64_t T = layer_tokens(d), BT = static_cast<int64_t>(d.B) * T;
    const int64_t srows = (d.pool_total_rows > 0 ? d.pool_total_rows : 1) * T;
    size_t at = kWsHeader;
    scores = topk = idx = hist = 0;
    tickets = at;
    at += a256(static_cast<size_t>(d.B) * sizeof(uint32_t));
    if (d.kind == HSA_LAYER_C4) {
      scores = at;
      if (!d.scores) at += a256(static_cast<size_t>(srows) * 4);
      topk = at;
      at += a256(topk_workspace_bytes(BT, d.pool_total_rows * T, d.k));
      idx = at;
      if (!d.topk_idx) at += a256(static_cast<size_t>(BT) * d.k * 4);
      if (layer_fused(d)) {
        hist = at;
        at += a256(static_cast<size_t>(BT) * kRowHistBins * sizeof(uint32_t));
      }
    }
    attn = at;
    at += a256(attn_workspace_bytes(pl, BT, d.Hq, d.Dv));
    total = at;
  }
};

}  // namespace

size_t layer_workspace_bytes(const hsa_layer_desc& d) {
  return LayerWs(d, layer_attn_plan(d)).total;
}

int layer_launch_count(const hsa_layer_desc& d) {
  const AttnPlan pl = layer_attn_plan(d);
  int n = 1 + 1 + (pl.S > 1 && !pl.cl ? 1 : 0);  // append, attention (+ combine)
  if (d.kind == HSA_LAYER_C4)
    n += (d.pool_total_rows > 0 ? 1 : 0) +
         (layer_fused(d) ? 0 : topk_launch_count(d.pool_total_rows * layer_tokens(d), d.max_pool_rows));
  return n;
}

cudaError_t launch_layer(const hsa_layer_desc& d, void* ws, cudaStream_t stream) {
  const int r = d.kind;
  const AttnPlan pl = layer_attn_plan(d);
  const LayerWs L(d, pl);
  char* w = static_cast<char*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(w);

  AppendParams ap;
  ap.kind = d.kind;
  ap.r = r;
  ap.B = d.B;
  ap.Dqk = d.Dqk;
  ap.Di = d.kind == HSA_LAYER_C4 ? d.Di : 0;
  ap.W = d.W;
  ap.seq_len_in = d.seq_len_in;
  ap.seq_len_out = d.seq_len_out;
  ap.pool_offsets = d.pool_offsets;
  ap.pool_total_rows = d.pool_total_rows;
  ap.kv_new = static_cast<const uint4*>(d.kv_new);
  ap.z_new = static_cast<const uint4*>(d.z_new);
  ap.b_kv = d.b_kv;
  ap.ik_new = static_cast<const uint4*>(d.ik_new);
  ap.iz_new = static_cast<const uint4*>(d.iz_new);
  ap.b_ik = d.b_ik;
  ap.swa = static_cast<uint4*>(d.swa);
  ap.kv_ring = static_cast<uint4*>(d.kv_ring);
  ap.z_ring = static_cast<uint4*>(d.z_ring);
  ap.ik_ring = static_cast<uint4*>(d.ik_ring);
  ap.iz_ring = static_cast<uint4*>(d.iz_ring);
  ap.kv_pool = static_cast<uint4*>(d.kv_pool);
  ap.key_pool = static_cast<uint4*>(d.key_pool);
  ap.key_scale = d.kind == HSA_LAYER_C4 && d.key_fp8 ? d.key_scale : nullptr;
  ap.status = status;
  ap.tickets = reinterpret_cast<uint32_t*>(w + L.tickets);
  // (blocks of more than kShortBlock rows) CTAs per sequence: the block's
  // chunk-lane items in one round of each CTA's threads
  ap.G = (d.Dqk / 8 * block_split(r) + kAppendThreads - 1) / kAppendThreads;
  const int T = layer_tokens(d);
  ap.T = T;
  ap.Wr = d.W + T - 1;
  auto mark = [&](int i) -> cudaError_t {
    return d.stage_events ? cudaEventRecord(static_cast<cudaEvent_t>(d.stage_events[i]), stream)
                          : cudaSuccess;
  };
  cudaError_t e = mark(0);
  if (e != cudaSuccess) return e;
  // (one instantiation per token count: the rows of a step live in registers)
  if (ap.r > kShortBlock)
    layer_append_long_kernel<<<d.B * ap.G, kAppendThreads, 0, stream>>>(ap);
  else if (T == 1) layer_append_kernel<1><<<d.B, kAppendThreads, 0, stream>>>(ap);
  else if (T == 2) layer_append_kernel<2><<<d.B, kAppendThreads, 0, stream>>>(ap);
  else if (T == 3) layer_append_kernel<3><<<d.B, kAppendThreads, 0, stream>>>(ap);
  else layer_append_kernel<4><<<d.B, kAppendThreads, 0, stream>>>(ap);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = mark(1)) != cudaSuccess) return e;

  // a3-a5 read the live prefix L/r of each sequence's pool rows (per query
  // token: token t of a step of T sees L - (T - 1 - t) tokens).  sp / sp_in
  // count the sequence's rows for its last token (the indexer's tiles); the
  // token spans (tk) give token b * T + t its own count and score row.
  const Spans sp{d.pool_offsets, d.seq_len_out, 0, r, d.pool_total_rows};
  auto tokens = [&](const Spans& s) {
    Spans t = s;
    t.add = s.add - (T - 1);
    t.T = T;
    t.tstride = d.pool_total_rows;
    return t;
  };
  const int32_t* idx = nullptr;
  if (d.kind == HSA_LAYER_C4) {
    float* scores = d.scores ? d.scores : reinterpret_cast<float*>(w + L.scores);
    int32_t* tidx = d.topk_idx ? d.topk_idx : reinterpret_cast<int32_t*>(w + L.idx);
    // The lengths after the append are the ones before it plus one, so the
    // indexer and the top-k can read their row geometry before the append has
    // finished, and the indexer streams every key the append cannot have
    // written (all but a completed block's new row) while it runs.  When the
    // output lengths overwrite the input ones, the geometry is read from the
    // output lengths after the append instead.
    const bool alias = d.seq_len_out == d.seq_len_in;
    const Spans sp_in{d.pool_offsets, d.seq_len_in, T, r, d.pool_total_rows};
    const bool fused = layer_fused(d);
    uint32_t* hist = fused ? reinterpret_cast<uint32_t*>(w + L.hist) : nullptr;
    e = launch_indexer(d.iq, d.w, d.key_pool, alias ? sp : sp_in, d.B, d.Hi, d.Di,
                       d.pool_total_rows, scores, status, stream, true, alias ? 0 : 2, hist,
                       d.key_fp8 ? d.key_scale : nullptr, T);
    if (e != cudaSuccess) return e;
    if ((e = mark(2)) != cudaSuccess) return e;
    if (fused) {
      // the attention selects the top-k itself (its geometry from the input
      // lengths + 1, as the top-k's would be)
      if ((e = mark(3)) != cudaSuccess) return e;
      AttnArgs a;
      a.q = d.q;
      a.swa = d.swa;
      a.seq_len = alias ? d.seq_len_out : d.seq_len_in;
      a.len_add = alias ? 1 - T : 1;  // token t: L_in + 1 + t
      a.W = d.W;
      a.T = T;
      a.Wr = d.W + T - 1;
      a.extra = d.kv_pool;
      a.sp = tokens(alias ? sp : sp_in);
      a.idx = nullptr;
      a.k = d.k;
      a.max_rows = 0;
      a.B = static_cast<int64_t>(d.B) * T;
      a.Hq = d.Hq;
      a.Dqk = d.Dqk;
      a.Dv = d.Dv;
      a.scale = d.scale;
      a.out = d.out;
      a.out_dtype = d.out_dtype;
      a.lse = d.lse;
      a.only_idx_pending = true;
      a.sel_scores = scores;
      a.row_hist = hist;
      a.cand_ws = topk_cand_area(w + L.topk, static_cast<int64_t>(d.B) * T, d.pool_total_rows * T, d.k);
      a.topk_out = d.topk_idx;
      bool pdl = true;
      if (d.q_ready_event) {
        e = cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(d.q_ready_event), 0);
        if (e != cudaSuccess) return e;
        pdl = false;
      }
      e = launch_attn(a, pl, w + L.attn, status, stream, pdl);
      if (e != cudaSuccess) return e;
      return mark(4);
    }
    e = launch_topk(scores, tokens(alias ? sp : sp_in), d.B * T, d.pool_total_rows * T, d.k, tidx,
                    nullptr, w + L.topk, status, stream, d.max_pool_rows, true);
    if (e != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    idx = tidx;
  } else {
    if ((e = mark(2)) != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
  }
  // C128: with separate output lengths the attention takes its geometry from
  // the input lengths (plus one per token) and starts while the append runs
  const bool early = d.kind == HSA_LAYER_C128 && d.seq_len_out != d.seq_len_in;
  const Spans sp_in{d.pool_offsets, d.seq_len_in, T, r, d.pool_total_rows};
  AttnArgs a;
  a.q = d.q;
  a.swa = d.swa;
  a.seq_len = early ? d.seq_len_in : d.seq_len_out;
  a.len_add = early ? 1 : 1 - T;  // token t: L_in + 1 + t = L_out - (T - 1 - t)
  a.W = d.W;
  a.T = T;
  a.Wr = d.W + T - 1;
  a.extra = d.kv_pool;
  a.sp = tokens(early ? sp_in : sp);
  a.idx = idx;
  a.k = d.kind == HSA_LAYER_C4 ? d.k : 0;
  a.max_rows = d.kind == HSA_LAYER_C4 ? 0 : d.max_pool_rows;
  a.B = static_cast<int64_t>(d.B) * T;
  a.Hq = d.Hq;
  a.Dqk = d.Dqk;
  a.Dv = d.Dv;
  a.scale = d.scale;
  a.out = d.out;
  a.out_dtype = d.out_dtype;
  a.lse = d.lse;
  a.only_idx_pending = d.kind == HSA_LAYER_C4;  // C128: the append comes right before
  a.append_pending = early;
  bool pdl = true;
  if (d.q_ready_event) {
    // q may still be arriving on another stream: the attention waits for it
    e = cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(d.q_ready_event), 0);
    if (e != cudaSuccess) return e;
    pdl = false;
  }
  e = launch_attn(a, pl, w + L.attn, status, stream, pdl);
  if (e != cudaSuccess) return e;
  return mark(4);
}

}  // namespace hsa
