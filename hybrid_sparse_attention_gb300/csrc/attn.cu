// Fused hybrid attention: one softmax over the SWA window plus the selected
// C4 entries (sparse) or all C128 entries (dense), on tcgen05 tensor cores.
//
// [KD] "DeepSeek-V4: optimización de inferencia y RL ...", §Flujo de
// Inferencia step 5 and the technology table (FlashMLA: SWA and the extra
// C4/C128 attention fused in one kernel); [LH] "DeepSeek-V4: SGLang và Miles
// ...", §Tích hợp Kernel (SWA and the extra attention in one kernel call);
// [WK] "与 SGLang 团队聊 DeepSeek V4", §核心观点 (SWA sees the latest tokens,
// C4 attends its top-k, C128 attends everything).
//
// Per query token b and head h, over the attended slots t (window rows, then
// the listed / all compressed rows; keys are Dqk-wide rows of one shared
// latent KV head, values their first Dv channels):
//   o[b,h] = sum_t softmax_t(scale * q[b,h] . K_t) V_t,   lse[b,h] = log sum_t e^(...)
//
// Design (sm_103a):
//  * The keys are the M = 128 side of both contractions, so one gathered tile
//    of 128 key rows in shared memory feeds both MMAs without re-layout:
//      S^T[key, head] = K_tile . Q^T      (A = K tile, K-major over Dqk)
//      O^T[dv, head] += V_tile^T . P^T    (A = the same tile, MN-major view)
//    Q (a group of 32 heads) and P^T are the N side.  S^T, O^T live in TMEM.
//  * The K tile is stored as Dqk/64 slices of [128 keys x 64 channels] in the
//    128-byte swizzled layout; slice j always lives in buffer j, so slices 2m
//    and 2m+1 (the value channels of O^T M-tile m) sit 16 KB apart, which is
//    the MN-major descriptor's leading-byte offset.  A buffer is refilled for
//    the next tile as soon as its last reader commits (the rope slices after
//    the S^T MMAs, value slices after their O^T M-tile), so the gather of
//    tile t+1 overlaps the softmax and O^T of tile t.
//  * Warp roles: warps 0-3 own TMEM lanes 0-127 (softmax of one key each, then
//    the epilogue of one value channel each); warp 4 allocates TMEM and one
//    lane issues every tcgen05.mma; warps 5-7 gather rows with 16-byte
//    cp.async (8 consecutive threads per 128-byte row segment, zero-fill for
//    masked slots) from a per-tile table of row addresses in shared memory.
//  * Softmax: per-head maxima by a warp transpose-reduction plus one shared
//    exchange; lazy rescaling (the running maximum only moves when a tile
//    raises it by more than 2^8, so P <= 256 and O^T is corrected in TMEM
//    only then); row sums accumulate per thread and reduce once at the end.
//  * Long key lists are split over CTAs; each split writes an fp32 partial
//    output and log-sum-exp that a combine kernel merges.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kKeys = 128;
constexpr int kSmWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kProdThreads = 96;
constexpr int kThreads = 32 * 8;
constexpr int kMaxSlices = 9;
constexpr uint32_t kSliceBytes = kKeys * 128;
constexpr float kRescaleLog2 = 8.f;

struct AttnParams {
  const uint16_t* q;      // [B, Hq, Dqk]
  const uint16_t* swa;    // [B, W, Dqk]
  const int32_t* seq_len;
  int32_t len_add;
  int W;
  const uint16_t* extra;  // compressed pool rows (may be null)
  Spans sp;
  const int32_t* idx;     // [B, k] or null (dense)
  int k;
  int64_t max_rows;       // dense: cap on compressed rows per sequence
  int B, Hq, Dqk, Dv;
  int HG, G, S, tps;
  float scale_log2;
  void* out;
  int out_dtype;
  float* lse;
  float* po;              // partial outputs [B, S, Hq, Dv] (S > 1)
  float* plse;            // partial lse [B, S, Hq] (S > 1)
  uint32_t* status;
};

struct SeqGeom {
  int64_t L, off, nb;
  int n_swa;
  int64_t n_extra;
};

HSA_DEVINL SeqGeom seq_geom(const AttnParams& p, int b) {
  SeqGeom g;
  int64_t L = static_cast<int64_t>(p.seq_len[b]) + p.len_add;
  g.L = L < 0 ? 0 : L;
  g.n_swa = static_cast<int>(g.L < p.W ? g.L : p.W);
  g.off = 0;
  g.nb = 0;
  g.n_extra = 0;
  if (p.extra) {
    g.off = p.sp.start(b);
    g.nb = p.sp.count(b);
    if (p.idx) {
      g.n_extra = p.k;
    } else {
      g.n_extra = g.nb < p.max_rows ? g.nb : p.max_rows;
    }
  }
  return g;
}

// Global row of attended slot `slot` of sequence b, or null when the slot is
// masked (past the end, or a -1 / out-of-range index; the latter is flagged).
HSA_DEVINL const uint16_t* slot_row(const AttnParams& p, int b, const SeqGeom& g, int64_t slot,
                                    bool report) {
  if (slot < g.n_swa) {
    const int64_t pos = g.L - g.n_swa + slot;
    return p.swa + (static_cast<int64_t>(b) * p.W + pos % p.W) * p.Dqk;
  }
  const int64_t e = slot - g.n_swa;
  if (e >= g.n_extra) return nullptr;
  int64_t j = e;
  if (p.idx) {
    j = p.idx[static_cast<int64_t>(b) * p.k + e];
    if (j < 0) return nullptr;
    if (j >= g.nb) {
      if (report) set_status(p.status, HSA_DEV_BOUNDS);
      return nullptr;
    }
  }
  return p.extra + (g.off + j) * p.Dqk;
}

// Order in which the slices of a tile are loaded and multiplied: the
// channels past Dv (rope) first, since their buffers free up first.
HSA_DEVINL int slice_order(int jj, int NSL, int NV) {
  return jj < NSL - NV ? NV + jj : jj - (NSL - NV);
}

// Byte offset of element (row, 16-byte chunk) in a 128-byte-swizzled
// K-major block whose rows are 128 bytes (8-row atoms of 1024 bytes).
HSA_DEVINL uint32_t sw128(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
}

// Column reduction of a 32 x kN register tile held one row per lane: on
// return lane l holds the reduction of column (l mod kN) over the warp.
template <int kN, bool kMax>
HSA_DEVINL float warp_transpose_reduce(float (&v)[kN]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int width = kN / 2; width >= 1; width >>= 1) {
    const bool upper = (lane & width) != 0;
#pragma unroll
    for (int i = 0; i < width; ++i) {
      const float send = upper ? v[i] : v[i + width];
      const float keep = upper ? v[i + width] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, width);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
  if (kN == 16) {
    const float o = __shfl_xor_sync(0xffffffffu, r, 16);
    r = kMax ? fmaxf(r, o) : r + o;
  }
  return r;
}

struct Shared {
  uint64_t full[kMaxSlices], empty[kMaxSlices];
  uint64_t s_full[2], s_empty[2], o_done[2];
  uint64_t p_full, q_full, fin;
  uint32_t tmem;
  int abort;
  float red[kSmWarps][32];
  float bc[32];
  float m[32];      // running maximum per head (log2 units), identical for every thread
  float alpha[32];  // rescale factor of the current tile per head
  const uint16_t* rows[2][kKeys];  // gather table of the producers (per tile parity)
};

// Bounded wait that also gives up when another role has aborted.
HSA_DEVINL bool wait_or_abort(Shared& sh, uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_timer();
  for (uint32_t i = 0;; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*reinterpret_cast<volatile int*>(&sh.abort)) return false;
      if (tc::global_timer() - t0 > tc::kSpinNanos || i > tc::kSpinPolls) {
        set_status(status, HSA_DEV_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sh.abort) = 1;
        return false;
      }
    }
  }
}

template <int kN>
HSA_DEVINL void write_result(const AttnParams& p, int b, int g, int s, int h, int dv, float o) {
  const int64_t head = static_cast<int64_t>(b) * p.Hq + g * p.HG + h;
  if (p.S == 1) {
    if (p.out_dtype == HSA_BF16)
      reinterpret_cast<__nv_bfloat16*>(p.out)[head * p.Dv + dv] = __float2bfloat16_rn(o);
    else
      reinterpret_cast<float*>(p.out)[head * p.Dv + dv] = o;
  } else {
    p.po[((static_cast<int64_t>(b) * p.S + s) * p.Hq + g * p.HG + h) * p.Dv + dv] = o;
  }
}

HSA_DEVINL void write_lse(const AttnParams& p, int b, int g, int s, int h, float v) {
  if (p.S == 1) {
    if (p.lse) p.lse[static_cast<int64_t>(b) * p.Hq + g * p.HG + h] = v;
  } else {
    p.plse[(static_cast<int64_t>(b) * p.S + s) * p.Hq + g * p.HG + h] = v;
  }
}

template <int kN>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % p.G;
  const int s = (blockIdx.x / p.G) % p.S;
  const int b = blockIdx.x / (p.G * p.S);
  const int NSL = p.Dqk / 64, NV = p.Dv / 64, NMT = p.Dv / 128;
  const SeqGeom geo = seq_geom(p, b);
  const int64_t n_slots = geo.n_swa + geo.n_extra;
  const int n_tiles = static_cast<int>((n_slots + kKeys - 1) / kKeys);
  const int t0 = s * p.tps;
  const int t1 = min(t0 + p.tps, n_tiles);
  const int nt = t1 - t0;

  if (nt <= 0) {  // nothing to attend in this split
    if (tid < kKeys) {
      if (p.S == 1)
        for (int h = 0; h < p.HG; ++h)
          for (int dv = tid; dv < p.Dv; dv += kKeys) write_result<kN>(p, b, g, s, h, dv, 0.f);
      if (tid < p.HG) write_lse(p, b, g, s, tid, -INFINITY);
    }
    return;
  }
  if (p.extra && !p.idx && geo.nb > p.max_rows && tid == 0 && s == 0 && g == 0)
    set_status(p.status, HSA_DEV_BOUNDS);

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t qslice = kN * 128;          // bytes of one Q slice (kN heads x 64 ch)
  const uint32_t pbytes = 2 * kN * 128;      // one P^T buffer (2 K-blocks of 64 keys)
  uint8_t* kbuf = smem;
  uint8_t* qs = kbuf + NSL * kSliceBytes;
  uint8_t* pt = qs + NSL * qslice;
  // TMEM columns: S^T of tile parity sb, partial accumulator a at (sb*4 + a)*kN;
  // O^T M-tile m at (8 + m)*kN.
  const uint32_t tmem_cols_needed = 8 * kN + NMT * kN;
  uint32_t tmem_cols = 32;
  while (tmem_cols < tmem_cols_needed) tmem_cols <<= 1;

  if (tid == 0) {
    for (int j = 0; j < NSL; ++j) {
      tc::mbar_init(&sh.full[j], kProdThreads);
      tc::mbar_init(&sh.empty[j], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh.s_full[i], 1);
      tc::mbar_init(&sh.s_empty[i], kKeys);
      tc::mbar_init(&sh.o_done[i], 1);
    }
    tc::mbar_init(&sh.p_full, kKeys);
    tc::mbar_init(&sh.q_full, kProdThreads);
    tc::mbar_init(&sh.fin, 1);
    sh.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&sh.tmem, tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem;

  if (warp >= kProdWarp0) {
    // ------------------------------------------------------------ producers
    const int pt_ = tid - kProdWarp0 * 32;
    const int nq = kN * NSL * 8;
    for (int i = pt_; i < nq; i += kProdThreads) {
      const int h = i / (NSL * 8), rem = i - h * NSL * 8, j = rem >> 3, c = rem & 7;
      const bool v = h < p.HG;
      const uint16_t* src =
          v ? p.q + (static_cast<int64_t>(b) * p.Hq + g * p.HG + h) * p.Dqk + j * 64 + c * 8 : p.q;
      tc::cp_async16(qs + j * qslice + sw128(h, c), src, v ? 16u : 0u);
    }
    tc::cp_async_commit();
    tc::cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(&sh.q_full);

    int64_t issued = 0, retired = 0;
    auto retire_to = [&](int keep) {
      if (issued - retired > keep) {
        tc::cp_async_wait_dyn(keep);
        tc::fence_proxy_async_smem();
        while (issued - retired > keep) {
          tc::mbar_arrive(&sh.full[slice_order(static_cast<int>(retired % NSL), NSL, NV)]);
          ++retired;
        }
      }
    };
    auto build_table = [&](int t) {
      const uint16_t** table = sh.rows[(t - t0) & 1];
      for (int r = pt_; r < kKeys; r += kProdThreads)
        table[r] = slot_row(p, b, geo, static_cast<int64_t>(t) * kKeys + r, true);
    };
    bool ok = true;
    build_table(t0);
    tc::named_barrier(2, kProdThreads);
    for (int t = t0; t < t1; ++t) {
      const int tt = t - t0;
      const uint16_t* const* table = sh.rows[tt & 1];
      for (int jj = 0; jj < NSL && ok; ++jj) {
        const int j = slice_order(jj, NSL, NV);
        // Buffer j is freed by the consumption of tile tt-1, whose slices were
        // all signalled before this tile began, so blocking here while this
        // tile's own slices are still in flight cannot stall the MMA.
        if (tt > 0 && !wait_or_abort(sh, &sh.empty[j], (tt - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        uint8_t* base = kbuf + j * kSliceBytes;
        for (int q = pt_; q < kKeys * 8; q += kProdThreads) {
          const int r = q >> 3, c = q & 7;
          const uint16_t* row = table[r];
          tc::cp_async16(base + sw128(r, c), row ? row + j * 64 + c * 8 : p.q, row ? 16u : 0u);
        }
        tc::cp_async_commit();
        ++issued;
      }
      // the next tile's rows (index loads) overlap this tile's copies; then every
      // slice of this tile is signalled before the producer can block again
      if (t + 1 < t1 && ok) build_table(t + 1);
      retire_to(0);
      if (tc::named_barrier_or(2, kProdThreads, !ok)) break;  // table visible; agree on abort
    }
    retire_to(0);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16_f32(kKeys, kN);
      const uint32_t idO = tc::idesc_bf16_f32(kKeys, kN, /*a_mn=*/true, /*b_mn=*/false);
      bool ok = wait_or_abort(sh, &sh.q_full, 0, p.status);
      for (int t = t0; t < t1 && ok; ++t) {
        const int tt = t - t0, sb = tt & 1;
        if (tt >= 2 && !wait_or_abort(sh, &sh.s_empty[sb], ((tt - 2) >> 1) & 1, p.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // Four independent partial accumulators (by K-step within a slice) keep
        // these small MMAs from waiting on each other's accumulation.
        const uint32_t d_s = tmem + sb * 4 * kN;
        for (int jj = 0; jj < NSL && ok; ++jj) {
          const int j = slice_order(jj, NSL, NV);
          if (!wait_or_abort(sh, &sh.full[j], tt & 1, p.status)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t ka = tc::smem_u32(kbuf + j * kSliceBytes);
          const uint32_t qa = tc::smem_u32(qs + j * qslice);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = tc::smem_desc(ka + ks * 32, 16, 1024, tc::kSwizzle128B);
            const uint64_t bq = tc::smem_desc(qa + ks * 32, 16, 1024, tc::kSwizzle128B);
            tc::mma_bf16(d_s + ks * kN, a, bq, idS, jj != 0);
          }
          if (j >= NV) tc::mma_commit(&sh.empty[j]);
        }
        if (!ok) break;
        tc::mma_commit(&sh.s_full[sb]);
        if (!wait_or_abort(sh, &sh.p_full, tt & 1, p.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t pa = tc::smem_u32(pt + sb * pbytes);
        // M-tiles are independent accumulators: interleave them
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t bp =
              tc::smem_desc(pa + (kk >> 2) * kN * 128 + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
          for (int m = 0; m < NMT; ++m) {
            const uint32_t va = tc::smem_u32(kbuf + 2 * m * kSliceBytes);
            const uint64_t a = tc::smem_desc(va + kk * 2048, kSliceBytes, 1024, tc::kSwizzle128B);
            tc::mma_bf16(tmem + (8 + m) * kN, a, bp, idO, (tt > 0 || kk > 0) ? 1u : 0u);
          }
        }
        for (int j = 0; j < NV; ++j) tc::mma_commit(&sh.empty[j]);
        tc::mma_commit(&sh.o_done[sb]);
      }
      // drain: every MMA this thread issued has completed before TMEM is freed
      tc::mma_commit(&sh.fin);
      tc::mbar_wait(&sh.fin, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float l_part[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) l_part[h] = 0.f;
    if (tid < kN) sh.m[tid] = -INFINITY;
    bool ok = true;
    for (int t = t0; t < t1; ++t) {
      const int tt = t - t0, sb = tt & 1;
      const bool valid = slot_row(p, b, geo, static_cast<int64_t>(t) * kKeys + tid, false) != nullptr;
      {
        const bool failed = !wait_or_abort(sh, &sh.s_full[sb], (tt >> 1) & 1, p.status);
        if (tc::named_barrier_or(1, kKeys, failed)) { ok = false; break; }
      }
      tc::fence_after_sync();
      __syncwarp();
      float sacc[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) sacc[h] = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
#pragma unroll
        for (int half = 0; half < kN / 16; ++half) {
          uint32_t raw[16];
          tc::tmem_ld16(tmem + lane_base + (sb * 4 + a) * kN + half * 16, raw);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) sacc[half * 16 + i] += __uint_as_float(raw[i]);
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&sh.s_empty[sb]);
      float x[kN], mx[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        x[h] = valid ? sacc[h] * p.scale_log2 : -INFINITY;
        mx[h] = x[h];
      }
      const float mcol = warp_transpose_reduce<kN, true>(mx);
      if (lane < kN) sh.red[warp][lane] = mcol;
      tc::named_barrier(1, kKeys);
      bool moved = false;
      if (tid < kN) {
        const float mt =
            fmaxf(fmaxf(sh.red[0][tid], sh.red[1][tid]), fmaxf(sh.red[2][tid], sh.red[3][tid]));
        const float mo = sh.m[tid];
        const float mn = fmaxf(mo, mt);
        moved = mn > mo + kRescaleLog2;
        sh.alpha[tid] = moved ? exp2f(mo - mn) : 1.f;
        if (moved) sh.m[tid] = mn;
      }
      const bool any = tc::named_barrier_or(1, kKeys, moved);
      if (any) {
#pragma unroll
        for (int h = 0; h < kN; ++h) l_part[h] *= sh.alpha[h];
        if (tt > 0) {
          const bool failed =
              !wait_or_abort(sh, &sh.o_done[(tt - 1) & 1], ((tt - 1) >> 1) & 1, p.status);
          if (tc::named_barrier_or(1, kKeys, failed)) { ok = false; break; }
          tc::fence_after_sync();
          __syncwarp();
          for (int m = 0; m < NMT; ++m) {
            const uint32_t col = tmem + lane_base + (8 + m) * kN;
#pragma unroll
            for (int half = 0; half < kN / 16; ++half) {
              uint32_t o[16];
              tc::tmem_ld16(col + half * 16, o);
              tc::tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                o[i] = __float_as_uint(__uint_as_float(o[i]) * sh.alpha[half * 16 + i]);
              tc::tmem_st16(col + half * 16, o);
            }
          }
          tc::tmem_st_wait();
        }
      }
      if (tt >= 2) {  // P^T buffer sb is free once O^T of tile tt-2 has completed
        const bool failed = !wait_or_abort(sh, &sh.o_done[sb], ((tt - 2) >> 1) & 1, p.status);
        if (tc::named_barrier_or(1, kKeys, failed)) { ok = false; break; }
      }
      float mreg[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) mreg[h] = sh.m[h];
      uint32_t pk[kN / 2];
#pragma unroll
      for (int h = 0; h < kN; h += 2) {
        const float p0 = mreg[h] == -INFINITY ? 0.f : tc::ex2_approx(x[h] - mreg[h]);
        const float p1 = mreg[h + 1] == -INFINITY ? 0.f : tc::ex2_approx(x[h + 1] - mreg[h + 1]);
        const __nv_bfloat162 q2 = __floats2bfloat162_rn(p0, p1);
        l_part[h] += __low2float(q2);
        l_part[h + 1] += __high2float(q2);
        pk[h / 2] = *reinterpret_cast<const uint32_t*>(&q2);
      }
      uint8_t* ptb = pt + sb * pbytes + (tid >> 6) * kN * 128;
      const int kc = (tid & 63) >> 3, ke = (tid & 7) << 1;
#pragma unroll
      for (int h = 0; h < kN; ++h)
        *reinterpret_cast<uint16_t*>(ptb + (h >> 3) * 1024 + (h & 7) * 128 + ((kc ^ (h & 7)) << 4) +
                                     ke) = static_cast<uint16_t>(pk[h / 2] >> ((h & 1) * 16));
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(&sh.p_full);
    }
    {
      // `ok` is uniform over the softmax warps here (every exit from the loop
      // went through an agreement barrier)
      bool failed = !ok;
      if (!failed) failed = !wait_or_abort(sh, &sh.o_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, p.status);
      ok = !tc::named_barrier_or(1, kKeys, failed);
    }
    // every softmax thread reaches these barriers, whether or not it aborted
    const float lcol = warp_transpose_reduce<kN, false>(l_part);
    if (lane < kN) sh.red[warp][lane] = lcol;
    tc::named_barrier(1, kKeys);
    if (tid < kN) sh.bc[tid] = (sh.red[0][tid] + sh.red[1][tid]) + (sh.red[2][tid] + sh.red[3][tid]);
    tc::named_barrier(1, kKeys);
    if (ok) {
      tc::fence_after_sync();
      __syncwarp();
      float inv[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) inv[h] = sh.bc[h] > 0.f ? 1.f / sh.bc[h] : 0.f;
      for (int m = 0; m < NMT; ++m) {
        const uint32_t col = tmem + lane_base + (8 + m) * kN;
        uint32_t acc[kN];
        tc::tmem_ld16(col, acc);
        if (kN == 32) tc::tmem_ld16(col + 16, acc + (kN == 32 ? 16 : 0));
        tc::tmem_ld_wait();
        const int dv = m * kKeys + tid;
#pragma unroll
        for (int h = 0; h < kN; ++h)
          if (h < p.HG) write_result<kN>(p, b, g, s, h, dv, __uint_as_float(acc[h]) * inv[h]);
      }
      if (tid < p.HG) {
        const float mh = sh.m[tid];
        const float l = sh.bc[tid];
        write_lse(p, b, g, s, tid, l > 0.f ? (mh + log2f(l)) * 0.69314718055994531f : -INFINITY);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

// Merges the split partials: o = sum_s e^(lse_s - lse) o_s, lse = log sum_s e^lse_s.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ po,
                                                          const float* __restrict__ plse, int S,
                                                          int Hq, int Dv, void* out, int out_dtype,
                                                          float* lse) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const float* ls = plse + static_cast<int64_t>(b) * S * Hq + h;
  float mx = -INFINITY;
  for (int s = 0; s < S; ++s) mx = fmaxf(mx, ls[static_cast<int64_t>(s) * Hq]);
  float tot = 0.f;
  for (int s = 0; s < S; ++s) {
    const float l = ls[static_cast<int64_t>(s) * Hq];
    if (l > -INFINITY) tot += __expf(l - mx);
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  const int64_t head = static_cast<int64_t>(b) * Hq + h;
  for (int dv = threadIdx.x; dv < Dv; dv += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float l = ls[static_cast<int64_t>(s) * Hq];
      if (l > -INFINITY)
        acc += __expf(l - mx) * po[((static_cast<int64_t>(b) * S + s) * Hq + h) * Dv + dv];
    }
    const float o = acc * inv;
    if (out_dtype == HSA_BF16)
      reinterpret_cast<__nv_bfloat16*>(out)[head * Dv + dv] = __float2bfloat16_rn(o);
    else
      reinterpret_cast<float*>(out)[head * Dv + dv] = o;
  }
  if (threadIdx.x == 0 && lse) lse[head] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

}  // namespace

AttnPlan attn_plan(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W, int64_t extra_slots) {
  AttnPlan pl;
  pl.HG = static_cast<int>(Hq <= 32 ? Hq : 32);
  pl.N = pl.HG <= 16 ? 16 : 32;
  pl.G = static_cast<int>(Hq / pl.HG);
  const int64_t slots = W + extra_slots;
  const int64_t tiles = slots > 0 ? (slots + kKeys - 1) / kKeys : 1;
  int64_t S = device_sms() / (B * pl.G);
  if (S < 1) S = 1;
  if (S > tiles) S = tiles;
  pl.tps = static_cast<int>((tiles + S - 1) / S);
  pl.S = static_cast<int>((tiles + pl.tps - 1) / pl.tps);
  const int NSL = static_cast<int>(Dqk / 64);
  pl.smem = static_cast<size_t>(NSL) * kSliceBytes + static_cast<size_t>(NSL) * pl.N * 128 +
            2 * 2 * pl.N * 128 + 1024;
  // keep co-resident CTAs within the SM's 512 TMEM columns
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(8 * pl.N + (Dv / 128) * pl.N)) cols <<= 1;
  // (at most n = 512 / cols CTAs fit the TMEM, so shared memory must keep
  // n + 1 of them from being resident together)
  const size_t per_sm = 227 * 1024;
  const size_t floor_bytes = per_sm / (512 / cols + 1) + 1;
  if (pl.smem < floor_bytes) pl.smem = floor_bytes;
  return pl;
}

size_t attn_workspace_bytes(const AttnPlan& pl, int64_t B, int64_t Hq, int64_t Dv) {
  size_t bytes = kWsHeader;
  if (pl.S > 1) {
    bytes += (static_cast<size_t>(B) * pl.S * Hq * Dv * 4 + 255) & ~size_t(255);
    bytes += (static_cast<size_t>(B) * pl.S * Hq * 4 + 255) & ~size_t(255);
  }
  return bytes;
}

cudaError_t launch_attn(const AttnArgs& a, const AttnPlan& pl, void* ws, uint32_t* status,
                        cudaStream_t stream, bool pdl) {
  AttnParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.swa = static_cast<const uint16_t*>(a.swa);
  p.seq_len = a.seq_len;
  p.len_add = a.len_add;
  p.W = static_cast<int>(a.W);
  p.extra = static_cast<const uint16_t*>(a.extra);
  p.sp = a.sp;
  p.idx = a.idx;
  p.k = static_cast<int>(a.k);
  p.max_rows = a.max_rows;
  p.B = static_cast<int>(a.B);
  p.Hq = static_cast<int>(a.Hq);
  p.Dqk = static_cast<int>(a.Dqk);
  p.Dv = static_cast<int>(a.Dv);
  p.HG = pl.HG;
  p.G = pl.G;
  p.S = pl.S;
  p.tps = pl.tps;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = a.out;
  p.out_dtype = a.out_dtype;
  p.lse = a.lse;
  p.status = status;
  char* w = static_cast<char*>(ws) + kWsHeader;
  p.po = reinterpret_cast<float*>(w);
  p.plse = reinterpret_cast<float*>(
      w + ((static_cast<size_t>(a.B) * pl.S * a.Hq * a.Dv * 4 + 255) & ~size_t(255)));
  const unsigned grid = static_cast<unsigned>(a.B * pl.G * pl.S);
  auto* kernel = pl.N == 16 ? attn_kernel<16> : attn_kernel<32>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(pl.smem));
  if (e != cudaSuccess) return e;
  e = launch_k(kernel, dim3(grid), dim3(kThreads), pl.smem, stream, pdl, p);
  if (e != cudaSuccess || pl.S == 1) return e;
  return launch_k(attn_combine_kernel, dim3(static_cast<unsigned>(a.B * a.Hq)), dim3(128), 0, stream,
                  true, static_cast<const float*>(p.po), static_cast<const float*>(p.plse), pl.S,
                  p.Hq, p.Dv, a.out, a.out_dtype, a.lse);
}

}  // namespace hsa
