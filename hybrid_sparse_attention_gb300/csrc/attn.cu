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
// Design (sm_103a).  The kernel is bound by how fast each SM can gather key
// rows, so it keeps that gather streaming and reads every row once per
// sequence (all heads of a token in one CTA, up to 64):
//  * Keys are the M = 128 side of both contractions, so a gathered block of
//    128 key rows feeds both MMAs without re-layout:
//      S^T[key, head] = K_tile . Q^T      (A = K, K-major over Dqk)
//      O^T[dv, head] += V_tile^T . P^T    (A = the same rows, MN-major view)
//  * Rows arrive through a ring of four 32 KB pair slots (two 64-channel
//    slices of 128 rows each, 128-byte swizzled, 16 KB apart = the MN-major
//    leading-byte offset), filled by three gather warps with 16-byte
//    cp.async (each keeps up to two of its items in flight) and drained by
//    one MMA-issuing thread.  Q (needed by pass 1 only) shares its region
//    with the odd tiles' P^T buffer; the even tiles' P^T buffer has its own
//    (it is written while the chunk's pass 1 may still read Q).
//  * A token's slots are split over S CTAs in whole 128-slot tiles.
//  * Two passes per chunk of up to four 128-slot tiles: pass 1 streams all
//    Dqk channels of the chunk's tiles into S^T accumulators (one per tile,
//    in TMEM); as each tile's S^T lands the softmax warps fold its maximum
//    into the running maximum and write its P^T (online softmax; the running
//    maximum moves lazily, only by more than 2^8, and O^T and l are then
//    rescaled), and pass 2 streams the value channels again (now from L2)
//    into O^T against P^T.
//  * Long key lists are split over CTAs.  Two to four splits of a token form
//    one thread-block cluster and merge through distributed shared memory;
//    with more, each split writes an fp32 partial output and log-sum-exp that
//    a combine kernel merges.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "select_core.cuh"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kKeys = 128;
constexpr int kSmWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;
constexpr int kProdThreads = 96;
constexpr int kThreads = 32 * 8;    // (9 warps would cap registers at 168 per thread)
constexpr int kRing = 4;            // pair slots
constexpr int kMaxTC = 4;           // tiles per chunk
constexpr uint32_t kSliceBytes = kKeys * 128;
constexpr uint32_t kPairBytes = 2 * kSliceBytes;
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxCl = 4;           // splits merged inside one cluster
constexpr uint32_t kUnitBytes = kKeys * 16 * 4;  // one merge unit: 128 lanes x 16 fp32 columns
static_assert(16 * kUnitBytes <= kRing * kPairBytes, "the units a split receives fit its ring");
constexpr size_t kMergeScratch = 8 * 2 * 16 * 32 * 4;  // eight warps' two 16 x 32 fp32 transpose tiles

// Dynamic shared memory after the ring: the Q region (Q during pass 1; then
// the odd tiles' P^T buffer; at the end the merge's transpose tiles), then the
// even tiles' P^T buffer, which is never part of Q (it is written while the
// chunk's pass 1 may still read Q).
__host__ __device__ inline uint32_t attn_q_region(int NSL, int N) {
  const uint32_t q = static_cast<uint32_t>(NSL) * N * 128, pb = 2u * N * 128;
  uint32_t r = q > pb ? q : pb;
  return r > kMergeScratch ? r : static_cast<uint32_t>(kMergeScratch);
}

struct AttnParams {
  const uint16_t* q;      // [B, Hq, Dqk] (B tokens)
  const uint16_t* swa;    // [B / T, Wr, Dqk] window rings
  const int32_t* seq_len; // [B / T]
  int32_t len_add;
  int W;                  // window rows attended
  int T;                  // query tokens per sequence: token b is token b % T of sequence b / T
  int Wr;                 // ring rows (slot = position mod Wr)
  const uint16_t* extra;  // compressed pool rows (may be null)
  Spans sp;
  const int32_t* idx;     // [B, k] or null (dense)
  int k;
  int64_t max_rows;       // dense: cap on compressed rows per sequence
  int B, Hq, Dqk, Dv;
  int HG, G, S, TC;
  int64_t sps;            // attended slots per split
  float scale_log2;
  void* out;
  int out_dtype;
  float* lse;
  float* po;              // partial outputs [B, S, Hq, Dv] (S > 1)
  float* plse;            // partial lse [B, S, Hq] (S > 1)
  uint32_t* status;
  int early;              // 1: the previous kernel writes only idx; 2: it is the append (see AttnArgs)
  int cl;                 // the S splits form a cluster and merge in shared memory
  // Fused selection (the layer's C4 path; sel_scores != null): idx is null and
  // the last split of every token selects the token's top-k itself from the
  // indexer's scores and per-row key histogram (see select_token).
  const float* sel_scores;  // scores at the pool's row positions
  uint32_t* row_hist;       // [B, kRowHistBins], zeroed again by the selection
  uint64_t* cand_ws;        // heavy-tie candidates, at the pool's row positions
  int32_t* topk_out;        // [B, k] the selection in order (may be null)
};

// Token b's geometry: its sequence bs, window length L (the token's own
// position + 1), pool start off, live compressed rows nb and the start soff of
// its score / candidate rows (off + t * the per-token stride).
struct SeqGeom {
  int64_t L, off, nb, soff;
  int bs;
  int n_swa;
  int64_t n_extra;
};

HSA_DEVINL SeqGeom seq_geom(const AttnParams& p, int b) {
  SeqGeom g;
  g.bs = p.T == 1 ? b : b / p.T;
  int64_t L = static_cast<int64_t>(p.seq_len[g.bs]) + p.len_add + (p.T == 1 ? 0 : b % p.T);
  g.L = L < 0 ? 0 : L;
  g.n_swa = static_cast<int>(g.L < p.W ? g.L : p.W);
  g.off = 0;
  g.soff = 0;
  g.nb = 0;
  g.n_extra = 0;
  if (p.extra) {
    g.off = p.sp.pool_start(b);
    g.soff = p.sp.start(b);
    g.nb = p.sp.count(b);
    if (p.idx || p.sel_scores) {
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
    return p.swa + (static_cast<int64_t>(g.bs) * p.Wr + pos % p.Wr) * p.Dqk;
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

// slot_row with the list entry for `slot` already loaded (j; ignored for
// window slots and dense lists).
HSA_DEVINL const uint16_t* slot_row_j(const AttnParams& p, int b, const SeqGeom& g, int64_t slot,
                                      int64_t j, bool report) {
  if (slot < g.n_swa) {
    const int64_t pos = g.L - g.n_swa + slot;
    return p.swa + (static_cast<int64_t>(g.bs) * p.Wr + pos % p.Wr) * p.Dqk;
  }
  const int64_t e = slot - g.n_swa;
  if (e >= g.n_extra) return nullptr;
  if (!p.idx && !p.sel_scores) j = e;
  if (j < 0) return nullptr;
  if (j >= g.nb) {
    if (report) set_status(p.status, HSA_DEV_BOUNDS);
    return nullptr;
  }
  return p.extra + (g.off + j) * p.Dqk;
}

// List entry of slot `slot` (0 when the slot is a window slot or past the list).
HSA_DEVINL int64_t slot_index(const AttnParams& p, int b, const SeqGeom& g, int64_t slot) {
  const int64_t e = slot - g.n_swa;
  return (p.idx && e >= 0 && e < g.n_extra) ? static_cast<int64_t>(p.idx[static_cast<int64_t>(b) * p.k + e])
                                             : 0;
}

// 16-byte asynchronous copy issued only when `pred` (predicated, no branch).
HSA_DEVINL void cp_async16_if(uint32_t dst, const void* src, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t"
      "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(dst),
      "l"(src), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

// Column reduction of a 32 x 32 register tile held one row per lane: on
// return lane l holds the reduction of column l over the warp.
template <bool kMax>
HSA_DEVINL float warp_transpose_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int width = 16; width >= 1; width >>= 1) {
    const bool upper = (lane & width) != 0;
#pragma unroll
    for (int i = 0; i < width; ++i) {
      const float send = upper ? v[i] : v[i + width];
      const float keep = upper ? v[i + width] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, width);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

struct Shared {
  uint64_t full[kRing], empty[kRing];
  uint64_t s_full[kMaxTC], s_empty;  // S^T of chunk tile tc written; S^T columns free again
  uint64_t p_full[2], o_done[2];     // P^T buffer written; O^T of that buffer's tile done
  uint64_t q_full, fin;
  uint32_t tmem;
  int abort;
  float red[kSmWarps][64];  // softmax: per-warp column reductions; merge: every split's weight
  float m[64];      // running maximum per head (log2 units), identical for every thread
  float alpha[64];  // rescale factor of the current chunk per head
  float inv[64];    // 1 / softmax denominator per head (0 when nothing was attended)
  float l[64];      // softmax denominator per head (relative to m)
  float xm[kMaxCl][64], xl[kMaxCl][64];  // cluster merge: every split's m and l
  int xok[kMaxCl];  // cluster merge: the split has a partial output
  int done_ok;      // the softmax warps finished without an abort: O^T may be written out
  const uint16_t* rows[kMaxTC][kKeys];  // gather tables of the producers (this chunk)
  // fused selection: this split's share of the token's selected entries
  // (row-local indices, 0xffff past the selection), their total, and the
  // barrier the selecting split arrives on once both are written
  alignas(16) uint16_t sel[kMaxTC * kKeys];
  uint32_t sel_n;
  uint64_t sel_full;
  uint64_t sel_cp;  // the selecting split's copy of its row's scores landed
};
static_assert(kKeys * kMaxTC >= 512, "a split's share of a fused selection (k <= 512) fits");

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

// ---------------------------------------------------------------- fused selection
//
// In the layer's C4 path the token's last split selects the token's top-k
// itself, after the indexer, from its scores and from the per-row histogram
// of the top kRowHistBits order-key bits that the indexer built while writing
// them (Lightning TopK: [KD] §Arquitectura del Sistema; [WK] §推理侧优化).  It
// finds the threshold bin d (fewer than k scores above it, at least k at or
// above it), keeps the scores above bin d and in it in one pass over the row,
// sorts those survivors by composite (value descending, lower index first) and
// takes the first k: the same list, in the same order, as the standalone
// top-k.  The other splits of the token attend the rows that need no
// selection (the window) meanwhile, and wait for the selecting split to write
// their share of the list into their shared memory.

constexpr int kSelRowMax = 32768;  // scores per row the fused selection handles
static_assert(kRing * kPairBytes >= 4 * kSelRowMax, "a selected row's scores fit the ring");
static_assert(kRowHistBins % (4 * kThreads) == 0, "whole 16-byte histogram loads per thread");
constexpr int kSelMax = 2048;      // composites of the selection's shared-memory buffer
constexpr int kSelSort = 1024;     // winners + candidates held in shared memory, at most
constexpr int kSelRank = 512;      // candidates ranked by counting, at most
constexpr int kSelMaxK = 512;      // k the fused selection handles

// Asynchronous 4-byte store to cluster shared memory whose completion counts
// its bytes on the barrier at cluster address `bar` (same CTA as `addr`).
HSA_DEVINL void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(v), "r"(bar)
               : "memory");
}

// Bounded wait (acquire, cluster scope) for the barrier's phase `parity`;
// also gives up when another role has aborted.
HSA_DEVINL bool wait_cluster_or_abort(int* abort, uint64_t* bar, uint32_t parity, uint32_t* status) {
  const uint32_t a = tc::smem_u32(bar);
  const uint64_t t0 = tc::global_timer();
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 63u) == 63u) {
      if (*reinterpret_cast<volatile int*>(abort)) return false;
      if (tc::global_timer() - t0 > tc::kSpinNanos || i > tc::kSpinPolls) {
        set_status(status, HSA_DEV_TIMEOUT);
        *reinterpret_cast<volatile int*>(abort) = 1;
        return false;
      }
    }
  }
}

// First C4 entry of split q's share of a token's selection.
HSA_DEVINL int64_t share_first(const AttnParams& p, int n_swa, int q) {
  const int64_t e = static_cast<int64_t>(q) * p.sps - n_swa;
  return e < 0 ? 0 : (e > p.k ? p.k : e);
}

// Bytes the selecting split stores into split q's shared memory: q's share
// of the list as 16-bit entries in 4-byte pairs, and the list's length.
HSA_DEVINL uint32_t sel_bytes(const AttnParams& p, int n_swa, int q) {
  const int64_t e1 = q + 1 < p.S ? share_first(p, n_swa, q + 1) : p.k;
  return 4u * static_cast<uint32_t>((e1 - share_first(p, n_swa, q) + 1) >> 1) + 4u;
}


// 4-byte asynchronous global -> shared copy (any 4-byte-aligned source).
HSA_DEVINL void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src)
               : "memory");
}

// Selects token b's top-k and hands every split of the token its share (every
// thread of the CTA calls it; the ring and `sbuf` (kSelMax composites) are
// free scratch).  n: the row's live scores (at most kSelRowMax); rank: this
// CTA's rank in the token's cluster.  No step appends through a shared
// counter: survivors get their places from one block-wide scan of per-thread
// counts, and candidates are chosen by counting ranks, so every step is a few
// block-wide phases whatever the row holds.  The list the splits attend is in
// a fixed order (not sorted by value); its sorted copy, when asked for, is
// written at the end of the kernel (write_topk_sorted).
HSA_DEVINL void select_token(const AttnParams& p, Shared& sh, uint8_t* ring, uint64_t* sbuf, int b,
                             const SeqGeom& g, int n, uint32_t rank) {
  __shared__ uint32_t s_scan[33], s_out[3], s_cnt;
  __shared__ __align__(16) uint32_t s_hbins[kRowHistBins / kThreads];
  const int t = threadIdx.x;
  uint32_t* s_row = reinterpret_cast<uint32_t*>(ring);  // [kSelRowMax] score bits
  const uint32_t kk = static_cast<uint32_t>(n < p.k ? n : p.k);
  const bool all = n <= p.k;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(p.sel_scores + g.soff);
  // Loops stay rolled throughout: this code runs once per launch, and its
  // instruction fetches cost more than loop overhead.
  // (1) the row's scores to shared memory, every copy in flight at once: the
  // 16-byte-aligned body to s_row[0, 4 nv), then the at most 3 + 3 scores
  // before and after it; and the sum of this thread's kPer bins of the row's
  // histogram (bins counted from the top bin down)
  constexpr int kPer = kRowHistBins / kThreads;
  const int lo = kRowHistBins - kPer * (t + 1);  // this thread's bins: [lo, lo + kPer)
  uint4* gh = reinterpret_cast<uint4*>(p.row_hist + static_cast<int64_t>(b) * kRowHistBins + lo);
  const int head = static_cast<int>(
      min(static_cast<uintptr_t>(n), ((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) >> 2));
  const int nv = (n - head) >> 2, body = 4 * nv;
  if (t == 0 && nv > 0) {  // the body: bulk copies (32 KB each) completing on sel_cp
    const uint32_t bytes = 16u * static_cast<uint32_t>(nv);
    tc::mbar_arrive_expect_tx(&sh.sel_cp, bytes);
#pragma unroll 1
    for (uint32_t o = 0; o < bytes; o += 32768u)
      tc::bulk_load(reinterpret_cast<uint8_t*>(s_row) + o, reinterpret_cast<const uint8_t*>(row + head) + o,
                    bytes - o < 32768u ? bytes - o : 32768u, &sh.sel_cp);
  }
#pragma unroll 1
  for (int j = t; j < n - body; j += kThreads) cp_async4(s_row + body + j, row + (j < head ? j : body + j));
  tc::cp_async_commit();
  uint4 hv[kPer / 4];  // this thread's bins, kept for the threshold search
#pragma unroll
  for (int i = 0; i < kPer / 4; ++i) hv[i] = __ldcg(gh + i);
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < kPer / 4; ++i) sum += (hv[i].x + hv[i].y) + (hv[i].z + hv[i].w);
  // (2) the threshold bin d: fewer than kk scores above it, at least kk at or
  // above it.  One scan of the per-thread sums finds the thread whose bins
  // hold it; that thread hands its bins to warp 0 (shared memory), which
  // scans them.
  uint32_t d = 0;
  if (!all) {
    uint32_t total;
    const uint32_t a = block_inclusive_sum<uint32_t>(sum, s_scan, &total) - sum;
    if (a < kk && a + sum >= kk) {
      uint4* hb = reinterpret_cast<uint4*>(s_hbins);
#pragma unroll
      for (int i = 0; i < kPer / 4; ++i) hb[i] = hv[i];
      s_out[0] = static_cast<uint32_t>(lo);
      s_out[1] = a;
    }
    __syncthreads();
    if (t < 32) {
      const uint32_t blo = s_out[0], above = s_out[1];
      const uint32_t cnt = s_hbins[kPer - 1 - t];  // lane 0: the range's top bin
      uint32_t incl = cnt;
#pragma unroll 1
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (t >= o) incl += y;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, above + incl >= kk);
      if (t == 0) s_out[2] = blo + kPer - 1 - (hit ? __ffs(hit) - 1 : 0);
    }
    __syncthreads();
    d = s_out[2];
  }
  // the histogram is zeroed again for the next step
#pragma unroll
  for (int i = 0; i < kPer / 4; ++i) gh[i] = make_uint4(0u, 0u, 0u, 0u);
  tc::cp_async_wait<0>();
  if (nv > 0) tc::mbar_wait(&sh.sel_cp, 0, p.status);
  __syncthreads();
  // (3) winners (above bin d; every score when all) and candidates (in bin d).
  // One pass classifies every score and keeps, per thread, masks of its
  // winners and candidates (kGrp slots per group, at most kGroups groups) and
  // their counts; one scan gives every thread its places; the second pass
  // visits only the masked slots.  Slot s of s_row holds row entry idx(s).
  // Group gi covers slots [gi * kThreads * kGrp, (gi + 1) * kThreads * kGrp);
  // thread t reads its 16-byte chunks gi * (kGrp / 4) * kThreads + q * kThreads
  // + t (consecutive lanes, consecutive chunks).
  constexpr int kGrp = 16;                              // slots per thread per group
  constexpr int kGroups = kSelRowMax / (kThreads * kGrp);
  auto slot_of = [&](int gi, int bit) { return ((gi * (kGrp / 4) + (bit >> 2)) * kThreads + t) * 4 + (bit & 3); };
  // Float compares against the bins' first scores (bar_float): winners lie at
  // or above bin d + 1's, candidates at or above bin d's and below; NaN
  // scores pass neither and are caught by a NaN-propagating max.
  const float fw = all ? -INFINITY
                       : (d + 1 < static_cast<uint32_t>(kRowHistBins)
                              ? bar_float((d + 1) << kRowHistShift)
                              : __uint_as_float(0x7fffffffu));  // (top bin: no winners)
  const float fc = all ? -INFINITY : bar_float(d << kRowHistShift);
  float nanacc = 0.0f;
  uint32_t wmask[kGroups], cmask[kGroups];
  uint32_t cnt = 0;
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {
    wmask[gi] = cmask[gi] = 0u;
    if (gi * kThreads * kGrp >= n) continue;      // (uniform)
    const bool whole = (gi + 1) * kThreads * kGrp <= n;  // (uniform)
#pragma unroll
    for (int q4 = 0; q4 < kGrp / 4; ++q4) {
      const float4 w = reinterpret_cast<const float4*>(s_row)[(gi * (kGrp / 4) + q4) * kThreads + t];
      const float f4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int bit = 4 * q4 + e;
        const bool in = whole || slot_of(gi, bit) < n;
        const bool win = f4[e] >= fw, cand = !win && f4[e] >= fc;
        nanacc = max_nan(nanacc, in ? f4[e] : 0.0f);
        wmask[gi] |= (in && win ? 1u : 0u) << bit;
        cmask[gi] |= (in && !all && cand ? 1u : 0u) << bit;
      }
    }
    cnt += __popc(wmask[gi]) + (__popc(cmask[gi]) << 16);
  }
  uint32_t total;
  const uint32_t off = block_inclusive_sum<uint32_t>(cnt, s_scan, &total) - cnt;
  const uint32_t nw = total & 0xffffu, ncd = total >> 16;
  // winners then candidates, contiguous in sbuf, when both fit the merge sort;
  // otherwise ("heavy") the candidates go to the row's workspace
  const bool heavy = nw + ncd > static_cast<uint32_t>(kSelSort);  // (uniform)
  uint64_t* cand = heavy ? p.cand_ws + g.soff : sbuf + nw;
  uint32_t wo = off & 0xffffu, co = off >> 16;
  const bool nan = nanacc != nanacc;
#pragma unroll
  for (int gi = 0; gi < kGroups; ++gi) {  // (unrolled: the masks stay in registers)
    uint32_t m = wmask[gi] | cmask[gi];
#pragma unroll 1
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      const int slot = slot_of(gi, bit);
      const uint32_t u = s_row[slot];
      const int ix = slot < body ? slot + head : (slot - body < head ? slot - body : slot);
      const uint64_t x = composite(order_key(u), static_cast<uint32_t>(ix));
      if ((wmask[gi] >> bit) & 1u) {
        if (wo < static_cast<uint32_t>(kSelMaxK)) sbuf[wo] = x;
        ++wo;
      } else {
        if (co < static_cast<uint32_t>(n)) cand[co] = x;
        ++co;
      }
    }
  }
  if (nan) set_status(p.status, HSA_DEV_NAN);
  __syncthreads();
  // (4) the attended list: the winners in the order of the pass (fixed by the
  // scan, so every run lists them alike), then the `need` largest candidates
  // by their rank among the candidates (few: ranked by counting; many: radix
  // select).  The list, as composites, is kept in the row's workspace for the
  // ordered copy (topk_out) written at the end of the kernel.
  uint32_t nsel = nw < kk ? nw : kk;
  if (!all && kk > nsel && ncd > 0) {
    const uint32_t need = kk - nsel;
    if (need >= ncd) {
      for (uint32_t i = t; i < ncd; i += kThreads) sbuf[nsel + i] = cand[i];
      nsel += ncd;
    } else if (!heavy && ncd <= static_cast<uint32_t>(kSelRank)) {
      // candidate c's rank = the number of candidates greater than it (unique
      // composites); one candidate per thread when they fit, else kQ
      constexpr int kQ = kSelRank / kThreads;
      auto rank_by_count = [&](auto nq) {
        constexpr int Q = decltype(nq)::value;
        uint64_t x[Q];
        uint32_t r[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const uint32_t ci = t + q * kThreads;
          x[q] = ci < ncd ? cand[ci] : ~0ull;
          r[q] = 0;
        }
#pragma unroll 4
        for (uint32_t i = 0; i < ncd; ++i) {
          const uint64_t y = cand[i];
#pragma unroll
          for (int q = 0; q < Q; ++q) r[q] += y > x[q] ? 1u : 0u;
        }
        __syncthreads();  // every candidate read before the list grows over them
#pragma unroll
        for (int q = 0; q < Q; ++q)
          if (t + q * kThreads < static_cast<int>(ncd) && r[q] < need) sbuf[nsel + r[q]] = x[q];
      };
      if (ncd <= static_cast<uint32_t>(kThreads)) rank_by_count(std::integral_constant<int, 1>());
      else rank_by_count(std::integral_constant<int, kQ>());
      nsel += need;
    } else {
      if (t == 0) s_cnt = nsel;
      __syncthreads();
      select_rest<2048 / kThreads>(cand, ncd < static_cast<uint32_t>(n) ? ncd : static_cast<uint32_t>(n),
                                   need, sbuf, &s_cnt, kSelMaxK, s_row, s_scan, s_out,
                                   64 - kRowHistBits);  // 11-bit digits
      __syncthreads();
      nsel = s_cnt < kk ? s_cnt : kk;
    }
  }
  __syncthreads();
  // (5) every split's share of the list (the list kept for the ordered copy),
  // and then this split's own rows prefetched into L2 for its gather (the
  // other splits start theirs at once).  Split q attends entries [bnd[q],
  // bnd[q + 1]) (S <= kMaxCl).  Its share (16-bit entries, in pairs) and the
  // list's length reach another split's shared memory by asynchronous stores
  // that count their bytes on its sel_full barrier, which that split armed
  // with exactly those bytes at launch (sel_bytes): its phase ends once they
  // have landed (no fence, no remote arrive, no wait here).  The selecting
  // split writes its own share with plain stores and arrives on its barrier.
  int bnd[kMaxCl + 1];
#pragma unroll
  for (int q = 0; q <= kMaxCl; ++q) bnd[q] = q < p.S ? static_cast<int>(share_first(p, g.n_swa, q)) : p.k;
  if (p.topk_out)
    for (int e = t; e < static_cast<int>(nsel); e += kThreads) p.cand_ws[g.soff + e] = sbuf[e];
  auto entry = [&](int e) -> uint32_t {  // row-local index, 0xffff past the selection
    return e < static_cast<int>(nsel) ? (0xffffffffu - static_cast<uint32_t>(sbuf[e])) & 0xffffu
                                      : 0xffffu;
  };
#pragma unroll
  for (int q = 0; q < kMaxCl; ++q) {
    if (q >= p.S) break;
    const int npairs = (bnd[q + 1] - bnd[q] + 1) >> 1;
    const bool own = q == static_cast<int>(rank);
    const uint32_t bar = own ? 0u : map_rank(&sh.sel_full, static_cast<uint32_t>(q));
    const uint32_t dst = own ? 0u : map_rank(&sh.sel[0], static_cast<uint32_t>(q));
    if (t == kThreads - 1) {
      if (own) sh.sel_n = nsel;
      else st_async_u32(map_rank(&sh.sel_n, static_cast<uint32_t>(q)), nsel, bar);
    }
    for (int i = t; i < npairs; i += kThreads) {
      const int e = bnd[q] + 2 * i;
      const uint32_t hi = e + 1 < bnd[q + 1] ? entry(e + 1) : 0xffffu;
      const uint32_t v = entry(e) | (hi << 16);
      if (own) reinterpret_cast<uint32_t*>(sh.sel)[i] = v;
      else st_async_u32(dst + 4u * static_cast<uint32_t>(i), v, bar);
    }
  }
  // this split's own share: plain stores, then a local arrive
  __syncthreads();
  if (t == 0) tc::mbar_arrive(&sh.sel_full);
  int own_first = 0, own_end = 0;  // this split's share
#pragma unroll
  for (int q = 0; q < kMaxCl; ++q)
    if (q == static_cast<int>(rank)) {
      own_first = bnd[q];
      own_end = min(static_cast<int>(nsel), bnd[q + 1]);
    }
  for (int e = own_first + t; e < own_end; e += kThreads) {
    const uint32_t j = 0xffffffffu - static_cast<uint32_t>(sbuf[e]);
    const uint16_t* rowp = p.extra + (g.off + j) * p.Dqk;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(rowp),
                 "r"(static_cast<uint32_t>(p.Dqk * 2))
                 : "memory");
  }
}

// The selection of token b in order (value descending, lower index first),
// to topk_out: the listed composites, kept in the row's workspace by the
// selection, sorted in shared memory (every thread of the selecting CTA,
// after its attention; the ring is free).
HSA_DEVINL void write_topk_sorted(const AttnParams& p, uint8_t* ring, int b, const SeqGeom& g,
                                  int nsel) {
  const int t = threadIdx.x;
  uint64_t* a = reinterpret_cast<uint64_t*>(ring);
  for (int i = t; i < nsel; i += kThreads) a[i] = p.cand_ws[g.soff + i];
  int P = 32;
  while (P < nsel) P <<= 1;
  merge_sort_desc<kSelMaxK / kThreads>(a, a + kSelMaxK, nsel, P);
  int32_t* o = p.topk_out + static_cast<int64_t>(b) * p.k;
  for (int e = t; e < p.k; e += kThreads)
    o[e] = e < nsel ? static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(a[e])) : -1;
}

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

// Merge of the S splits of one (token, head group) inside their cluster (all
// threads of every CTA call it).  Unit u (128 value channels x 16 heads of
// O^T) is finished by split u % S.  After a cluster barrier (every split's ring
// is free), each split reads from TMEM the units the other splits finish and
// stores them, as posted distributed-shared-memory stores, into the owner's
// ring (slot: the sender's place among the others x units per owner + u / S);
// m and l go to every split.  After a second barrier every owner combines its
// own part (from TMEM) with the received parts (local shared memory):
//   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s,
// with no remote load anywhere.  The loops are kept rolled: this code runs
// once per launch, so its size (the instruction fetches) costs more than its
// loop overhead.
template <int kN>
HSA_DEVINL void cluster_merge(const AttnParams& p, Shared& sh, uint8_t* ring, uint8_t* scratch,
                              uint32_t tmem, int b, int g, bool own, int TC, int NMT) {
  constexpr int kQ = kN / 16;  // 16-head column groups
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int rank = static_cast<int>(cluster_rank());
  const int U = NMT * kQ;
  const int upo = (U + S - 1) / S;  // units per owner
  // warp w reads TMEM lane quarter w & 3 (value channels); the two warps of a
  // quarter (halves hw) take alternate units
  const int quarter = warp & 3, hw = warp >> 2, row = quarter * 32 + lane;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  auto unit_col = [&](int u) { return lane_addr + (TC + u / kQ) * kN + (u % kQ) * 16; };
  // slot of sender s's part of unit u in the owner's ring
  auto slot = [&](int s, int u) {
    const int o = u % S;
    return (s < o ? s : s - 1) * upo + u / S;
  };
  if (tid < kN) {
    const float mv = own ? sh.m[tid] : -INFINITY, lv = own ? sh.l[tid] : 0.f;
    for (int q = 0; q < S; ++q) {
      st_cluster_u32(map_rank(&sh.xm[rank][tid], q), __float_as_uint(mv));
      st_cluster_u32(map_rank(&sh.xl[rank][tid], q), __float_as_uint(lv));
    }
  }
  if (tid < S) st_cluster_u32(map_rank(&sh.xok[rank], tid), own ? 1u : 0u);
  cluster_sync();  // every split's roles are done: its ring may receive
  if (own) {
    tc::fence_after_sync();
    // the units other splits finish, straight from TMEM into their rings; two
    // per round (both TMEM loads in flight before one wait)
#pragma unroll 1
    for (int u = hw; u < U; u += 4) {
      const int u2 = u + 2 < U ? u + 2 : u;
      uint32_t a[16], c[16];
      tc::tmem_ld16(unit_col(u), a);
      tc::tmem_ld16(unit_col(u2), c);
      tc::tmem_ld_wait();
      if (u % S != rank) {
        const uint32_t d = map_rank(ring + slot(rank, u) * kUnitBytes + row * 16, u % S);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          st_cluster_f32x4(d + c4 * (kKeys * 16u), __uint_as_float(a[4 * c4]), __uint_as_float(a[4 * c4 + 1]),
                           __uint_as_float(a[4 * c4 + 2]), __uint_as_float(a[4 * c4 + 3]));
      }
      if (u2 != u && u2 % S != rank) {
        const uint32_t d = map_rank(ring + slot(rank, u2) * kUnitBytes + row * 16, u2 % S);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          st_cluster_f32x4(d + c4 * (kKeys * 16u), __uint_as_float(c[4 * c4]), __uint_as_float(c[4 * c4 + 1]),
                           __uint_as_float(c[4 * c4 + 2]), __uint_as_float(c[4 * c4 + 3]));
      }
    }
  }
  cluster_sync();  // every part and statistic has landed; no remote access follows
  if (tid < kN) {
    float M = -INFINITY;
    for (int r = 0; r < S; ++r)
      if (sh.xl[r][tid] > 0.f) M = fmaxf(M, sh.xm[r][tid]);
    float L = 0.f;
    for (int r = 0; r < S; ++r) {
      const float w = sh.xl[r][tid] > 0.f ? tc::ex2_approx(sh.xm[r][tid] - M) : 0.f;
      sh.red[r][tid] = w;  // (the softmax's reduction scratch is free by now)
      L += w * sh.xl[r][tid];
    }
    sh.inv[tid] = L > 0.f ? __frcp_rn(L) : 0.f;
    if (rank == 0 && tid < p.HG && p.lse)
      p.lse[static_cast<int64_t>(b) * p.Hq + g * p.HG + tid] =
          L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  const bool bf = p.out_dtype == HSA_BF16;
  const int64_t head0 = static_cast<int64_t>(b) * p.Hq + g * p.HG;
  // Warp half hw finishes units u = rank + S*hw + 2S*k, one per round (two
  // per round, their TMEM loads in flight together, measured 0.7 us slower
  // per layer: this code runs once per launch, and the larger loop body costs
  // more in instruction fetches than the overlap saves).  When 2S is a
  // multiple of kQ those units share one 16-head group, whose weights and
  // 1/L then stay in registers (else they are read per unit).
  const bool fixed = (2 * S) % kQ == 0;
  float wr[kMaxCl][16], wown[16], ivr[16];
  auto load_w = [&](int q16) {
#pragma unroll
    for (int r = 0; r < kMaxCl; ++r)
#pragma unroll
      for (int e = 0; e < 16; ++e) wr[r][e] = r < S ? sh.red[r][q16 * 16 + e] : 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      wown[e] = sh.red[rank][q16 * 16 + e];
      ivr[e] = sh.inv[q16 * 16 + e];
    }
  };
  if (fixed) load_w((rank + S * hw) % kQ);
  uint8_t* tr0 = scratch + warp * (2 * 16 * 32 * 4);  // the warp's transpose buffer
  // combines unit u's parts (own: a, from TMEM) into o, scaled by 1/L
  auto combine = [&](int u, const uint32_t (&a)[16], float (&o)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = own ? __uint_as_float(a[e]) * wown[e] : 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCl; ++r) {
      if (r >= S || r == rank || !sh.xok[r]) continue;
      const float4* src = reinterpret_cast<const float4*>(ring + slot(r, u) * kUnitBytes + row * 16);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 v = src[c4 * kKeys];
        o[4 * c4] = fmaf(v.x, wr[r][4 * c4], o[4 * c4]);
        o[4 * c4 + 1] = fmaf(v.y, wr[r][4 * c4 + 1], o[4 * c4 + 1]);
        o[4 * c4 + 2] = fmaf(v.z, wr[r][4 * c4 + 2], o[4 * c4 + 2]);
        o[4 * c4 + 3] = fmaf(v.w, wr[r][4 * c4 + 3], o[4 * c4 + 3]);
      }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] *= ivr[e];
  };
  // transposes o (lane l: channel l of 16 heads) through tr and writes 16
  // contiguous bytes of one head per lane
  auto write_out = [&](int u, const float (&o)[16], uint8_t* tr) {
    const int q16 = u % kQ;
    const int64_t base = (head0 + q16 * 16) * p.Dv + (u / kQ) * kKeys + quarter * 32;
    if (bf) {
      __nv_bfloat16* t = reinterpret_cast<__nv_bfloat16*>(tr);
#pragma unroll
      for (int e = 0; e < 16; ++e) t[e * 32 + lane] = __float2bfloat16_rn(o[e]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = lane + 32 * j, h = c >> 2, part = c & 3;  // 4 chunks of 8 channels per head
        if (q16 * 16 + h < p.HG)
          *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + base + h * p.Dv + part * 8) =
              *reinterpret_cast<const uint4*>(t + h * 32 + part * 8);
      }
    } else {
      float* t = reinterpret_cast<float*>(tr);
#pragma unroll
      for (int e = 0; e < 16; ++e) t[e * 32 + lane] = o[e];
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = lane + 32 * j, h = c >> 3, part = c & 7;  // 8 chunks of 4 channels per head
        if (q16 * 16 + h < p.HG)
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + base + h * p.Dv + part * 4) =
              *reinterpret_cast<const float4*>(t + h * 32 + part * 4);
      }
    }
  };
#pragma unroll 1
  for (int u = rank + S * hw; u < U; u += 2 * S) {
    uint32_t a[16];
    if (own) {
      tc::tmem_ld16(unit_col(u), a);
      tc::tmem_ld_wait();
    }
    float o[16];
    if (!fixed) load_w(u % kQ);
    combine(u, a, o);
    __syncwarp();  // the transpose buffer is free (previous round's reads done)
    write_out(u, o, tr0);
  }
}

// Q of token b, head group g into the Q region by TMA: NSL boxes of 64
// channels x kN heads (128-byte swizzled, the layout the S^T MMA reads), one
// issuing thread, completing on q_full.  Heads past the group's (kN > HG)
// load the next rows of q, which no output reads (zeros past the tensor).
template <int kN>
HSA_DEVINL void issue_q_tma(const CUtensorMap* qmap, Shared& sh, uint8_t* qs, int NSL, int row0) {
  tc::mbar_arrive_expect_tx(&sh.q_full, static_cast<uint32_t>(NSL) * kN * 128);
#pragma unroll 1
  for (int j = 0; j < NSL; ++j) tc::tma_load_2d(qs + j * (kN * 128), qmap, j * 64, row0, &sh.q_full);
}

// kSel: the fused selection of the layer's C4 path (see select_token).
template <int kN, bool kSel>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ CUtensorMap qmap,
                                                          const __grid_constant__ CUtensorMap swamap,
                                                          int swa_tma,
                                                          const __grid_constant__ CUtensorMap poolmap,
                                                          int pool_tma, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  // Programmatic dependent launch.  When the previous kernel is the top-k
  // (p.early 1), it triggered this launch only after its own wait, so
  // everything older (the append's window rows and lengths, q) is complete and
  // only the index lists need the wait, which the gather and softmax threads
  // take right before reading them.  When it is the append of a dense layer
  // (p.early 2), the lengths come from the step's input and the gatherers wait
  // right before the first tile holding a row the append writes.  Otherwise
  // every thread waits first.
  if (!p.early) {
    pdl_wait();
    pdl_trigger();
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the S splits of a (token, head group) are consecutive CTAs (one cluster with cl)
  const int s = blockIdx.x % p.S;
  const int g = (blockIdx.x / p.S) % p.G;
  const int b = blockIdx.x / (p.G * p.S);
  const int NSL = p.Dqk / 64, NMT = p.Dv / 128, NP1 = (NSL + 1) / 2, TC = p.TC;
  const SeqGeom geo = seq_geom(p, b);
  const int64_t n_slots = geo.n_swa + geo.n_extra;
  // this split's slots [a0, a1), covered by tiles [t0, t1)
  const int64_t a0 = static_cast<int64_t>(s) * p.sps;
  const int64_t a1 = min(a0 + p.sps, n_slots);
  const int t0 = static_cast<int>(a0 / kKeys);
  const int nt = a1 > a0 ? static_cast<int>((a1 + kKeys - 1) / kKeys) - t0 : 0;
  const int t1 = t0 + nt;

  if (nt <= 0 && !p.cl) {  // nothing to attend in this split (a cluster member still merges)
    if (tid < kKeys) {
      if (p.S == 1)
        for (int h = 0; h < p.HG; ++h)
          for (int dv = tid; dv < p.Dv; dv += kKeys) write_result(p, b, g, s, h, dv, 0.f);
      if (tid < p.HG) write_lse(p, b, g, s, tid, -INFINITY);
    }
    if (!kSel && p.early == 2 && tid == 0) pdl_wait();  // the grid completes only after the previous kernel
    return;
  }
  if (!kSel && p.extra && !p.idx && geo.nb > p.max_rows && tid == 0 && s == 0 && g == 0)
    set_status(p.status, HSA_DEV_BOUNDS);
  // Chunks of up to TC tiles.  With the fused selection the leading tiles that
  // hold window rows only form a chunk of their own, attended while the
  // token's last split selects the rest; chunks holding compressed rows wait
  // for that selection.
  const int win_tiles = kSel ? max(0, min(geo.n_swa / kKeys - t0, min(nt, TC))) : 0;
  auto chunk_tb = [&](int c) { return c == 0 ? t0 : t0 + win_tiles + (win_tiles > 0 ? c - 1 : c) * TC; };
  auto chunk_nct = [&](int c) { return min(c == 0 && win_tiles > 0 ? win_tiles : TC, t1 - chunk_tb(c)); };
  auto chunk_sel = [&](int c) {
    return kSel && static_cast<int64_t>(chunk_tb(c) + chunk_nct(c)) * kKeys > geo.n_swa;
  };
  const int nchunks = win_tiles > 0 ? 1 + (nt - win_tiles + TC - 1) / TC : (nt + TC - 1) / TC;
  // Q shares its region with P^T buffer 1, which the tiles with an odd index
  // (counted over the split's chunks) use: chunk c reloads Q only when chunk
  // c - 1 had such a tile (a one-tile window chunk leaves Q in place)
  auto q_reload = [&](int c) {
    return c > 0 && (chunk_nct(c - 1) >= 2 || ((chunk_tb(c - 1) - t0) & 1) != 0);
  };
  const uint32_t crank = p.cl ? cluster_rank() : 0u;
  const bool selector = kSel && s == p.S - 1;
  const int64_t sel_e0 = kSel ? share_first(p, geo.n_swa, s) : 0;  // first entry of this split's share

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t qslice = kN * 128;       // bytes of one Q slice (kN heads x 64 channels)
  uint8_t* ring = smem;
  uint8_t* qs = ring + kRing * kPairBytes;  // Q during pass 1 ...
  // P^T buffers (2 K-blocks of 64 keys x kN heads each; with 64 heads instead
  // one 128-byte row of 64 heads per key, MN-major for the O^T MMA, so that a
  // softmax thread writes its key's row with 16-byte stores): tile gt uses
  // buffer gt & 1; buffer 1 is the start of the Q region, written only once
  // the chunk's pass 1 is complete
  uint8_t* const pbuf0 = qs + attn_q_region(NSL, kN);
  uint8_t* const pbuf1 = qs;
  // TMEM columns: S^T of chunk tile tc at tc*kN; O^T M-tile m at (TC + m)*kN
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>((TC + NMT) * kN)) tmem_cols <<= 1;

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&sh.full[i], 32);
      tc::mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < kMaxTC; ++i) tc::mbar_init(&sh.s_full[i], 1);
    tc::mbar_init(&sh.s_empty, kKeys);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh.p_full[i], kKeys);
      tc::mbar_init(&sh.o_done[i], 1);
    }
    tc::mbar_init(&sh.q_full, 1);
    tc::mbar_init(&sh.fin, 1);
    if (kSel) {
      tc::mbar_init(&sh.sel_full, 1);
      tc::mbar_init(&sh.sel_cp, 1);
      // another split's share arrives by the selecting split's asynchronous
      // stores, whose bytes complete the phase (the selecting split arrives
      // on its own barrier)
      if (!selector) tc::mbar_arrive_expect_tx(&sh.sel_full, sel_bytes(p, geo.n_swa, s));
    }
    sh.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&sh.tmem, tmem_cols);
    tc::tmem_relinquish();
  }
  // the ring starts zeroed: rows that are never gathered hold finite values
  for (int i = tid; i < static_cast<int>(kRing * kPairBytes / 16); i += kThreads)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0u, 0u, 0u, 0u);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem;
  if (kSel) {
    // every split's barriers exist before the selecting split arrives on them
    if (p.cl) cluster_sync();
    // the window rows this split attends first, into L2 while the previous
    // kernels finish (the append's new row included: a prefetch brings no
    // stale copy, the append's store updates L2)
#pragma unroll 1
    for (int r = tid; r < win_tiles * kKeys; r += kThreads) {
      const int64_t pos = geo.L - geo.n_swa + static_cast<int64_t>(t0) * kKeys + r;
      const uint16_t* rowp = p.swa + (static_cast<int64_t>(geo.bs) * p.Wr + pos % p.Wr) * p.Dqk;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(rowp),
                   "r"(static_cast<uint32_t>(p.Dqk * 2))
                   : "memory");
    }
    if (selector) {
      // Q first (the previous kernel does not write it), then the selection,
      // which needs the indexer's scores and histogram
      if (tid == kProdWarp0 * 32) issue_q_tma<kN>(&qmap, sh, qs, NSL, b * p.Hq + g * p.HG);
      // an invalid span (bad offsets or a live count above the capacity), or a
      // row longer than the host-checked bound: flagged, treated as empty (the
      // offsets and lengths are older than the previous kernel, like geo)
      const bool bad = !p.sp.valid(b) || geo.nb > kSelRowMax;
      const int n = bad ? 0 : static_cast<int>(geo.nb);
      pdl_wait();
      if (bad && tid == 0) set_status(p.status, HSA_DEV_BOUNDS);
      // survivors: the even tiles' P^T buffer when it holds kSelMax composites,
      // else the region the plan adds after it
      uint8_t* sel_buf = 2 * kN * 128 >= kSelMax * 8 ? pbuf0 : pbuf0 + 2 * kN * 128;
      select_token(p, sh, ring, reinterpret_cast<uint64_t*>(sel_buf), b, geo, n, crank);
      // the ring held scores: zeroed again (rows never gathered must be finite)
      for (int i = tid; i < static_cast<int>(kRing * kPairBytes / 16); i += kThreads)
        reinterpret_cast<uint4*>(ring)[i] = make_uint4(0u, 0u, 0u, 0u);
      tc::fence_proxy_async_smem();
      __syncthreads();
    }
  }

  if (warp >= kProdWarp0) {
    // ------------------------------------------------------------ gatherers
    // Gather warp w issues ring items w, w + 3, w + 6, ... (slot item % kRing)
    // and keeps up to two of them in flight: its cp.async groups retire in
    // order, each signalling its slot.  Q arrives by TMA on q_full.
    constexpr int kProdWarps = kProdThreads / 32;
    const int pt_ = tid - kProdWarp0 * 32, pw = warp - kProdWarp0;
    bool ok = true;
    int64_t pend0 = 0, pend1 = 0;  // this warp's unsignalled groups, oldest first
    int np = 0;
    auto signal = [&](int64_t it) { tc::mbar_arrive(&sh.full[it % kRing]); };
    auto retire_all = [&]() {  // signal each pending group as soon as it has landed
      if (np == 2) {
        tc::cp_async_wait<1>();
        tc::fence_proxy_async_smem();
        signal(pend0);
        pend0 = pend1;
        np = 1;
      }
      if (np == 1) {
        tc::cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        signal(pend0);
        np = 0;
      }
    };
    auto push = [&](int64_t it) {  // right after committing group `it`
      if (np == 2) {  // three in flight: the oldest must land first
        tc::cp_async_wait<2>();
        tc::fence_proxy_async_smem();
        signal(pend0);
        pend0 = pend1;
        np = 1;
      }
      if (np == 0) pend0 = it; else pend1 = it;
      ++np;
    };
    bool q_pre = selector;  // the selecting split issued chunk 0's Q before selecting
    // (p.early 2) whether tile tt holds a row the append writes: a window row
    // (the step's tokens are among them) or a pool row of a block completed in
    // this step (rows L_in / r and later; here slot n_swa + e holds pool row e)
    bool dep_waited = kSel || p.early != 2;  // (compiled out of the fused-selection kernel)
    auto append_tile = [&](int tt) {
      const int64_t s0 = static_cast<int64_t>(tt) * kKeys;
      if (s0 < geo.n_swa) return true;
      const int64_t L_in = geo.L - 1 - (p.T == 1 ? 0 : b % p.T);
      return s0 + kKeys > geo.n_swa + L_in / p.sp.ratio;
    };
    auto issue_q = [&]() {  // Q by TMA, one thread
      if (q_pre) {
        q_pre = false;
        return;
      }
      if (pt_ == 0) issue_q_tma<kN>(&qmap, sh, qs, NSL, b * p.Hq + g * p.HG);
    };
    int64_t item = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int tb = chunk_tb(c), nct = chunk_nct(c);
      // every previous item is issued (its rows were read at issue): refill the
      // tables; a warp that gave up is known to all from here on
      if (tc::named_barrier_or(2, kProdThreads, !ok)) {
        ok = false;
        break;
      }
      if (c == 0) {
        issue_q();  // q is not written by the previous kernel: load it before waiting
        if (kSel || p.early != 2) pdl_wait();
        pdl_trigger();
      }
      if (chunk_sel(c)) {  // this chunk's compressed rows come from the selection
        const bool f = !wait_cluster_or_abort(&sh.abort, &sh.sel_full, 0, p.status);
        if (tc::named_barrier_or(2, kProdThreads, f)) {
          ok = false;
          break;
        }
      }
      {
        constexpr int kPer = (kMaxTC * kKeys + kProdThreads - 1) / kProdThreads;
        int64_t jv[kPer];
#pragma unroll
        for (int k2 = 0; k2 < kPer; ++k2) {  // the list entries first: loads in flight together
          const int r = pt_ + k2 * kProdThreads;
          const int64_t slot = static_cast<int64_t>(tb) * kKeys + r;
          if (kSel) {
            const int64_t e = slot - geo.n_swa;
            const uint16_t v = r < nct * kKeys && e >= 0 && e < p.k ? sh.sel[e - sel_e0] : uint16_t(0);
            jv[k2] = v == 0xffff ? -1 : static_cast<int64_t>(v);
          } else {
            jv[k2] = r < nct * kKeys ? slot_index(p, b, geo, slot) : 0;
          }
        }
#pragma unroll
        for (int k2 = 0; k2 < kPer; ++k2) {
          const int r = pt_ + k2 * kProdThreads;
          const int64_t slot = static_cast<int64_t>(tb) * kKeys + r;
          if (r < nct * kKeys)
            sh.rows[r / kKeys][r % kKeys] =
                slot >= a0 && slot < a1 ? slot_row_j(p, b, geo, slot, jv[k2], true) : nullptr;
        }
      }
      tc::named_barrier(2, kProdThreads);
      if (q_reload(c)) {
        // Q shares its region with the P^T buffers of the previous chunk, free
        // once that chunk's last O^T MMAs are done
        const int lt = tb - t0 - 1;
        const bool f = !wait_or_abort(sh, &sh.o_done[lt & 1], (lt >> 1) & 1, p.status);
        if (tc::named_barrier_or(2, kProdThreads, f)) {
          ok = false;
          break;
        }
        issue_q();
      }
      // pass 1: every channel pair of every tile; pass 2: the value pairs again
      for (int pass = 0; pass < 2; ++pass) {
        const int nit = pass == 0 ? NP1 : NMT;
        for (int tc_ = 0; tc_ < nct; ++tc_) {
          if (!dep_waited && append_tile(tb + tc_)) {
            pdl_wait();
            dep_waited = true;
          }
          const uint16_t* const* table = sh.rows[tc_];
          // this lane's rows r0 + 4k of the tile, held in registers for the
          // tile's items: the copy loop below then issues back to back (its
          // shared-memory table loads were on the ring's critical path)
          const uint16_t* rp[kKeys / 4];
#pragma unroll
          for (int k = 0; k < kKeys / 4; ++k) rp[k] = table[(lane >> 3) + 4 * k];
          // A full window tile (the token's 128 ring rows, every one a window
          // row) arrives by TMA: the ring's rows in slot order, 64-channel
          // boxes, 128-byte swizzled as the MMA reads them.
          const bool win_tma = swa_tma && tb + tc_ == 0 && geo.n_swa == kKeys && a0 == 0;
          // A dense tile of 128 live compressed rows (contiguous in the pool)
          // arrives by TMA too, from a map over the pool's rows.
          const int64_t tile_slot = static_cast<int64_t>(tb + tc_) * kKeys;
          const int64_t e_first = tile_slot - geo.n_swa;
          const bool pool_tile = pool_tma && e_first >= 0 && e_first + kKeys <= geo.n_extra &&
                                 tile_slot >= a0 && tile_slot + kKeys <= a1;
          for (int it = 0; it < nit; ++it, ++item) {
            if (!ok || item % kProdWarps != pw) continue;
            const int slot = static_cast<int>(item % kRing);
            if (item >= kRing) {
              const uint32_t par = static_cast<uint32_t>((item / kRing - 1) & 1);
              if (!tc::mbar_test_wait(&sh.empty[slot], par)) {
                retire_all();  // signal everything issued before blocking
                ok = __all_sync(0xffffffffu, wait_or_abort(sh, &sh.empty[slot], par, p.status));
                if (!ok) continue;
              }
            }
            if (win_tma || pool_tile) {
              // lane 0 arms the slot with the bytes and issues both slices; the
              // other lanes arrive (the slot's barrier counts 32 arrivals)
              const int j0 = 2 * it;
              const bool two = j0 + 1 < NSL;
              if (lane == 0) {
                const CUtensorMap* map = win_tma ? &swamap : &poolmap;
                const int32_t y = win_tma ? b * p.W : static_cast<int32_t>(geo.off + e_first);
                tc::mbar_arrive_expect_tx(&sh.full[slot], (two ? 2u : 1u) * kSliceBytes);
                tc::tma_load_2d(ring + slot * kPairBytes, map, j0 * 64, y, &sh.full[slot]);
                if (two)
                  tc::tma_load_2d(ring + slot * kPairBytes + kSliceBytes, map, (j0 + 1) * 64, y,
                                  &sh.full[slot]);
              } else {
                tc::mbar_arrive(&sh.full[slot]);
              }
              continue;
            }
            // Masked rows are not copied (no memory request): the slot keeps finite
            // data (zeroed at start, or rows of this token gathered earlier) that
            // the softmax weighs with 0.
            const uint32_t dst = tc::smem_u32(ring + slot * kPairBytes);
            // lane: 16-byte chunk cc of rows r0 + 4k (k < 32) of both slices of the pair
            const int cc = lane & 7, r0 = lane >> 3, j0 = 2 * it;
            const bool two = j0 + 1 < NSL;
#pragma unroll
            for (int k = 0; k < kKeys / 4; ++k) {
              const int r = r0 + 4 * k;
              const uintptr_t row = reinterpret_cast<uintptr_t>(rp[k]);
              const bool live = row != 0;
              const uint32_t off = (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4);
              const uintptr_t src = row + (j0 * 64 + cc * 8) * sizeof(uint16_t);
              cp_async16_if(dst + off, reinterpret_cast<const void*>(src), live);
              cp_async16_if(dst + kSliceBytes + off, reinterpret_cast<const void*>(src + 128), live && two);
            }
            tc::cp_async_commit();
            push(item);
          }
        }
      }
      retire_all();  // the chunk's Q and items are all signalled
    }
    retire_all();
    if (!dep_waited) pdl_wait();  // the grid completes only after the previous kernel
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = tc::idesc_bf16_f32(kKeys, kN);
      const uint32_t idO = tc::idesc_bf16_f32(kKeys, kN, /*a_mn=*/true, /*b_mn=*/kN == 64);
      bool ok = true;
      int64_t item = 0;
      int gt = 0;  // tiles through pass 2 so far (P^T buffer gt & 1)
      int nq = 0;  // Q loads waited for
      for (int c = 0; c < nchunks && ok; ++c) {
        const int nct = chunk_nct(c);
        if (c > 0 && !wait_or_abort(sh, &sh.s_empty, (c - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        if ((c == 0 || q_reload(c)) && !wait_or_abort(sh, &sh.q_full, (nq++) & 1, p.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        for (int tc_ = 0; tc_ < nct && ok; ++tc_) {
          const uint32_t d_s = tmem + tc_ * kN;
          for (int it = 0; it < NP1; ++it, ++item) {
            const int slot = static_cast<int>(item % kRing);
            if (!wait_or_abort(sh, &sh.full[slot], static_cast<uint32_t>((item / kRing) & 1),
                               p.status)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t ka0 = tc::smem_u32(ring + slot * kPairBytes);
            for (int half = 0; half < 2; ++half) {
              const int j = 2 * it + half;
              if (j >= NSL) break;
              const uint32_t ka = ka0 + half * kSliceBytes;
              const uint32_t qa = tc::smem_u32(qs + j * qslice);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = tc::smem_desc(ka + ks * 32, 16, 1024, tc::kSwizzle128B);
                const uint64_t bq = tc::smem_desc(qa + ks * 32, 16, 1024, tc::kSwizzle128B);
                tc::mma_bf16(d_s, a, bq, idS, (j | ks) != 0 ? 1u : 0u);
              }
            }
            tc::mma_commit(&sh.empty[slot]);
          }
          if (ok) tc::mma_commit(&sh.s_full[tc_]);
        }
        for (int tc_ = 0; tc_ < nct && ok; ++tc_, ++gt) {
          const int buf = gt & 1;
          if (!wait_or_abort(sh, &sh.p_full[buf], (gt >> 1) & 1, p.status)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t pa = tc::smem_u32(buf ? pbuf1 : pbuf0);
          for (int m = 0; m < NMT; ++m, ++item) {
            const int slot = static_cast<int>(item % kRing);
            if (!wait_or_abort(sh, &sh.full[slot], static_cast<uint32_t>((item / kRing) & 1),
                               p.status)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t va = tc::smem_u32(ring + slot * kPairBytes);
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              // P: 16 keys (K) per step; 64 heads are one 128-byte row per key
              // (MN-major), fewer heads a K-major row per head
              const uint64_t bp =
                  kN == 64 ? tc::smem_desc(pa + kk * 2048, 16, 1024, tc::kSwizzle128B)
                           : tc::smem_desc(pa + (kk >> 2) * kN * 128 + (kk & 3) * 32, 16, 1024,
                                           tc::kSwizzle128B);
              const uint64_t a = tc::smem_desc(va + kk * 2048, kSliceBytes, 1024, tc::kSwizzle128B);
              tc::mma_bf16(tmem + (TC + m) * kN, a, bp, idO, (gt > 0 || kk > 0) ? 1u : 0u);
            }
            tc::mma_commit(&sh.empty[slot]);
          }
          if (ok) tc::mma_commit(&sh.o_done[buf]);
        }
      }
      // drain: every MMA this thread issued has completed before TMEM is freed
      if (nchunks > 0) {
        tc::mma_commit(&sh.fin);
        tc::mbar_wait(&sh.fin, 0, p.status);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    // thread tid owns key lane tid of every S^T tile; heads in groups of 32 columns
    constexpr int kGroups = (kN + 31) / 32, kGW = kN < 32 ? kN : 32;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float l_part[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) l_part[h] = 0.f;
    if (tid < kN) sh.m[tid] = -INFINITY;
    bool ok = true;
    int gt = 0;
    // bit i: phase parity of s_full[i] in the current chunk (chunks may use
    // different numbers of tiles, so each barrier keeps its own count)
    uint32_t sf_par = 0;
    auto agree = [&](bool failed) { return !tc::named_barrier_or(1, kKeys, failed); };
    // S^T columns [col, col + kGW) of this lane, scaled to log2 units; -inf when masked
    auto load_s = [&](uint32_t col, bool valid, float (&x)[32]) {
      uint32_t raw[32];
      tc::tmem_ld16(tmem + lane_base + col, raw);
      if (kGW == 32) tc::tmem_ld16(tmem + lane_base + col + 16, raw + 16);
      tc::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i)
        x[i] = (i < kGW && valid) ? __uint_as_float(raw[i]) * p.scale_log2 : -INFINITY;
    };
    for (int c = 0; c < nchunks && ok; ++c) {
      const int tb = chunk_tb(c), nct = chunk_nct(c);
      // which of this lane's slots are attended, per chunk tile (loads issued before any wait)
      if (c == 0 && (kSel || p.early != 2)) pdl_wait();  // the index lists come from the previous kernel
      if (chunk_sel(c) && !agree(!wait_cluster_or_abort(&sh.abort, &sh.sel_full, 0, p.status))) {
        ok = false;
        break;
      }
      uint32_t vmask = 0;
      for (int tc_ = 0; tc_ < nct; ++tc_) {
        const int64_t slot = static_cast<int64_t>(tb + tc_) * kKeys + tid;
        bool v;
        if (kSel)  // window rows, and the selected entries (sel_n of them)
          v = slot < geo.n_swa || (slot - geo.n_swa < static_cast<int64_t>(sh.sel_n) &&
                                   slot - geo.n_swa < p.k);
        else
          v = slot_row(p, b, geo, slot, false) != nullptr;
        vmask |= (slot >= a0 && slot < a1 && v ? 1u : 0u) << tc_;
      }
      // ---- tile by tile, as soon as its S^T lands (online softmax): the tile's
      // maximum per head moves the running maximum m only when it rises by more
      // than 2^8 (O^T and l are then rescaled); P^T = 2^(S^T - m) goes to the
      // buffer its O^T pass reads, so the first tiles' P^T is ready before the
      // chunk's last S^T
      for (int tc_ = 0; tc_ < nct; ++tc_, ++gt) {
        if (!agree(!wait_or_abort(sh, &sh.s_full[tc_], (sf_par >> tc_) & 1u, p.status))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        __syncwarp();
        const bool valid = (vmask >> tc_) & 1u;
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          float x[32];
          load_s(tc_ * kN + gi * 32, valid, x);
          const float mcol = warp_transpose_reduce32<true>(x);
          if (gi * 32 + lane < kN) sh.red[warp][gi * 32 + lane] = mcol;
        }
        tc::named_barrier(1, kKeys);
        bool rescale = false;  // O^T holds earlier tiles weighted by a finite old maximum
        if (tid < kN) {
          const float mt =
              fmaxf(fmaxf(sh.red[0][tid], sh.red[1][tid]), fmaxf(sh.red[2][tid], sh.red[3][tid]));
          const float mo = sh.m[tid];
          const float mn = fmaxf(mo, mt);
          const bool moved = mn > mo + kRescaleLog2 || (mo == -INFINITY && mn > -INFINITY);
          sh.alpha[tid] = moved ? exp2f(mo - mn) : 1.f;
          if (moved) sh.m[tid] = mn;
          rescale = moved && mo > -INFINITY;
        }
        if (tc::named_barrier_or(1, kKeys, rescale)) {
#pragma unroll
          for (int h = 0; h < kN; ++h) l_part[h] *= sh.alpha[h];
          if (gt > 0) {
            // wait for the earlier tiles' O^T MMAs, then rescale O^T in TMEM
            const int lt = gt - 1;
            if (!agree(!wait_or_abort(sh, &sh.o_done[lt & 1], (lt >> 1) & 1, p.status))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            __syncwarp();
            for (int m = 0; m < NMT; ++m) {
              const uint32_t col = tmem + lane_base + (TC + m) * kN;
#pragma unroll
              for (int q16 = 0; q16 < kN / 16; ++q16) {
                uint32_t o[16];
                tc::tmem_ld16(col + q16 * 16, o);
                tc::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  o[i] = __float_as_uint(__uint_as_float(o[i]) * sh.alpha[q16 * 16 + i]);
                tc::tmem_st16(col + q16 * 16, o);
              }
            }
            tc::tmem_st_wait();
          }
        }
        // (a head whose old maximum was -inf has weighed everything with 0 so far:
        // its O^T columns and l are 0 and need no rescale)
        const int buf = gt & 1;
        if (gt >= 2) {  // the buffer is free once O^T of tile gt-2 has completed
          const int lt = gt - 2;
          if (!agree(!wait_or_abort(sh, &sh.o_done[buf], (lt >> 1) & 1, p.status))) {
            ok = false;
            break;
          }
        }
        if (buf == 1 && tc_ < nct - 1) {
          // buffer 1 overlays Q: wait until the chunk's pass 1 has read it for the last time
          if (!agree(!wait_or_abort(sh, &sh.s_full[nct - 1], (sf_par >> (nct - 1)) & 1u, p.status))) {
            ok = false;
            break;
          }
        }
        // P = 2^(S^T - m), rounded to bf16 (l sums the rounded values)
        auto p_pair = [&](const float (&x)[32], int i, int h) {
          const float m0 = sh.m[h], m1 = sh.m[h + 1];
          const float p0 = m0 == -INFINITY ? 0.f : tc::ex2_approx(x[i] - m0);
          const float p1 = m1 == -INFINITY ? 0.f : tc::ex2_approx(x[i + 1] - m1);
          const __nv_bfloat162 q2 = __floats2bfloat162_rn(p0, p1);
          l_part[h] += __low2float(q2);
          l_part[h + 1] += __high2float(q2);
          return *reinterpret_cast<const uint32_t*>(&q2);
        };
        if constexpr (kN == 64) {
          // key tid's row: 8 chunks of 8 heads, 128-byte swizzled (chunk c at c ^ (tid & 7))
          uint8_t* prow = (buf ? pbuf1 : pbuf0) + (tid >> 3) * 1024 + (tid & 7) * 128;
#pragma unroll
          for (int gi = 0; gi < kGroups; ++gi) {
            float x[32];
            load_s(tc_ * kN + gi * 32, valid, x);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) w[j] = p_pair(x, c4 * 8 + 2 * j, gi * 32 + c4 * 8 + 2 * j);
              const int c = gi * 4 + c4;
              *reinterpret_cast<uint4*>(prow + ((c ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          uint8_t* ptb = (buf ? pbuf1 : pbuf0) + (tid >> 6) * kN * 128;
          const int kc = (tid & 63) >> 3, ke = (tid & 7) << 1;
#pragma unroll
          for (int gi = 0; gi < kGroups; ++gi) {
            float x[32];
            load_s(tc_ * kN + gi * 32, valid, x);
#pragma unroll
            for (int i = 0; i < kGW; i += 2) {
              const int h = gi * 32 + i;
              const uint32_t pk = p_pair(x, i, h);
              *reinterpret_cast<uint16_t*>(ptb + (h >> 3) * 1024 + (h & 7) * 128 +
                                           ((kc ^ (h & 7)) << 4) + ke) = static_cast<uint16_t>(pk);
              const int h1 = h + 1;
              *reinterpret_cast<uint16_t*>(ptb + (h1 >> 3) * 1024 + (h1 & 7) * 128 +
                                           ((kc ^ (h1 & 7)) << 4) + ke) = static_cast<uint16_t>(pk >> 16);
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&sh.p_full[buf]);
      }
      if (!ok) break;
      sf_par ^= (1u << nct) - 1u;  // s_full[0 .. nct) each completed one phase
      // this chunk's S^T columns may be overwritten by the next chunk
      tc::fence_before_sync();
      tc::mbar_arrive(&sh.s_empty);
    }
    {
      // `ok` is uniform over the softmax warps here (every exit from the loop
      // went through an agreement barrier)
      bool failed = !ok;
      if (!failed && gt > 0) {
        const int lt = gt - 1;
        failed = !wait_or_abort(sh, &sh.o_done[lt & 1], (lt >> 1) & 1, p.status);
      }
      ok = agree(failed);
    }
    // every softmax thread reaches these barriers, whether or not it aborted
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
      float lv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) lv[i] = (i < kGW) ? l_part[gi * 32 + (i < kGW ? i : 0)] : 0.f;
      const float lcol = warp_transpose_reduce32<false>(lv);
      if (gi * 32 + lane < kN) sh.red[warp][gi * 32 + lane] = lcol;
    }
    tc::named_barrier(1, kKeys);
    if (tid < kN) {
      const float l = (sh.red[0][tid] + sh.red[1][tid]) + (sh.red[2][tid] + sh.red[3][tid]);
      sh.inv[tid] = l > 0.f ? 1.f / l : 0.f;
      sh.l[tid] = l;
      if (ok && tid < p.HG && !p.cl)
        write_lse(p, b, g, s, tid, l > 0.f ? (sh.m[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY);
    }
    if (tid == 0) sh.done_ok = ok ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (p.cl) {
    cluster_merge<kN>(p, sh, ring, qs, tmem, b, g, nt > 0 && sh.done_ok, p.TC, NMT);
  } else if (sh.done_ok) {
    // ---- O^T / l, written by all eight warps: warp w reads TMEM lane quarter
    // w & 3 (value channels) and every other 16-head column group from w >> 2
    tc::fence_after_sync();
    const int quarter = warp & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool part = p.S > 1, bf = !part && p.out_dtype == HSA_BF16;
    const int64_t head0 = static_cast<int64_t>(b) * p.Hq + g * p.HG;
    float* of = part ? p.po + ((static_cast<int64_t>(b) * p.S + s) * p.Hq + g * p.HG) * p.Dv
                     : reinterpret_cast<float*>(p.out) + head0 * p.Dv;
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.out) + head0 * p.Dv;
    for (int m = 0; m < NMT; ++m) {
      const int dv = m * kKeys + quarter * 32 + lane;
      for (int q16 = warp >> 2; q16 < kN / 16; q16 += 2) {
        uint32_t acc[16];
        tc::tmem_ld16(lane_addr + (TC + m) * kN + q16 * 16, acc);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = q16 * 16 + i;
          if (h < p.HG) {
            const float o = __uint_as_float(acc[i]) * sh.inv[h];
            const int64_t at = static_cast<int64_t>(h) * p.Dv + dv;
            if (bf) ob[at] = __float2bfloat16_rn(o);
            else of[at] = o;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
  if (selector && p.topk_out) write_topk_sorted(p, ring, b, geo, static_cast<int>(sh.sel_n));
}

// Merges the split partials: o = sum_s e^(lse_s - lse) o_s, lse = log sum_s e^lse_s.
// One thread per two 16-byte groups of value channels of one head: it loads
// the head's S partial log-sum-exps itself (the same few words for every
// thread of a head: cached), forms the weights in registers and combines with
// every split's partial loads in flight; no shared memory, no barriers.
constexpr int kMaxSplits = 1024;
constexpr int kCombineBlock = 128;  // threads per combine CTA
constexpr int kCombineChunk = 8;    // splits whose loads are in flight together

// One thread per 4 output channels of one head: the splits' partial outputs
// and log-sum-exps, combined in chunks of kCombineChunk splits (every load of
// a chunk in flight before its arithmetic) with a running maximum.
__global__ void __launch_bounds__(kCombineBlock) attn_combine_kernel(const float* __restrict__ po,
                                                                   const float* __restrict__ plse,
                                                                   int S, int64_t BH, int Hq, int Dv,
                                                                   void* out, int out_dtype,
                                                                   float* lse) {
  pdl_wait();
  pdl_trigger();
  const int d4n = Dv / 4;
  const int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gi >= BH * d4n) return;
  const int64_t head = gi / d4n;  // b * Hq + h
  const int d4 = static_cast<int>(gi % d4n);
  const int64_t b = head / Hq, h = head % Hq;
  const float* ls = plse + b * S * Hq + h;
  const float4* p4 = reinterpret_cast<const float4*>(po + (b * S * Hq + h) * Dv) + d4;
  const int64_t split4 = static_cast<int64_t>(Hq) * Dv / 4;  // float4s between splits
  float mx = -INFINITY, tot = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
  for (int s0 = 0; s0 < S; s0 += kCombineChunk) {
    float l[kCombineChunk];
    float4 v[kCombineChunk];
#pragma unroll
    for (int j = 0; j < kCombineChunk; ++j) {
      const int s = s0 + j;
      l[j] = s < S ? __ldg(ls + static_cast<int64_t>(s) * Hq) : -INFINITY;
      v[j] = s < S ? __ldcs(p4 + s * split4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < kCombineChunk; ++j) cm = fmaxf(cm, l[j]);
    if (cm == -INFINITY) continue;  // nothing attended in this chunk
    const float nm = fmaxf(mx, cm);
    const float r = mx == -INFINITY ? 0.f : __expf(mx - nm);  // rescales what came before
    tot *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int j = 0; j < kCombineChunk; ++j) {
      const float w = l[j] == -INFINITY ? 0.f : __expf(l[j] - nm);
      tot += w;
      acc.x = fmaf(w, v[j].x, acc.x);
      acc.y = fmaf(w, v[j].y, acc.y);
      acc.z = fmaf(w, v[j].z, acc.z);
      acc.w = fmaf(w, v[j].w, acc.w);
    }
    mx = nm;
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  const int64_t at = head * Dv + 4 * d4;
  if (out_dtype == HSA_BF16) {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&p0);
    pk.y = *reinterpret_cast<const uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + at) = pk;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + at) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (d4 == 0 && lse) lse[head] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

}  // namespace

AttnPlan attn_plan(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W, int64_t extra_slots) {
  AttnPlan pl;
  // every head of a token in one CTA when they fit the MMA width (one gather per row)
  pl.HG = static_cast<int>(Hq <= 32 ? Hq : (Hq % 64 == 0 ? 64 : 32));
  pl.N = pl.HG <= 16 ? 16 : (pl.HG <= 32 ? 32 : 64);
  pl.G = static_cast<int>(Hq / pl.HG);
  const int64_t slots = W + extra_slots;
  const int64_t tiles = slots > 0 ? (slots + kKeys - 1) / kKeys : 1;
  int64_t S = device_sms() / (B * pl.G);
  if (S < 1) S = 1;
  if (S > kMaxSplits) S = kMaxSplits;
  if (S > tiles) S = tiles;
  // whole tiles per split: a ring item's time is set by the gather latency,
  // not by its live rows, so a partly masked tile costs about a full one
  const int64_t tps = (tiles + S - 1) / S;
  pl.sps = tps * kKeys;
  pl.S = static_cast<int>((tiles + tps - 1) / tps);
  pl.cl = pl.S >= 2 && pl.S <= kMaxCl ? 1 : 0;
  const int NSL = static_cast<int>(Dqk / 64), NMT = static_cast<int>(Dv / 128);
  const int tc_fit = 512 / pl.N - NMT;  // TMEM columns left for S^T tiles
  pl.TC = tc_fit < kMaxTC ? tc_fit : kMaxTC;
  pl.smem = static_cast<size_t>(kRing) * kPairBytes + attn_q_region(NSL, pl.N) + 2 * pl.N * 128 + 1024;
  // a fused selection's survivors live in the even tiles' P^T buffer, or
  // after it when it is smaller than kSelMax composites
  if (2 * pl.N * 128 < kSelMax * 8) pl.smem += kSelMax * 8;
  // keep co-resident CTAs within the SM's 512 TMEM columns
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>((pl.TC + NMT) * pl.N)) cols <<= 1;
  // (at most n = 512 / cols CTAs fit the TMEM, so shared memory must keep
  // n + 1 of them from being resident together)
  const size_t per_sm = 227 * 1024;
  const size_t floor_bytes = per_sm / (512 / cols + 1) + 1;
  if (pl.smem < floor_bytes) pl.smem = floor_bytes;
  return pl;
}

bool attn_fused_ok(const AttnPlan& pl, int64_t k, int64_t max_row) {
  return k >= 1 && k <= kSelMaxK && max_row > 0 && max_row <= kSelRowMax && pl.G == 1 &&
         (pl.S == 1 || pl.cl);
}

size_t attn_workspace_bytes(const AttnPlan& pl, int64_t B, int64_t Hq, int64_t Dv) {
  size_t bytes = kWsHeader;
  if (pl.S > 1 && !pl.cl) {
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
  p.T = a.T < 1 ? 1 : a.T;
  p.Wr = static_cast<int>(a.Wr > 0 ? a.Wr : a.W);
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
  p.sps = pl.sps;
  p.TC = pl.TC;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.out = a.out;
  p.out_dtype = a.out_dtype;
  p.lse = a.lse;
  p.status = status;
  p.early = a.only_idx_pending ? 1 : (a.append_pending && !a.idx && !a.sel_scores ? 2 : 0);
  p.cl = pl.cl;
  p.sel_scores = a.sel_scores;
  p.row_hist = a.row_hist;
  p.cand_ws = a.cand_ws;
  p.topk_out = a.topk_out;
  const bool fused = a.sel_scores != nullptr;
  char* w = static_cast<char*>(ws) + kWsHeader;
  p.po = reinterpret_cast<float*>(w);
  p.plse = reinterpret_cast<float*>(
      w + ((static_cast<size_t>(a.B) * pl.S * a.Hq * a.Dv * 4 + 255) & ~size_t(255)));
  const unsigned grid = static_cast<unsigned>(a.B * pl.G * pl.S);
  CUtensorMap qmap, swamap;
  cudaError_t e = make_tmap_2d_bf16(&qmap, a.q, a.Dqk, a.B * a.Hq, 64, pl.N, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  // full 128-row windows are loaded by TMA (a map over the ring's rows; the
  // ring then holds exactly the window)
  const int swa_tma = a.swa && a.W == kKeys && p.Wr == a.W && p.T == 1 ? 1 : 0;
  swamap = qmap;  // (unused unless swa_tma)
  if (swa_tma) {
    e = make_tmap_2d_bf16(&swamap, a.swa, a.Dqk, a.B * a.W, 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  // dense tiles of 128 live compressed rows are loaded by TMA (a map over
  // the pool's rows)
  CUtensorMap poolmap = qmap;  // (unused unless pool_tma)
  const int pool_tma = !fused && a.extra && !a.idx && a.sp.limit > 0 ? 1 : 0;
  if (pool_tma) {
    e = make_tmap_2d_bf16(&poolmap, a.extra, a.Dqk, a.sp.limit, 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  auto* kernel = fused ? (pl.N == 16 ? attn_kernel<16, true>
                                     : (pl.N == 32 ? attn_kernel<32, true> : attn_kernel<64, true>))
                       : (pl.N == 16 ? attn_kernel<16, false>
                                     : (pl.N == 32 ? attn_kernel<32, false> : attn_kernel<64, false>));
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(pl.smem));
  if (e != cudaSuccess) return e;
  e = launch_kc(kernel, dim3(grid), dim3(kThreads), pl.smem, stream, pdl,
                static_cast<unsigned>(pl.cl ? pl.S : 0), qmap, swamap, swa_tma, poolmap, pool_tma,
                p);
  if (e != cudaSuccess || pl.S == 1 || pl.cl) return e;
  const int64_t bh = a.B * a.Hq;
  const int64_t threads = bh * (a.Dv / 4);  // one per 4 channels of a head
  return launch_k(attn_combine_kernel,
                  dim3(static_cast<unsigned>((threads + kCombineBlock - 1) / kCombineBlock)),
                  dim3(kCombineBlock),
                  0, stream, true, static_cast<const float*>(p.po),
                  static_cast<const float*>(p.plse), pl.S, bh, p.Hq, p.Dv, a.out, a.out_dtype,
                  a.lse);
}

}  // namespace hsa
