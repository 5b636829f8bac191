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
// the K-major layout the MMA descriptors describe.
//
// The kernel is bound by the key bytes (2*Di bytes per entry against 4*Hi*Di
// flops), so it is built to keep HBM busy: two persistent CTAs per SM each
// walk a contiguous range of 128-key tiles (tiles never straddle two
// sequences) through a two-stage TMA ring; warp 0 issues the loads, one lane
// of warp 1 issues the MMAs into alternating TMEM accumulators, and warps 2-5
// (one TMEM lane quarter each) drain the accumulators while the next tiles
// load.  Two CTAs with two stages each stream the pool faster than one CTA
// with four or six stages (the same or more bytes in flight per SM: 58 against
// 60-62 us over 1.18 M bf16 keys; 40 against 42-44 us for E4M3), and more
// than two CTAs per SM are slower again.
//
// E4M3 key pool (kFp8): the keys are 8-bit codes with one fp32 scale per entry
// (half the bytes), the MMAs are kind::f8f6f4 E4M3 x E4M3, and the queries
// are quantized the same way per (sequence, head) row inside the kernel: the
// epilogue warps write the E4M3 query rows of the CTA's next sequences into
// two shared-memory buffers ahead of the MMA (a buffer is refilled once the
// last tile of its previous sequence has been drained), so the kernel reads
// nothing the previous kernel writes before its first key tile.  With
// qhat = sq * code(q) and khat = sk * code(k), sq, sk > 0:
//     s[j] = sum_h w_h max(0, qhat_h . khat_j)
//          = sk_j * sum_h (w_h sq_h) max(0, code(q_h) . code(k_j)).
#include <cuda.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kTileRows = 128;  // M
constexpr int kQRows = 16;      // N (heads, padded)
constexpr int kStagesBf16 = 2;  // 36 KB stages (keys + queries)
constexpr int kStagesFp8 = 2;   // 16 KB stages (keys)
constexpr int kMaxStages = 2;
constexpr int kCtasPerSm = 2;
// Dynamic shared memory a CTA asks for at least, so that no third CTA shares
// an SM: two CTAs hold all 512 TMEM columns (kTmemCols each), and a third
// would wait in tcgen05.alloc until one of them has finished.
constexpr size_t kMinSmem = 80 * 1024;
constexpr int kFp8Di = 128;     // E4M3 keys: one 128-byte swizzle row per entry
constexpr uint32_t kQ8Bytes = kQRows * kFp8Di;  // one sequence's E4M3 query rows
constexpr int kThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMaxT = 4;        // query tokens per sequence
constexpr int kMaxSeqs = 4096;  // tile prefix table (built in a stage buffer before the ring starts)
constexpr int kAcc = 4;         // accumulators in TMEM (tiles the MMA may run ahead of the epilogue)
constexpr int kParts = 4;           // independent partial accumulators per tile
constexpr uint32_t kTmemCols = kAcc * kParts * kQRows;
static_assert(kCtasPerSm * kTmemCols <= 512, "the resident CTAs' accumulators exceed TMEM");
static_assert((kCtasPerSm + 1) * kMinSmem > 228 * 1024, "a further CTA would fit in shared memory");

struct IndexerParams {
  const float* w;  // [B, Hi]
  Spans sp;
  // Hi: query rows per sequence, T tokens of Hi / T heads each (multi-token
  // queries: row h belongs to token h / (Hi / T)); the sequence's key rows are
  // its last token's (sp counts them); token t scores the first
  // (seq_len + add - (T - 1 - t)) / ratio of them, into scores + t * tstride
  int B, Hi, Di, T;
  int64_t tstride;
  float* scores;
  uint32_t* status;
  int wait_mode;   // programmatic dependent launch: see launch_indexer in internal.h
  uint32_t* row_hist;  // per-sequence order-key histograms for the top-k (may be null)
  const float* key_scale;  // E4M3 keys: fp32 [total_rows]
  const uint16_t* iq;      // E4M3 keys: the bf16 queries [B, Hi, Di], quantized in the kernel
  uint64_t spin_ns;        // a pipeline wait gives up after this long ...
  uint32_t spin_polls;     // ... or this many polls (then HSA_DEV_TIMEOUT and the abort)
};

struct Shared {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t acc_full[kAcc], acc_empty[kAcc];
  uint64_t q8_full[2];      // E4M3 query buffer written (128 epilogue arrivals)
  float q8w[2][kQRows];     // the buffer's w[b, h] * query scale (0 past Hi)
  uint64_t fin;
  uint32_t tmem;
  int abort;
  int ntiles;
  int b0, first0;  // sequence owning this CTA's first tile, and its first tile
};

// Bounded wait of a pipeline role that also gives up when another role has
// aborted: after p.spin_polls failed checks (the first a non-blocking test) or
// p.spin_ns nanoseconds it sets HSA_DEV_TIMEOUT and the shared abort flag.
HSA_DEVINL bool wait_or_abort(Shared& sh, uint64_t* bar, uint32_t parity, const IndexerParams& p) {
  if (tc::mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_timer();
  for (uint32_t i = 1;; ++i) {
    if (*reinterpret_cast<volatile int*>(&sh.abort)) return false;
    if (i >= p.spin_polls || tc::global_timer() - t0 > p.spin_ns) {
      set_status(p.status, HSA_DEV_TIMEOUT);
      *reinterpret_cast<volatile int*>(&sh.abort) = 1;
      return false;
    }
    if (tc::mbar_try_wait(bar, parity)) return true;
  }
}

// Walks a CTA's contiguous range of tiles in order, keeping the owning
// sequence's first tile, pool start and live count in registers: a new
// sequence costs a few loads, a tile none, so no tile waits on a global load.
struct SeqCursor {
  int b = -1;
  int first = 0, next = 0;  // tiles [first, next) belong to sequence b
  int64_t start = 0, count = 0;
  HSA_DEVINL void load(const IndexerParams& p) {
    start = p.sp.start(b);
    count = p.sp.count(b);
    next = first + static_cast<int>((count + kTileRows - 1) / kTileRows);
  }
  // Tile of the current sequence holding a row the previous kernel may have
  // just written, or -1: the last live row, when one of the step's T tokens
  // completed a block (the lengths here are the ones after the previous
  // kernel; at most one block completes in a step of T <= ratio tokens).
  HSA_DEVINL int appended_tile(const IndexerParams& p) const {
    if (!p.sp.seq_len || count <= 0) return -1;
    const int64_t L = static_cast<int64_t>(p.sp.seq_len[b]) + p.sp.add;
    const int64_t L0 = L - p.T;
    if (L0 >= 0 && L / p.sp.ratio == L0 / p.sp.ratio) return -1;
    return first + static_cast<int>((count - 1) / kTileRows);
  }
  // Moves to the first sequence of the CTA's range (start) or to the next
  // sequence owning tiles; false when that sequence's tiles start at or past
  // t_end (or there is none).
  HSA_DEVINL bool step(const Shared& sh, const IndexerParams& p, bool start, int t_end) {
    if (start) {
      b = sh.b0;
      first = sh.first0;
      load(p);
      return first < t_end;
    }
    do {
      if (b + 1 >= p.B) return false;
      ++b;
      first = next;
      load(p);
    } while (next == first);
    return first < t_end;
  }
  HSA_DEVINL bool seek(const Shared& sh, const IndexerParams& p, int t) {
    if (b >= 0 && t < next) return false;
    if (b < 0) {
      b = sh.b0;
      first = sh.first0;
      load(p);
    }
    while (t >= next) {  // (empty sequences own no tiles and are stepped over)
      ++b;
      first = next;
      load(p);
    }
    return true;  // moved to a new sequence
  }
};

// E4M3 query rows of sequence b into buffer `buf` (the 128 epilogue threads,
// e = 0..127: head e / 8, channels 16 (e % 8) .. +16): per row amax over the
// 8 lanes of the head, code = e4m3(q * (448 / amax)) (round to nearest even,
// saturating), stored 128-byte swizzled as the MMA's K-major B operand; the
// head's weight w[b, h] * amax / 448 goes to q8w.  Then the buffer's barrier.
HSA_DEVINL void quantize_queries(const IndexerParams& p, Shared& sh, uint8_t* q8, int b, int buf,
                                 int e) {
  const int h = e >> 3, part = e & 7;
  float x[16];
  if (h < p.Hi) {
    const uint4* src = reinterpret_cast<const uint4*>(p.iq + (static_cast<int64_t>(b) * p.Hi + h) * kFp8Di +
                                                      part * 16);
    bf16x8_to_f32(__ldg(src), x);
    bf16x8_to_f32(__ldg(src + 1), x + 8);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.f;
  }
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const float inv = am > 0.f ? __fdiv_rn(448.f, am) : 0.f;
  uint32_t w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(x[4 * i], inv), __fmul_rn(x[4 * i + 1], inv)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(x[4 * i + 2], inv), __fmul_rn(x[4 * i + 3], inv)), __NV_SATFINITE, __NV_E4M3);
    w4[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  uint8_t* buf_base = q8 + buf * kQ8Bytes;
  *reinterpret_cast<uint4*>(buf_base + (h >> 3) * 1024 + (h & 7) * 128 + ((part ^ (h & 7)) << 4)) =
      make_uint4(w4[0], w4[1], w4[2], w4[3]);
  if (part == 0)
    sh.q8w[buf][h] = h < p.Hi ? p.w[static_cast<int64_t>(b) * p.Hi + h] * __fdiv_rn(am, 448.f) : 0.f;
  tc::fence_proxy_async_smem();
  tc::mbar_arrive(&sh.q8_full[buf]);
}

// kMulti: more than one query token per sequence (p.T > 1); the single-token
// instantiation carries none of the per-token bookkeeping.
template <bool kFp8, bool kMulti>
__global__ void __launch_bounds__(kThreads, 2) indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap qmap,
                                                             IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Programmatic dependent launch (wait_mode): 0 every thread waits first;
  // otherwise the prologue (tile table, barriers, TMEM) needs nothing the
  // previous kernel writes and only the TMA producer waits — before its first
  // key load (1), or right before the first tile holding a key the previous
  // kernel may have written, after triggering the next kernel (2).
  if (p.wait_mode == 0) {
    pdl_wait();
    pdl_trigger();
  }

  constexpr int kStages = kFp8 ? kStagesFp8 : kStagesBf16;
  const int kb_elems = kFp8 ? kFp8Di : (p.Di >= 64 ? 64 : p.Di);  // elements of one swizzle row
  const int nkb = kFp8 ? 1 : p.Di / kb_elems;
  const uint32_t a_kb = kFp8 ? kTileRows * kFp8Di : kTileRows * kb_elems * 2;
  const uint32_t b_kb = kFp8 ? 0u : kQRows * kb_elems * 2;
  const uint32_t stage_bytes = nkb * (a_kb + b_kb);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q8 = smem + kStages * stage_bytes;  // (kFp8) two E4M3 query buffers

  // tiles per sequence -> prefix table (block-wide scan in chunks of blockDim),
  // kept in the (not yet used) stage buffers just long enough to find the
  // sequence owning this CTA's first tile
  int* prefix = reinterpret_cast<int*>(smem);
  __shared__ int s_scan[33];
  int carry = 0;
  for (int base = 0; base < p.B; base += kThreads) {
    const int b = base + threadIdx.x;
    const int nt = b < p.B ? static_cast<int>((p.sp.count(b) + kTileRows - 1) / kTileRows) : 0;
    int total;
    const int incl = block_inclusive_sum<int>(nt, s_scan, &total);
    if (b < p.B) prefix[b] = carry + incl - nt;
    carry += total;
    __syncthreads();  // s_scan is reused by the next chunk
  }
  if (threadIdx.x == 0) {
    prefix[p.B] = carry;
    sh.ntiles = carry;
  }
  __syncthreads();
  const int ntiles = sh.ntiles;
  const int t_begin = static_cast<int>(static_cast<int64_t>(ntiles) * blockIdx.x / gridDim.x);
  const int t_end = static_cast<int>(static_cast<int64_t>(ntiles) * (blockIdx.x + 1) / gridDim.x);
  if (t_begin >= t_end) {
    if (p.wait_mode != 0 && threadIdx.x == 0) pdl_wait();  // complete only after the previous kernel
    return;
  }
  if (threadIdx.x == 0) {
    int lo = 0, hi = p.B - 1;  // largest b with prefix[b] <= t_begin
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= t_begin) lo = mid; else hi = mid - 1;
    }
    sh.b0 = lo;
    sh.first0 = prefix[lo];
  }
  __syncthreads();  // the stage buffers are free again

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&sh.full[s], 1);
      tc::mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      tc::mbar_init(&sh.acc_full[a], 1);
      tc::mbar_init(&sh.acc_empty[a], 128);
    }
    for (int q = 0; q < 2; ++q) tc::mbar_init(&sh.q8_full[q], 128);
    tc::mbar_init(&sh.fin, 1);
    sh.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sh.tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::tma_prefetch_map(&kmap);
      tc::tma_prefetch_map(&qmap);
      bool waited = p.wait_mode == 0;
      if (p.wait_mode == 1) {
        pdl_wait();
        waited = true;
      }
      pdl_trigger();
      (void)b_kb;
      SeqCursor cur;
      // the keys are read once: they leave L2 first, so the scores and
      // histograms written here stay for the top-k that reads them next
      const uint64_t keys_policy = tc::l2_policy_evict_first();
      int dep = -1;  // (wait_mode 2) tile that must wait for the previous kernel
      int issued = 0;
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int s = i % kStages;
        // before the wait: a new sequence's loads overlap it
        if (cur.seek(sh, p, t) && !waited) dep = cur.appended_tile(p);
        if (!waited && t == dep) {
          pdl_wait();
          waited = true;
        }
        if (i >= kStages &&
            !wait_or_abort(sh, &sh.empty[s], ((i / kStages) & 1) ^ 1, p))
          break;
        const int b = cur.b;
        const int64_t row0 = cur.start + static_cast<int64_t>(t - cur.first) * kTileRows;
        uint8_t* st = smem + s * stage_bytes;
        tc::mbar_arrive_expect_tx(&sh.full[s], stage_bytes);
        for (int kb = 0; kb < nkb; ++kb) {
          tc::tma_load_2d_hint(st + kb * a_kb, &kmap, kb * kb_elems, static_cast<int32_t>(row0),
                               &sh.full[s], keys_policy);
          if (!kFp8)
            tc::tma_load_2d(st + nkb * a_kb + kb * b_kb, &qmap, kb * kb_elems, b * p.Hi,
                            &sh.full[s]);
        }
        issued = i + 1;
      }
      // Every load issued lands in this CTA's shared memory before the CTA may
      // exit: after an abort the MMA may not have waited for the last stages.
      // (Only the last kStages can be outstanding; each stage's barrier is then
      // at most one phase behind.  The default bound: these loads do complete.)
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        tc::mbar_wait(&sh.full[j % kStages], (j / kStages) & 1, p.status);
      if (!waited) pdl_wait();  // the grid completes only after the previous kernel
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const tc::Swizzle sw = kFp8 || kb_elems == 64 ? tc::kSwizzle128B : tc::kSwizzle64B;
      const uint32_t sbo = kFp8 ? 8u * kFp8Di : 8u * kb_elems * 2;  // bytes between 8-row groups
      const uint32_t idesc =
          kFp8 ? tc::idesc_e4m3_f32(kTileRows, kQRows) : tc::idesc_bf16_f32(kTileRows, kQRows);
      SeqCursor mc;
      int ord = -1;  // (kFp8) ordinal of the tile's sequence in this CTA's range
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int s = i % kStages, a = i % kAcc;
        if (kFp8 && mc.seek(sh, p, t)) {
          ++ord;
          if (!wait_or_abort(sh, &sh.q8_full[ord & 1], (ord >> 1) & 1, p)) break;
        }
        if (!wait_or_abort(sh, &sh.full[s], (i / kStages) & 1, p)) break;
        if (i >= kAcc && !wait_or_abort(sh, &sh.acc_empty[a], ((i / kAcc) & 1) ^ 1, p))
          break;
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(smem + s * stage_bytes);
        if (kFp8) {
          // K = 32 codes (32 bytes) per MMA; each K-step into its own partial
          const uint32_t sb = tc::smem_u32(q8 + (ord & 1) * kQ8Bytes);
#pragma unroll
          for (int ks = 0; ks < kFp8Di / 32; ++ks) {
            const uint64_t da = tc::smem_desc(sa + ks * 32, 16, sbo, sw);
            const uint64_t db = tc::smem_desc(sb + ks * 32, 16, sbo, sw);
            tc::mma_f8(tmem + (a * kParts + ks % kParts) * kQRows, da, db, idesc, ks >= kParts);
          }
          tc::mma_commit(&sh.empty[s]);
          tc::mma_commit(&sh.acc_full[a]);
          continue;
        }
        const uint32_t sb = sa + nkb * a_kb;
        // K-step kk accumulates into partial kk % kParts: chains of small-N
        // MMAs on one accumulator would serialize
        for (int kb = 0; kb < nkb; ++kb) {
          for (int ks = 0; ks < kb_elems / 16; ++ks) {
            const int kk = kb * (kb_elems / 16) + ks;
            const uint64_t da = tc::smem_desc(sa + kb * a_kb + ks * 32, 16, sbo, sw);
            const uint64_t db = tc::smem_desc(sb + kb * b_kb + ks * 32, 16, sbo, sw);
            tc::mma_bf16(tmem + (a * kParts + kk % kParts) * kQRows, da, db, idesc, kk >= kParts);
          }
        }
        tc::mma_commit(&sh.empty[s]);
        tc::mma_commit(&sh.acc_full[a]);
      }
      tc::mma_commit(&sh.fin);  // drain before TMEM is freed
      tc::mbar_wait(&sh.fin, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;
    const int e = threadIdx.x - 64;  // 0..127 over the epilogue warps
    const int nparts = kFp8 ? kFp8Di / 32 : (p.Di / 16 < kParts ? p.Di / 16 : kParts);  // partials in use
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    SeqCursor cur;
    float wv[kQRows];
    int64_t nt[kMulti ? kMaxT : 1];  // (kMulti) each token's live rows of the current sequence
    const int hpt = p.Hi / p.T;      // heads per token
    // (kFp8) the E4M3 queries of the range's first two sequences; `ahead` is the
    // sequence of the last buffer written, `made` how many were written
    SeqCursor ahead;
    int made = 0, ord = -1;
    if (kFp8) {
      if (ahead.step(sh, p, true, t_end)) {
        quantize_queries(p, sh, q8, ahead.b, 0, e);
        made = 1;
        if (ahead.step(sh, p, false, t_end)) {
          quantize_queries(p, sh, q8, ahead.b, 1, e);
          made = 2;
        }
      }
      tc::named_barrier(1, 128);  // every buffer's weights visible to every epilogue thread
    }
    // A warp whose wait gave up (an abort) stops working; with kFp8 it keeps
    // walking the tiles so that every epilogue thread reaches the same named
    // barriers, where the warps agree on the abort.
    bool dead = false;
    // (kFp8) this thread's key scales of the next kPf tiles, loaded kPf tiles
    // ahead (a DRAM round trip per tile would otherwise bound the loop).  With
    // wait_mode 2 the scale of a row the previous kernel may have just written
    // is read only after the wait for that kernel, as the producer loads that
    // row's codes.
    constexpr int kPf = 4;
    float ksr[kPf];
    SeqCursor pc;
    bool ewaited = !kFp8 || p.wait_mode != 2;
    int pdep = -1;
    auto fetch_scale = [&](int tt) -> float {
      if (tt >= t_end) return 0.f;
      if (pc.seek(sh, p, tt) && !ewaited) pdep = pc.appended_tile(p);
      if (!ewaited && tt == pdep) {
        pdl_wait();
        ewaited = true;
      }
      const int64_t pp = tt - pc.first;
      return r < pc.count - pp * kTileRows ? p.key_scale[pc.start + pp * kTileRows + r] : 0.f;
    };
    if (kFp8) {
#pragma unroll
      for (int j = 0; j < kPf; ++j) ksr[j] = fetch_scale(t_begin + j);
    }
    for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
      const int a = i % kAcc;
      if (cur.seek(sh, p, t)) {
        ++ord;
        if (!kFp8) {
#pragma unroll
          for (int h = 0; h < kQRows; ++h)
            wv[h] = h < p.Hi ? __ldg(p.w + static_cast<int64_t>(cur.b) * p.Hi + h) : 0.f;
        }
        // each token's live rows (the last token's are the sequence's count)
        if (kMulti) {
#pragma unroll
          for (int q = 0; q < kMaxT; ++q) {
            int64_t n = cur.count;
            if (q < p.T - 1 && p.sp.seq_len) {
              n = (static_cast<int64_t>(p.sp.seq_len[cur.b]) + p.sp.add - (p.T - 1 - q)) / p.sp.ratio;
              n = n < 0 ? 0 : (n > cur.count ? cur.count : n);
            }
            nt[q] = q < p.T ? n : 0;
          }
        }
      }
      const int64_t piece = t - cur.first;
      const int64_t left = cur.count - piece * kTileRows;
      const int64_t row = cur.start + piece * kTileRows + r;
      float ks = 1.f;
      if (kFp8) {
        ks = ksr[0];
#pragma unroll
        for (int j = 0; j + 1 < kPf; ++j) ksr[j] = ksr[j + 1];
        ksr[kPf - 1] = dead ? 0.f : fetch_scale(t + kPf);
      }
      if (!dead) dead = !__all_sync(0xffffffffu, wait_or_abort(sh, &sh.acc_full[a], (i / kAcc) & 1, p));
      if (dead && !kFp8) break;
      if (!dead) {
      if (kFp8) {
        // written by the epilogue threads before the named barrier that
        // followed (at the start, or at the end of the previous sequence)
#pragma unroll
        for (int h = 0; h < kQRows; ++h) wv[h] = sh.q8w[ord & 1][h];
      }
      tc::fence_after_sync();
      float dot[kQRows];
#pragma unroll
      for (int h = 0; h < kQRows; ++h) dot[h] = 0.f;
      for (int pa = 0; pa < nparts; ++pa) {
        uint32_t acc[16];
        tc::tmem_ld16(tmem + lane_addr + (a * kParts + pa) * kQRows, acc);
        tc::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < kQRows; ++h) dot[h] += __uint_as_float(acc[h]);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&sh.acc_empty[a]);
      if (!kMulti) {
        const bool live = r < left;
        float sc = 0.f;
        if (live) {
#pragma unroll
          for (int h = 0; h < kQRows; ++h)
            if (h < p.Hi) sc = fmaf(wv[h], fmaxf(dot[h], 0.f), sc);
          if (kFp8) sc *= ks;
          p.scores[row] = sc;
        }
        // the top-k's histogram: one count in the bin of the score's top key
        // bits (a reduction: nothing waits for it).  The scores crowd into a
        // few bins, so the warp's lanes of one bin add once, by their count
        // (one atomic per score cost the E4M3 stream 6 us over 1.18 M keys).
        // The whole warp is here: `dead` is uniform over it.
        if (p.row_hist) {
          const uint32_t bin = live ? order_key(__float_as_uint(sc)) >> kRowHistShift : 0xffffffffu;
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (live && (threadIdx.x & 31) == __ffs(peers) - 1)
            atomicAdd(p.row_hist + static_cast<int64_t>(cur.b) * kRowHistBins + bin,
                      static_cast<uint32_t>(__popc(peers)));
        }
      } else {
        // token q: heads [q * hpt, (q + 1) * hpt), the rows visible to it
        const int64_t jrow = piece * kTileRows + r;  // row within the sequence
#pragma unroll
        for (int q = 0; q < (kMulti ? kMaxT : 1); ++q) {
          if (q < p.T && jrow < nt[q] && r < left) {
            float sc = 0.f;
#pragma unroll
            for (int h = 0; h < kQRows; ++h)
              if (h >= q * hpt && h < (q + 1) * hpt) sc = fmaf(wv[h], fmaxf(dot[h], 0.f), sc);
            if (kFp8) sc *= ks;
            p.scores[q * p.tstride + row] = sc;
            if (p.row_hist)
              atomicAdd(p.row_hist + (static_cast<int64_t>(cur.b) * p.T + q) * kRowHistBins +
                            (order_key(__float_as_uint(sc)) >> kRowHistShift),
                        1u);
          }
        }
      }
      }  // !dead
      if (kFp8 && (t + 1 == cur.next || t + 1 == t_end) && made == ord + 2) {
        // the sequence's last tile here is drained: its MMAs (and every
        // earlier one) are complete, so its buffer takes sequence ord + 2,
        // once every epilogue thread has read the buffer's weights (and
        // agreed whether any warp gave up)
        dead = tc::named_barrier_or(1, 128, dead);
        if (!dead && ahead.step(sh, p, false, t_end)) {
          quantize_queries(p, sh, q8, ahead.b, ord & 1, e);
          ++made;
        }
        tc::named_barrier(1, 128);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t indexer_smem_bytes(int Di, bool fp8) {
  const size_t need = fp8 ? static_cast<size_t>(kStagesFp8) * kTileRows * kFp8Di + 2 * kQ8Bytes + 1024
                          : static_cast<size_t>(kStagesBf16) * Di * 2 * (kTileRows + kQRows) + 1024;
  return need > kMinSmem ? need : kMinSmem;
}

cudaError_t launch_indexer(const void* iq, const float* w, const void* keys, Spans sp, int B, int Hi,
                           int Di, int64_t total_rows, float* scores, uint32_t* status,
                           cudaStream_t stream, bool pdl, int wait_mode, uint32_t* row_hist,
                           const float* key_scale, int T) {
  if (total_rows == 0) return cudaSuccess;
  if (B > kMaxSeqs || T < 1 || T > kMaxT || Hi * T > kQRows) return cudaErrorInvalidValue;
  Hi *= T;  // query rows per sequence
  const bool fp8 = key_scale != nullptr;
  if (fp8 && (Di != kFp8Di || Hi > kQRows)) return cudaErrorInvalidValue;
  const int kb_elems = Di >= 64 ? 64 : Di;
  const CUtensorMapSwizzle sw = kb_elems == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap kmap, qmap;
  cudaError_t e;
  if (fp8) {
    e = make_tmap_2d_u8(&kmap, keys, Di, total_rows, kFp8Di, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
    qmap = kmap;  // (unused: the queries are quantized in the kernel)
  } else {
    e = make_tmap_2d_bf16(&kmap, keys, Di, total_rows, kb_elems, kTileRows, sw);
    if (e == cudaSuccess)
      e = make_tmap_2d_bf16(&qmap, iq, Di, static_cast<int64_t>(B) * Hi, kb_elems, kQRows, sw);
  }
  if (e != cudaSuccess) return e;
  const size_t smem = indexer_smem_bytes(Di, fp8);
  auto kernel = fp8 ? (T > 1 ? indexer_kernel<true, true> : indexer_kernel<true, false>)
                    : (T > 1 ? indexer_kernel<false, true> : indexer_kernel<false, false>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(fp8 ? smem : indexer_smem_bytes(128)));
  if (e != cudaSuccess) return e;
  // persistent: two CTAs per SM, fewer when there are fewer tiles
  const int64_t tiles_bound = (total_rows + kTileRows - 1) / kTileRows + B;
  const int nres = kCtasPerSm * device_sms();
  const int grid = static_cast<int>(tiles_bound < nres ? tiles_bound : nres);
  IndexerParams p{w, sp, B, Hi, Di, T, total_rows, scores, status, pdl ? wait_mode : 0, row_hist,
                  key_scale, static_cast<const uint16_t*>(iq), wait_limit_ns(), wait_limit_polls()};
  return launch_k(kernel, dim3(grid), dim3(kThreads), smem, stream, pdl, kmap, qmap, p);
}

}  // namespace hsa
