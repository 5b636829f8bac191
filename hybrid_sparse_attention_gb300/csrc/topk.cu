// Lightning TopK: exact top-k per ragged row by radix select.
//
// [KD] "DeepSeek-V4: optimización de inferencia y RL ...", §Arquitectura del
// Sistema: Lightning TopK replaces the global sort with a radix-select
// reduction for the indexer's top-k.  [WK] "与 SGLang 团队聊 DeepSeek V4",
// §推理侧优化 (Lightning topk: the per-token top-k at 1M context went from
// ~100 us in plain PyTorch to ~15 us by raising parallelism).
//
// Result (bit-exact): per row, the first min(k, N) row-local indices of the
// scores ordered by value descending, lower index first among equal values.
//
// Keys.  A score f maps to an order-preserving uint32 key (larger key <=>
// larger value; -0.0 is first folded onto +0.0 so the two compare equal).
// The composite (key << 32) | (0xffffffff - index) is unique per element and
// orders elements exactly as the result requires, so selection and the final
// sort work on composites.
//
// Rows of at most 32,768 scores (every C4 row up to a 128K context) take one
// launch: a thread-block cluster per row (see "short rows" below).
//
// Longer rows take one launch too: every row is cut into chunks of CH
// scores (about one chunk per SM), one CTA per chunk, each reading its chunk
// once; a CTA counts and keeps only keys that can still reach the row's top k
// (a bar that rises as it reads), and the row's last CTA to finish (an
// atomic ticket, no waiting) selects and sorts (see "long rows" below).
#include "common.cuh"
#include "internal.h"
#include "select_core.cuh"
#include "tc.cuh"

namespace hsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;       // 11-bit digits
constexpr int kShift1 = 21;       // digit 1: key bits 31..21
constexpr int kMaxK = 2048;       // final sort buffer
constexpr int kSmemCand = 2560;   // boundary candidates staged in shared memory when they fit
constexpr int kMinChunk = 4096;   // scores per CTA of the chunked passes, at least
constexpr int kFastSort = kThreads;  // survivors ranked by warp runs + merge up to this many
constexpr int kLBinsWs = 4096;    // digit-1 bins of the chunked path (12-bit digits)

struct RowState {
  uint32_t n_cand;   // clustered path, heavy ties: candidates written to the workspace
  uint32_t done1;    // chunked path: CTAs finished with their chunk
  uint32_t bar;      // chunked path: the highest final bar of the row's CTAs
  uint32_t nlow;     // chunked path: ~(the lowest final bar), 0 before any
};

struct Ws {
  uint32_t* status;
  RowState* rows;    // [B]
  uint32_t* hist;    // [B][kLBins] chunked path: the row's digit-1 histogram
  uint32_t* wcount;  // [chunks] chunked path: composites each CTA kept
  uint64_t* cand;    // [total_rows], row b uses [offsets[b], offsets[b] + N_b)
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t rows, hist, wcount, cand, total;
  WsLayout(int64_t B, int64_t total_rows, int64_t /*k*/) {
    // chunks are at least kMinChunk scores, plus at most one partial chunk per row
    const int64_t chunks = total_rows / kMinChunk + 1 + B;
    rows = kWsHeader;
    hist = rows + align256(sizeof(RowState) * B);
    wcount = hist + align256(sizeof(uint32_t) * kLBinsWs * B);
    cand = wcount + align256(sizeof(uint32_t) * chunks);
    total = cand + align256(sizeof(uint64_t) * (total_rows > 0 ? total_rows : 1));
  }
};

Ws ws_view(void* base, int64_t B, int64_t total_rows, int64_t k, uint32_t* status) {
  WsLayout L(B, total_rows, k);
  char* p = static_cast<char*>(base);
  return Ws{status,
            reinterpret_cast<RowState*>(p + L.rows),
            reinterpret_cast<uint32_t*>(p + L.hist),
            reinterpret_cast<uint32_t*>(p + L.wcount),
            reinterpret_cast<uint64_t*>(p + L.cand)};
}

// Live rows of sequence b (an invalid sequence is flagged and treated as
// empty).
HSA_DEVINL int64_t row_count(const Spans& sp, int b) { return sp.count(b); }

struct ChunkPieces {
  Spans sp;
  int64_t chunk;
  HSA_DEVINL int64_t operator()(int b) const {
    const int64_t n = row_count(sp, b);
    const int64_t c = (n + chunk - 1) / chunk;
    return c > 0 ? c : 1;  // every row gets a CTA, even an empty one
  }
};

// ---------------------------------------------------------------- short rows: one cluster per row
//
// Rows of at most kClMax scores (every C4 row up to a 128K context) take one
// launch: a thread-block cluster of kCl CTAs per row, each holding an equal
// slice of the row (at most kClSlice scores) in shared memory.  The CTAs' digit-1 histograms are summed
// through distributed shared memory (each CTA reduces a quarter of the bins
// and broadcasts it), so every CTA finds d1 itself; each CTA then compacts
// its keys at or above bin d1 into shared memory, CTA 0 gathers the lists,
// finishes the selection and sorts.  No global atomics, no second launch.
// A threshold bin too full for the shared lists (heavy ties) sends its
// candidates through the workspace instead.

constexpr int kCl = 4;                     // CTAs per row (one cluster)
constexpr int kClU = 16;                   // scores per thread (rounds over the slice)
constexpr int kClSlice = kThreads * kClU;  // 8,192 scores per CTA
constexpr int kClMax = kCl * kClSlice;     // rows up to 32,768
constexpr int kClList = 2048;              // per-CTA list of composites at or above bin d1
static_assert(kBins == kCl * kThreads, "each CTA reduces kThreads bins, one per thread");
static_assert(kCl == 4, "the list gather selects among four prefix counts");

constexpr size_t kClDynSmem = sizeof(uint64_t) * (2 * kClList + kMaxK) + sizeof(uint32_t) * kClSlice;

// 4-byte asynchronous copy global -> shared (any 4-byte-aligned score).
HSA_DEVINL void cp_async4(uint32_t* dst, const uint32_t* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThreads, 2)
    topk_cluster_kernel(const float* __restrict__ scores, Spans sp, int k, Ws ws,
                        int32_t* __restrict__ idx_out, float* __restrict__ vals_out) {
  __shared__ uint32_t s_hist[kBins];   // this CTA's digit-1 histogram; later select scratch
  __shared__ uint32_t s_tot[kBins];    // the row's digit-1 histogram
  extern __shared__ uint64_t s_dyn[];
  uint64_t* s_loc = s_dyn;                // [kClList] this CTA's composites at or above bin d1
  uint64_t* s_sel = s_loc + kClList;      // [kMaxK] CTA 0: winners, then every survivor
  uint64_t* s_cand = s_sel + kMaxK;       // [kClList] CTA 0: candidates (bin d1); sort runs
  // [kClSlice] this CTA's slice: score bits, then order keys
  uint32_t* s_key = reinterpret_cast<uint32_t*>(s_cand + kClList);
  __shared__ uint32_t s_scan[33], s_out[2], s_nloc, s_count, s_ccount;
  const int t = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int row = static_cast<int>(blockIdx.x) / kCl;
  const bool valid = sp.valid(row);
  const int64_t n_raw = valid ? sp.raw_count(row) : 0;
  // longer than the caller's bound: flagged below, treated as empty
  const int n = n_raw > kClMax ? 0 : static_cast<int>(n_raw);
  if (rank == 0 && t == 0 && (!valid || n_raw > kClMax))
    set_status(ws.status, HSA_DEV_BOUNDS);
  const int64_t off = valid ? sp.start(row) : 0;
  const uint32_t* base = reinterpret_cast<const uint32_t*>(scores + off);
  const uint32_t kk = static_cast<uint32_t>(n < k ? n : k);
  const bool all = n <= k;  // every score is selected
  // equal slices of the row per CTA (each at most kClSlice since n <= kClMax)
  const int slice = (n + kCl - 1) / kCl;
  const int s0 = static_cast<int>(rank) * slice;
  const int s1 = s0 + slice < n ? s0 + slice : n;
  for (int i = t; i < kBins; i += kThreads) s_hist[i] = 0;
  if (t == 0) {
    s_count = 0;
    s_ccount = 0;
  }
  __syncthreads();
  // the row's geometry needs only the append's lengths (older than the
  // previous kernel); the scores need the wait
  pdl_wait();
  pdl_trigger();
  // The slice goes to shared memory with every copy in flight at once; the
  // passes over it below are rolled loops (this code runs once per launch,
  // so its instruction fetches cost more than loop overhead).
  const int m = s1 > s0 ? s1 - s0 : 0;
  const uint32_t* src = base + s0;
#pragma unroll 1
  for (int i = t; i < m; i += kThreads) cp_async4(s_key + i, src + i);
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  bool nan = false;
#pragma unroll 1
  for (int i = t; i < m; i += kThreads) {
    const uint32_t v = s_key[i];
    nan |= is_nan_bits(v);
    const uint32_t key = order_key(v);
    s_key[i] = key;
    if (!all) atomicAdd(&s_hist[key >> kShift1], 1u);
  }
  if (nan) set_status(ws.status, HSA_DEV_NAN);
  cluster_sync();  // every CTA's histogram is complete (and every CTA is running)
  {
    // reduce bin `bin` over the cluster, then broadcast the sum to every CTA
    const uint32_t bin = rank * kThreads + t;
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < kCl; ++q) sum += ld_cluster_u32(map_rank(&s_hist[bin], q));
#pragma unroll
    for (int q = 0; q < kCl; ++q) st_cluster_u32(map_rank(&s_tot[bin], q), sum);
  }
  cluster_sync();  // s_tot holds the row's histogram in every CTA
  uint32_t d1 = 0, above1 = 0, in1 = 0;
  if (!all) {
    d1 = find_digit(s_tot, kBins, kk, &above1, s_scan, s_out);
    in1 = s_tot[d1];
  }
  // heavy ties: the candidates go through the workspace (the same decision in every CTA)
  const bool heavy = !all && above1 + in1 > static_cast<uint32_t>(kClList);
  RowState* rs = ws.rows + row;
  {
    // compact: each thread counts its kept keys, one block scan gives every
    // thread its place, no atomics
    auto taken = [&](uint32_t key) {
      const uint32_t dig = key >> kShift1;
      return all || dig > d1 || (!heavy && dig == d1);
    };
    uint32_t cnt = 0;
#pragma unroll 4
    for (int i = t; i < m; i += kThreads) cnt += taken(s_key[i]) ? 1u : 0u;
    uint32_t nloc;
    uint32_t pos = block_inclusive_sum<uint32_t>(cnt, s_scan, &nloc) - cnt;
    if (t == 0) s_nloc = nloc;
#pragma unroll 4
    for (int i = t; i < m; i += kThreads) {
      const uint32_t key = s_key[i];
      if (taken(key)) {
        if (pos < static_cast<uint32_t>(kClList)) s_loc[pos] = composite(key, static_cast<uint32_t>(s0 + i));
        ++pos;
      }
    }
    if (heavy) {
#pragma unroll 1
      for (int i = t; i < kClSlice; i += kThreads) {
        const bool c = i < m && (s_key[i] >> kShift1) == d1;
        const uint32_t q = warp_append(&rs->n_cand, c, 0xffffffffu);
        if (c) ws.cand[off + q] = composite(s_key[i], static_cast<uint32_t>(s0 + i));
      }
      __threadfence();
    }
  }
  cluster_sync();  // every CTA's list is complete
  if (rank == 0) {
    // gather the lists (all of them at once): winners to s_sel, candidates to s_cand
    uint32_t pre[kCl + 1];
    pre[0] = 0;
#pragma unroll
    for (int q = 0; q < kCl; ++q) {
      const uint32_t nq = ld_cluster_u32(map_rank(&s_nloc, q));
      pre[q + 1] = pre[q] + (nq < static_cast<uint32_t>(kClList) ? nq : kClList);
    }
    for (uint32_t i0 = 0; i0 < pre[kCl]; i0 += kThreads) {
      const uint32_t i = i0 + t;
      const bool v = i < pre[kCl];
      uint32_t q = 0;
#pragma unroll
      for (int r = 1; r < kCl; ++r) q += i >= pre[r] ? 1u : 0u;
      const uint32_t first = q == 0 ? 0u : (q == 1 ? pre[1] : (q == 2 ? pre[2] : pre[3]));
      const uint64_t x = v ? ld_cluster_u64(map_rank(&s_loc[i - first], q)) : 0ull;
      const uint32_t dig = static_cast<uint32_t>(x >> (32 + kShift1));
      const bool w = v && (all || dig > d1), c = v && !all && dig == d1;
      const uint32_t pw = warp_append(&s_count, w, 0xffffffffu);
      if (w && pw < static_cast<uint32_t>(kMaxK)) s_sel[pw] = x;
      const uint32_t pc = warp_append(&s_ccount, c, 0xffffffffu);
      if (c && pc < static_cast<uint32_t>(kClList)) s_cand[pc] = x;
    }
  }
  cluster_sync();  // CTA 0 has read every list: the other CTAs may leave
  if (rank != 0) return;
  const uint32_t n_win = s_count < kk ? s_count : kk;
  const uint32_t need = kk - n_win;
  if (t == 0) s_count = n_win;
  __syncthreads();
  if (need > 0) {
    if (heavy) {
      const uint32_t nc = __ldcg(&rs->n_cand);
      select_rest(ws.cand + off, nc, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out, 53);
    } else if (need >= s_ccount) {
      const uint32_t nc = s_ccount;
      for (uint32_t i = t; i < nc && n_win + i < kk; i += kThreads) s_sel[n_win + i] = s_cand[i];
      __syncthreads();
      if (t == 0) s_count = n_win + (nc < need ? nc : need);
    } else {
      select_rest(s_cand, s_ccount, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out, 53);
    }
  }
  __syncthreads();
  const uint32_t have = s_count < kk ? s_count : kk;
  int32_t* out_i = idx_out + static_cast<int64_t>(row) * k;
  float* out_v = vals_out ? vals_out + static_cast<int64_t>(row) * k : nullptr;
  if (have <= static_cast<uint32_t>(kFastSort)) {
    uint64_t x;
    const uint32_t r = rank_desc<kWarps>(s_sel, static_cast<int>(have), s_cand, &x);
    if (r < have) {
      const uint32_t j = 0xffffffffu - static_cast<uint32_t>(x);
      out_i[r] = static_cast<int32_t>(j);
      if (out_v) out_v[r] = __uint_as_float(__ldcg(base + j));
    }
  } else {
    int p = 1;
    while (p < static_cast<int>(have)) p <<= 1;
    for (int i = have + t; i < p; i += kThreads) s_sel[i] = 0;  // sorts last
    bitonic_sort_desc(s_sel, p);
    for (uint32_t i = t; i < have; i += kThreads) {
      const uint32_t j = 0xffffffffu - static_cast<uint32_t>(s_sel[i]);
      out_i[i] = static_cast<int32_t>(j);
      if (out_v) out_v[i] = __uint_as_float(__ldcg(base + j));
    }
  }
  for (int i = static_cast<int>(have) + t; i < k; i += kThreads) {
    out_i[i] = -1;
    if (out_v) out_v[i] = -INFINITY;
  }
  if (heavy && t == 0) rs->n_cand = 0;  // leave the workspace zeroed
}

// ---------------------------------------------------------------- long rows: one launch, a chunk per CTA
//
// Every CTA streams its chunk of the row once, through a ring of cp.async
// stages in shared memory (each thread copies and reads its own eight scores
// per stage, so a stage needs no block barrier).  Digit 1 has 12 bits (key
// bits 31..20).
//
// Rising bar.  The k-th largest key of any part of a row is at most the
// row's k-th largest, so the bin holding the part's k-th largest key never
// lies above the row's threshold bin d1; nor does any bin with at least k
// keys at or above it among some of the part's keys.  A CTA counts its first
// stage whole and takes that stage's threshold bin as its bar; from then on
// a score is counted and kept only when it is at or above the bar (one float
// compare: bar_float), and after each stage one warp, in turn, raises the
// bar from the counts so far (read while other warps still add, each count
// a count of some of the bin's keys).  Every bin at or above the bar stays
// exactly counted, and every key at or above bin d1 is kept.  The passing
// scores of a stage are listed by ballots and handled 32 at a time by the
// warp, converged (count, keep).
//
// A CTA's kept keys go to the row's workspace over the chunk's own positions
// (a chunk never keeps more than it holds).  At the end the CTA finds its
// final bar from its exact counts, raises the row's bar (the highest final
// bar so far, also never above d1), adds its counts at or above the higher
// of the two to the row's histogram, drops the kept keys below it and takes
// an atomic ticket.  The row's last CTA finds d1 from the row's histogram at
// or above the row's bar, gathers the lists (keys above bin d1 are winners,
// keys in it candidates), picks the missing winners by radix select over the
// candidates' other 52 composite bits, sorts and writes the row.  It leaves
// the row's workspace zeroed.

constexpr int kLBits = 12;                   // digit 1 of long rows
constexpr int kLShift = 32 - kLBits;         // key bits 31..20
constexpr int kLBins = 1 << kLBits;          // 4,096
static_assert(kLBins == kLBinsWs, "the workspace holds kLBins bins per row");
constexpr int kStage = 4096;                 // scores per stage (16 KB)
constexpr int kHalf = kStage / 2;            // each thread copies 4 scores of each half
constexpr int kRing = 4;                     // stages in flight per CTA
static_assert(kStage == 8 * kThreads, "eight scores per thread per stage");
static_assert(kMinChunk % kStage == 0, "chunks are whole stages");
static_assert(sizeof(uint64_t) * (kMaxK + kSmemCand) + sizeof(uint32_t) * kThreads <=
                  sizeof(uint32_t) * kRing * kStage,
              "the last CTA's selection buffers fit in the ring");

constexpr size_t kChunkDynSmem = sizeof(uint32_t) * (kRing * kStage + kLBins);
constexpr int kRowBarPieces = 8;  // rows cut into this many pieces or more also prune at the row's counts

// One warp raises the CTA's bar (atomicMax on *s_bar) to the threshold bin
// of the counts in `hist` as read now, while other warps may still be adding
// to it: each count read is the number of some of the bin's keys, so at
// least `need` keys lie at or above the bin found, and the bar stays at or
// below the true threshold bin.  Scans the bins at or above the current bar.
HSA_DEVINL void warp_raise_bar(const uint32_t* hist, uint32_t* s_bar, uint32_t need) {
  const int lane = threadIdx.x & 31;
  const uint32_t b0 = *reinterpret_cast<volatile uint32_t*>(s_bar) >> kLShift;
  // lane L takes `per` bins from the top, after L * per of them: an odd
  // per makes the lanes' reads conflict-free
  const uint32_t nb = kLBins - b0;
  const uint32_t per = ((nb + 31) / 32) | 1u;
  const int hi = kLBins - 1 - lane * static_cast<int>(per);  // this lane's top bin
  const int lo = max(static_cast<int>(b0), hi - static_cast<int>(per) + 1);
  uint32_t sum = 0;
#pragma unroll 4
  for (int b = hi; b >= lo; --b) sum += hist[b];
  uint32_t incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  const uint32_t cross = __ballot_sync(0xffffffffu, incl - sum < need && incl >= need);
  if (lane != __ffs(cross) - 1) return;  // (no lane: fewer than need counted so far)
  // this lane's bins again (a count read again is no smaller, so the
  // crossing lies among them)
  uint32_t a = incl - sum;
  for (int b = hi; b >= lo; --b) {
    a += hist[b];
    if (a >= need) {
      atomicMax(s_bar, static_cast<uint32_t>(b) << kLShift);
      return;
    }
  }
}

// The threshold bin among the bins [b0, kLBins) of a kLBins-bin shared
// histogram, counted from the top: the d with (#above d) < need <= (#above d)
// + hist[d].  Returns b0 when the bins hold fewer than need keys.  All threads
// call; returns synchronised.
HSA_DEVINL uint32_t find_top_bin(const uint32_t* hist, uint32_t b0, uint32_t need,
                                 uint32_t* s_scan, uint32_t* s_out) {
  const uint32_t nb = kLBins - b0;
  const uint32_t per = (nb + kThreads - 1) / kThreads;
  const uint32_t first = threadIdx.x * per;  // bins counted from the top
  uint32_t sum = 0;
  for (uint32_t i = 0; i < per; ++i)
    if (first + i < nb) sum += hist[kLBins - 1 - (first + i)];
  if (threadIdx.x == 0) s_out[0] = b0;  // ordered before the writes below by the scan's barriers
  uint32_t total;
  uint32_t a = block_inclusive_sum<uint32_t>(sum, s_scan, &total) - sum;
  for (uint32_t i = 0; i < per && a < need; ++i) {
    const uint32_t bb = first + i;
    if (bb >= nb) break;
    const uint32_t c = hist[kLBins - 1 - bb];
    if (a + c >= need) s_out[0] = kLBins - 1 - bb;
    a += c;
  }
  __syncthreads();
  const uint32_t d = s_out[0];
  __syncthreads();
  return d;
}

__global__ void __launch_bounds__(kThreads, 2) topk_chunk_kernel(const float* __restrict__ scores,
                                                             Spans sp, int B, int k,
                                                             int64_t chunk, Ws ws,
                                                             int32_t* __restrict__ idx_out,
                                                             float* __restrict__ vals_out) {
  extern __shared__ __align__(16) uint32_t s_dyn32[];
  uint32_t* s_ring = s_dyn32;                  // [kRing][kStage] staged scores
  uint32_t* s_hist = s_ring + kRing * kStage;  // [kLBins] this chunk's digit-1 counts
  __shared__ uint32_t s_scan[33], s_out[2], s_count, s_ccount, s_kept, s_bar;
  __shared__ uint16_t s_wbuf[kStage];  // per warp: offsets of a stage's passing scores
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  int row;
  int64_t piece, npieces;
  if (!locate_piece(B, blockIdx.x, ChunkPieces{sp, chunk}, &row, &piece, &npieces)) return;
  const int t = threadIdx.x, lane = t & 31;
  // an invalid row is flagged and treated as empty
  if (!sp.valid(row) && t == 0 && piece == 0) set_status(ws.status, HSA_DEV_BOUNDS);
  const int64_t n = row_count(sp, row);
  const bool all = n <= k;  // every score is selected: no threshold
  const int64_t off = sp.start(row);
  const uint32_t* base = reinterpret_cast<const uint32_t*>(scores + off);
  RowState* rs = ws.rows + row;
  const int64_t lo = piece * chunk;
  const int m = static_cast<int>(n > lo ? min(n - lo, chunk) : 0);  // this chunk's scores
  const uint32_t* src = base + lo;
  uint64_t* list = ws.cand + off + lo;  // this chunk's kept composites
  for (int i = t; i < kLBins; i += kThreads) s_hist[i] = 0;
  if (t == 0) {
    s_kept = 0;
    s_bar = 0;
  }
  __syncthreads();

  // thread t's scores of stage r: chunk positions r*kStage + h*kHalf + 4t + j
  // (h = 0, 1; j = 0..3), at the same offsets of the stage's ring slot
  const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  const int nst = (m + kStage - 1) / kStage;
  const int nfull = vec ? m / kStage : 0;  // stages copied whole, 16 bytes at a time
  const uint32_t s_own = tc::smem_u32(s_ring) + 16u * t;
  const uint32_t* g_own = src + 4 * t;
  auto issue = [&](int r) {
    if (r < nfull) {
      const uint32_t sa = s_own + (r % kRing) * (4u * kStage);
      const uint32_t* g = g_own + r * kStage;
      tc::cp_async16_s(sa, g, 16u);
      tc::cp_async16_s(sa + 4u * kHalf, g + kHalf, 16u);
    } else if (r < nst) {
      uint32_t* slot = s_ring + (r % kRing) * kStage;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = r * kStage + h * kHalf + 4 * t;
        if (p >= m) continue;
        const int left = m - p;
        if (vec) {
          tc::cp_async16(slot + h * kHalf + 4 * t, src + p, left >= 4 ? 16u : 4u * left);
        } else {
          for (int j = 0; j < 4 && j < left; ++j) cp_async4(slot + h * kHalf + 4 * t + j, src + p + j);
        }
      }
    }
    tc::cp_async_commit();  // one group per stage, empty past the chunk's end
  };
#pragma unroll 1
  for (int r = 0; r < kRing; ++r) issue(r);

  uint32_t bar = 0;         // keys at or above bar (a bin's first key) are counted and kept
  float nanacc = 0.0f;      // NaN once any score was NaN
  uint16_t* wb = s_wbuf + (t >> 5) * (kStage / kWarps);
  const uint32_t lt = (1u << lane) - 1u;
  // The passing scores of a stage: the warp lists their offsets in the stage
  // (one ballot per score slot j places them), then handles 32 at a time,
  // converged: count (hist), and append to the chunk's list (keep).
  auto pass = [&](const float* f, uint32_t live, float fbar, const uint32_t* slot, uint32_t ibase,
                  bool hist, bool keep) {
    uint32_t nw = 0;  // the warp's passing scores
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool tk = ((live >> j) & 1u) && (all || f[j] >= fbar);
      const uint32_t mj = __ballot_sync(0xffffffffu, tk);
      if (mj) {
        if (tk) wb[nw + __popc(mj & lt)] = static_cast<uint16_t>((j >> 2) * kHalf + 4 * t + (j & 3));
        nw += __popc(mj);
      }
    }
    __syncwarp();
    for (uint32_t e0 = 0; e0 < nw; e0 += 32) {
      const bool in = e0 + lane < nw;
      const int o = in ? wb[e0 + lane] : 0;
      const uint32_t key = order_key(slot[o]);
      if (hist && in) atomicAdd(&s_hist[key >> kLShift], 1u);
      if (keep) {
        uint32_t pos = 0;
        if (lane == 0) pos = atomicAdd(&s_kept, min(32u, nw - e0));
        pos = __shfl_sync(0xffffffffu, pos, 0);
        if (in) list[pos + lane] = composite(key, ibase + o);
      }
    }
    __syncwarp();  // the list is free for the next stage
  };
  auto stage = [&](int r, bool full) {
    tc::cp_async_wait<kRing - 1>();  // this thread's copies of stage r have landed
    // another warp may have raised the bar since this warp's last stage
    bar = max(bar, *reinterpret_cast<volatile uint32_t*>(&s_bar));
    const uint32_t* slot = s_ring + (r % kRing) * kStage;
    const float4 fa = *reinterpret_cast<const float4*>(slot + 4 * t);
    const float4 fb = *reinterpret_cast<const float4*>(slot + kHalf + 4 * t);
    const float f[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
    uint32_t live = 0xffu;
    if (!full) {  // the chunk's last stage may be partial
      const int p0 = r * kStage + 4 * t;
      live = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) live |= (p0 + (j >> 2) * kHalf + (j & 3) < m ? 1u : 0u) << j;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) nanacc = max_nan(nanacc, (full || ((live >> j) & 1u)) ? f[j] : 0.0f);
    const uint32_t ibase = static_cast<uint32_t>(lo + r * kStage);
    if (r == 0 && !all) {
      // the first stage is counted whole and sets the CTA's first bar
      pass(f, live, -INFINITY, slot, ibase, true, false);
      __syncthreads();
      if (min(m, kStage) >= k) {
        bar = find_top_bin(s_hist, 0, static_cast<uint32_t>(k), s_scan, s_out) << kLShift;
        if (t == 0) s_bar = bar;
      }
      pass(f, live, bar_float(bar), slot, ibase, false, true);
    } else {
      pass(f, live, bar_float(bar), slot, ibase, !all, true);
    }
    // one warp per stage, in turn, raises the bar from the counts so far
    if (!all && r > 0 && (t >> 5) == r % kWarps) warp_raise_bar(s_hist, &s_bar, static_cast<uint32_t>(k));
    issue(r + kRing);
  };
#pragma unroll 1
  for (int r = 0; r < nfull; ++r) stage(r, true);
#pragma unroll 1
  for (int r = nfull; r < nst; ++r) stage(r, false);
  const bool nan = nanacc != nanacc;
  tc::cp_async_wait<0>();
  if (nan) set_status(ws.status, HSA_DEV_NAN);
  __syncthreads();  // every count and kept composite of the chunk is in place

  // the chunk's final bar; only bins at or above it can hold d1
  uint32_t* gh = ws.hist + static_cast<int64_t>(row) * kLBins;
  uint32_t pbar = 0;  // the higher of this CTA's final bar and the row's bar before it
  if (!all) {
    bar = max(bar, s_bar);
    if (bar || m >= k)
      bar = find_top_bin(s_hist, bar >> kLShift, static_cast<uint32_t>(k), s_scan, s_out) << kLShift;
    // The row's bar so far (the highest final bar of its CTAs done before
    // this one) never lies above d1 either: every CTA adds its counts and
    // prunes its list at the higher of the two.  The list's first group is
    // read while the row's bar comes back.
    constexpr int kG = 8;
    const uint32_t nk = s_kept;
    uint64_t x[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const uint32_t e = g * kThreads + t;
      x[g] = e < nk ? list[e] : 0ull;
    }
    if (t == 0) {
      s_out[0] = atomicMax(&rs->bar, bar);
      atomicMax(&rs->nlow, ~bar);
    }
    __syncthreads();
    pbar = max(bar, s_out[0]);
    for (int i = (pbar >> kLShift) + t; i < kLBins; i += kThreads)
      if (s_hist[i]) atomicAdd(gh + i, s_hist[i]);
    if (npieces >= kRowBarPieces) {
      // Many pieces: the row's counts so far (this CTA's included) give a
      // higher bar still.  Each count read counts some of its bin's keys, so
      // at least k of the row's keys lie at or above the bin where their sum
      // from the top reaches k: that bin is no higher than d1.
      __threadfence();  // this CTA's adds are visible to its reads below
      __syncthreads();
      const uint32_t b0 = pbar >> kLShift;
      for (int i = b0 + t; i < kLBins; i += kThreads) s_hist[i] = __ldcg(gh + i);
      __syncthreads();
      pbar = max(pbar, find_top_bin(s_hist, b0, static_cast<uint32_t>(k), s_scan, s_out) << kLShift);
      if (t == 0) atomicMax(&rs->bar, pbar);
    }
    // drop the kept keys below pbar: per group, masks and one block scan place
    // the survivors (no shared counter); each group is read whole before any
    // survivor of it is written (the scan's barriers), and survivors only move down
    if (pbar) {
      uint32_t kept = 0;
#pragma unroll 1
      for (uint32_t e0 = 0; e0 < nk; e0 += kThreads * kG) {
        if (e0) {
#pragma unroll
          for (int g = 0; g < kG; ++g) {
            const uint32_t e = e0 + g * kThreads + t;
            x[g] = e < nk ? list[e] : 0ull;
          }
        }
        uint32_t mask = 0;
#pragma unroll
        for (int g = 0; g < kG; ++g) {
          const uint32_t e = e0 + g * kThreads + t;
          mask |= (e < nk && static_cast<uint32_t>(x[g] >> 32) >= pbar ? 1u : 0u) << g;
        }
        const uint32_t c = __popc(mask);
        uint32_t tot;
        uint32_t pos = kept + block_inclusive_sum<uint32_t>(c, s_scan, &tot) - c;
#pragma unroll
        for (int g = 0; g < kG; ++g)
          if ((mask >> g) & 1u) list[pos++] = x[g];
        kept += tot;
      }
      if (t == 0) s_kept = kept;
    }
  }
  if (t == 0) ws.wcount[blockIdx.x] = s_kept;
  // the row's last CTA finishes the selection
  __threadfence();
  __syncthreads();
  if (t == 0) s_last = atomicAdd(&rs->done1, 1u) == npieces - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  uint64_t* s_sel = reinterpret_cast<uint64_t*>(s_ring);  // [kMaxK] winners, then survivors
  uint64_t* s_cand = s_sel + kMaxK;                       // [kSmemCand] candidates; sort scratch
  const uint32_t kk = static_cast<uint32_t>(n < k ? n : k);
  const int64_t first_blk = static_cast<int64_t>(blockIdx.x) - piece;
  // the first kThreads lists' counts, loaded with the histogram
  uint32_t* s_wc = reinterpret_cast<uint32_t*>(s_cand + kSmemCand);  // [kThreads]
  s_wc[t] = t < npieces ? __ldcg(ws.wcount + first_blk + t) : 0u;
  uint32_t d1 = 0, low = 0;  // d1; the lowest bin any CTA of the row added to
  if (!all) {
    // Every CTA added its counts at or above a bar no higher than d1, so the
    // row's histogram is whole from d1 up; the search may start at pbar.
    const uint32_t nlow = __ldcg(&rs->nlow);
    const uint32_t b0 = pbar >> kLShift;
    for (int i = b0 + t; i < kLBins; i += kThreads) s_hist[i] = __ldcg(gh + i);
    __syncthreads();
    d1 = find_top_bin(s_hist, b0, kk, s_scan, s_out);
    low = ~nlow >> kLShift;
  }
  // visits every kept composite once, list by list (lists in kThreads-sized
  // groups: counts scanned into offsets), kG per thread per round, as
  // fn(x, e0, tot, carry): thread t holds x[u] = composite e0 + u * kThreads + t
  // of the group's tot (valid below tot), carry composites before the group
  constexpr int kG = 8;  // composites per thread per round: their loads in flight together
  auto for_each_round = [&](auto&& fn) {
    uint32_t carry = 0;
    for (int64_t l0 = 0; l0 < npieces; l0 += kThreads) {
      const int64_t l = l0 + t;
      const uint32_t c = l0 == 0 ? s_wc[t] : (l < npieces ? __ldcg(ws.wcount + first_blk + l) : 0u);
      uint32_t tot;
      const uint32_t incl = block_inclusive_sum<uint32_t>(c, s_scan, &tot);
      s_hist[t] = incl - c;
      __syncthreads();
      const int nlc = static_cast<int>(npieces - l0 < kThreads ? npieces - l0 : kThreads);
      for (uint32_t e0 = 0; e0 < tot; e0 += kThreads * kG) {
        uint64_t x[kG];
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const uint32_t e = e0 + u * kThreads + t;
          x[u] = 0;
          if (e < tot) {
            int a = 0, z = nlc - 1;  // the last list starting at or before e
            while (a < z) {
              const int mid = (a + z + 1) >> 1;
              if (s_hist[mid] <= e) a = mid; else z = mid - 1;
            }
            x[u] = __ldcg(ws.cand + off + (l0 + a) * chunk + (e - s_hist[a]));
          }
        }
        fn(x, e0, tot, carry);
      }
      __syncthreads();  // s_hist and s_scan are reused by the next group
      carry += tot;
    }
  };
  // winners (above bin d1) to s_sel, candidates (in it) to s_cand: per-thread
  // masks and one block scan of the packed counts place them, no atomics
  uint32_t n_w = 0, n_c = 0;
  for_each_round([&](const uint64_t* x, uint32_t e0, uint32_t tot, uint32_t) {
    uint32_t wm = 0, cm = 0;
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      const bool in = e0 + u * kThreads + t < tot;
      const uint32_t dig = static_cast<uint32_t>(x[u] >> (32 + kLShift));
      wm |= (in && (all || dig > d1) ? 1u : 0u) << u;
      cm |= (in && !all && dig == d1 ? 1u : 0u) << u;
    }
    const uint32_t packed = __popc(wm) | (__popc(cm) << 16);
    uint32_t sum;
    const uint32_t before = block_inclusive_sum<uint32_t>(packed, s_scan, &sum) - packed;
    uint32_t pw = n_w + (before & 0xffffu), pc = n_c + (before >> 16);
#pragma unroll
    for (int u = 0; u < kG; ++u) {
      if ((wm >> u) & 1u) {
        if (pw < static_cast<uint32_t>(kMaxK)) s_sel[pw] = x[u];
        ++pw;
      }
      if ((cm >> u) & 1u) {
        if (pc < static_cast<uint32_t>(kSmemCand)) s_cand[pc] = x[u];
        ++pc;
      }
    }
    n_w += sum & 0xffffu;
    n_c += sum >> 16;
  });
  if (t == 0) {
    s_count = n_w;
    s_ccount = n_c;
  }
  __syncthreads();
  const uint32_t n_win = s_count < kk ? s_count : kk;
  const uint32_t nc = s_ccount;
  const uint32_t need = kk - n_win;
  __syncthreads();
  if (t == 0) s_count = n_win;
  __syncthreads();
  if (need > 0) {
    if (nc <= static_cast<uint32_t>(kSmemCand)) {
      if (need >= nc) {
        for (uint32_t i = t; i < nc && n_win + i < kk; i += kThreads) s_sel[n_win + i] = s_cand[i];
        __syncthreads();
        if (t == 0) s_count = n_win + (nc < need ? nc : need);
      } else {
        select_rest(s_cand, nc, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out, 64 - kLBits);
      }
    } else {
      // heavy ties: pack every kept composite to the front of the row's
      // workspace (each read lies at or after its write, and every read of a
      // group precedes its writes), then select among those in bin d1
      uint32_t kept = 0;  // every kept composite of the row
      for (int64_t l = 0; l < npieces; ++l) kept += __ldcg(ws.wcount + first_blk + l);
      for_each_round([&](const uint64_t* x, uint32_t e0, uint32_t tot, uint32_t carry) {
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const uint32_t e = e0 + u * kThreads + t;
          if (e < tot) ws.cand[off + carry + e] = x[u];
        }
      });
      constexpr uint64_t kDigitMask = ((1ull << kLBits) - 1) << (64 - kLBits);
      select_rest(ws.cand + off, kept, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out,
                  64 - kLBits, static_cast<uint64_t>(d1) << (64 - kLBits), kDigitMask);
    }
  }
  __syncthreads();
  const uint32_t have = s_count < kk ? s_count : kk;
  int32_t* out_i = idx_out + static_cast<int64_t>(row) * k;
  float* out_v = vals_out ? vals_out + static_cast<int64_t>(row) * k : nullptr;
  if (have <= static_cast<uint32_t>(kFastSort)) {
    uint64_t x;
    const uint32_t r = rank_desc<kWarps>(s_sel, static_cast<int>(have), s_cand, &x);
    if (r < have) {
      const uint32_t j = 0xffffffffu - static_cast<uint32_t>(x);
      out_i[r] = static_cast<int32_t>(j);
      if (out_v) out_v[r] = __uint_as_float(__ldcg(base + j));
    }
  } else {
    int p2 = 1;
    while (p2 < static_cast<int>(have)) p2 <<= 1;
    for (int i = have + t; i < p2; i += kThreads) s_sel[i] = 0;  // sorts last
    bitonic_sort_desc(s_sel, p2);
    for (uint32_t i = t; i < have; i += kThreads) {
      const uint32_t j = 0xffffffffu - static_cast<uint32_t>(s_sel[i]);
      out_i[i] = static_cast<int32_t>(j);
      if (out_v) out_v[i] = __uint_as_float(__ldcg(base + j));
    }
  }
  for (int i = static_cast<int>(have) + t; i < k; i += kThreads) {
    out_i[i] = -1;
    if (out_v) out_v[i] = -INFINITY;
  }
  // leave the row's workspace zeroed for the next call
  if (!all)
    for (int i = low + t; i < kLBins; i += kThreads) gh[i] = 0;
  if (t == 0) {
    rs->done1 = 0;
    rs->bar = 0;
    rs->nlow = 0;
  }
}

}  // namespace

size_t topk_workspace_bytes(int64_t B, int64_t total_rows, int64_t k) {
  return WsLayout(B, total_rows, k).total;
}

size_t topk_zero_prefix_bytes(int64_t B, int64_t total_rows, int64_t k) {
  return WsLayout(B, total_rows, k).wcount;
}

uint64_t* topk_cand_area(void* ws, int64_t B, int64_t total_rows, int64_t k) {
  return reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + WsLayout(B, total_rows, k).cand);
}

int64_t topk_chunk(int64_t total_rows, int k) {
  // About one chunk per SM (a single wave), 4,096 to 65,536 scores, and at
  // least 16 k: a chunk keeps at least its own k best until the row's counts
  // prune it, so shorter chunks hand the row's last CTA many more kept keys
  // than the row's top k (measured on 4 rows of 262,144: 16 k best).
  const int64_t want = total_rows / static_cast<int64_t>(device_sms());
  int64_t c = kMinChunk;
  while (c < 16 * static_cast<int64_t>(k) && c < 65536) c *= 2;
  while (c * 2 <= want && c < 65536) c *= 2;
  return c;
}

int topk_launch_count(int64_t, int64_t) { return 1; }

cudaError_t launch_topk(const float* scores, Spans sp, int B, int64_t total_rows, int k,
                        int32_t* idx, float* vals, void* ws, uint32_t* status,
                        cudaStream_t stream, int64_t max_row, bool pdl) {
  Ws w = ws_view(ws, B, total_rows, k, status);
  if ((max_row > 0 && max_row <= kClMax) || total_rows <= kClMax) {
    // every row fits one cluster
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kClDynSmem));
    if (e != cudaSuccess) return e;
    return launch_k(topk_cluster_kernel, dim3(static_cast<unsigned>(B) * kCl), dim3(kThreads),
                    kClDynSmem, stream, pdl, scores, sp, k, w, idx, vals);
  }
  const int64_t chunk = topk_chunk(total_rows, k);
  const unsigned grid = static_cast<unsigned>((total_rows + chunk - 1) / chunk + B);  // >= chunks
  cudaError_t e = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kChunkDynSmem));
  if (e != cudaSuccess) return e;
  return launch_k(topk_chunk_kernel, dim3(grid), dim3(kThreads), kChunkDynSmem, stream, pdl, scores,
                  sp, B, k, chunk, w, idx, vals);
}

}  // namespace hsa
