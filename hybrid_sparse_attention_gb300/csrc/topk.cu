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
// Otherwise every row is cut into chunks of CH scores (about one chunk per
// SM), one CTA per chunk, in two launches:
//   1. histogram: each CTA histograms the top 11 key bits (digit 1) of its
//      chunk in shared memory (16-byte loads) and adds the non-zero bins into
//      the row's global histogram.  The row's last CTA to finish (atomic
//      ticket, no waiting) scans it from the top for the threshold digit d1:
//      fewer than k keys lie above bin d1, at least k at or above it.
//   2. select: each warp re-reads its share of the chunk (from L2: it was
//      just read) and keeps every key at or above bin d1 as a composite,
//      written over the share's own positions of the workspace, with its
//      count: no atomics, no reservations.  The row's last CTA gathers the
//      lists (keys above bin d1 are winners, keys in it candidates), picks
//      the missing winners by a radix select over the candidates' other 53
//      composite bits, sorts the k survivors (bitonic runs of 32 in each
//      warp, merged by binary-search ranking) and writes them.  It leaves the
//      row's workspace zeroed.
#include "common.cuh"
#include "internal.h"
#include "select_core.cuh"

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

struct RowState {
  uint32_t n_cand;   // clustered path, heavy ties: candidates written to the workspace
  uint32_t done1;    // CTAs finished with pass 1
  uint32_t done2;    // CTAs finished with pass 2
  uint32_t digit;    // threshold digit d1 (pass 1 result)
};

struct Ws {
  uint32_t* status;
  RowState* rows;    // [B]
  uint32_t* hist;    // [B][kBins] digit 1
  uint32_t* wcount;  // [chunks][kWarps] pass 2: composites each warp kept
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
    wcount = hist + align256(sizeof(uint32_t) * kBins * B);
    cand = wcount + align256(sizeof(uint32_t) * kWarps * chunks);
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

// Live rows of sequence b (an invalid sequence is flagged in pass 1 and
// treated as empty by both passes).
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

// ---------------------------------------------------------------- pass 1

__global__ void __launch_bounds__(kThreads, 2) topk_hist_kernel(const float* __restrict__ scores,
                                                            Spans sp, int B, int k,
                                                            int64_t chunk, Ws ws) {
  __shared__ uint32_t s_hist[kBins];
  __shared__ uint32_t s_scan[33], s_out[2];
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  int row;
  int64_t piece, npieces;
  if (!locate_piece(B, blockIdx.x, ChunkPieces{sp, chunk}, &row, &piece, &npieces)) return;
  if (!sp.valid(row)) {
    if (threadIdx.x == 0 && piece == 0) set_status(ws.status, HSA_DEV_BOUNDS);
    return;
  }
  const int64_t n = row_count(sp, row);
  if (n <= k) return;  // every score is selected: no threshold needed
  for (int i = threadIdx.x; i < kBins; i += kThreads) s_hist[i] = 0;
  __syncthreads();
  const uint32_t* base = reinterpret_cast<const uint32_t*>(scores + sp.start(row));
  const int64_t lo = piece * chunk, hi = min(n, lo + chunk);
  bool nan = false;
  auto count_key = [&](uint32_t u) {
    nan |= is_nan_bits(u);
    atomicAdd(&s_hist[order_key(u) >> kShift1], 1u);
  };
  // 16-byte loads when the chunk starts 16-byte aligned (eight in flight per thread)
  int64_t done = lo;
  if ((reinterpret_cast<uintptr_t>(base + lo) & 15u) == 0) {
    const int64_t nv = (hi - lo) >> 2;
    const uint4* b4 = reinterpret_cast<const uint4*>(base + lo);
    constexpr int kV = 8;
    for (int64_t v0 = threadIdx.x; v0 < nv; v0 += kThreads * kV) {
      uint4 w[kV];
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        const int64_t v = v0 + j * kThreads;
        w[j] = v < nv ? __ldcg(b4 + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        if (v0 + j * kThreads < nv) {
          count_key(w[j].x);
          count_key(w[j].y);
          count_key(w[j].z);
          count_key(w[j].w);
        }
      }
    }
    done = lo + nv * 4;
  }
  constexpr int kU = 16;  // scalar loads in flight per thread
  for (int64_t i0 = done + threadIdx.x; i0 < hi; i0 += kThreads * kU) {
    uint32_t u[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t i = i0 + j * kThreads;
      u[j] = i < hi ? __ldcg(base + i) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kU; ++j)
      if (i0 + j * kThreads < hi) count_key(u[j]);
  }
  if (nan) set_status(ws.status, HSA_DEV_NAN);
  __syncthreads();
  uint32_t* gh = ws.hist + static_cast<int64_t>(row) * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (s_hist[i]) atomicAdd(gh + i, s_hist[i]);
  // the row's last CTA finds the threshold digit
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&ws.rows[row].done1, 1u) == npieces - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = threadIdx.x; i < kBins; i += kThreads) s_hist[i] = __ldcg(gh + i);
  __syncthreads();
  uint32_t above;
  const uint32_t d = find_digit(s_hist, kBins, static_cast<uint32_t>(k), &above, s_scan, s_out);
  if (threadIdx.x == 0) {
    ws.rows[row].digit = d;
    ws.rows[row].done1 = 0;
  }
}

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

// ---------------------------------------------------------------- pass 2

// Warp w of a chunk's CTA keeps, from its contiguous share of the chunk,
// every score at or above bin d1 (every score when the row has at most k)
// as a composite, written to the row's workspace over the share's own
// positions (a share never keeps more than it holds), and records how many.
// No atomics.  The row's last CTA gathers those lists, settles the boundary
// and sorts.
__global__ void __launch_bounds__(kThreads, 2) topk_select_kernel(const float* __restrict__ scores,
                                                              Spans sp, int B, int k,
                                                              int64_t chunk, Ws ws,
                                                              int32_t* __restrict__ idx_out,
                                                              float* __restrict__ vals_out) {
  __shared__ uint64_t s_sel[kMaxK];
  __shared__ uint64_t s_cand[kSmemCand];
  __shared__ uint32_t s_hist[kBins];  // list offsets, then select scratch
  __shared__ uint32_t s_scan[33], s_out[2], s_count, s_ccount;
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  int row;
  int64_t piece, npieces;
  if (!locate_piece(B, blockIdx.x, ChunkPieces{sp, chunk}, &row, &piece, &npieces)) return;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  const int64_t n = row_count(sp, row);
  const bool all = n <= k;
  const uint32_t d1 = all ? 0u : __ldcg(&ws.rows[row].digit);
  const int64_t off = sp.start(row);
  const uint32_t* base = reinterpret_cast<const uint32_t*>(scores + off);
  RowState* rs = ws.rows + row;
  const int64_t lo = piece * chunk, hi = min(n, lo + chunk);
  const int64_t wsub = chunk / kWarps;
  const int64_t wlo = lo + warp * wsub, whi = min(hi, wlo + wsub);
  {
    uint64_t* dst = ws.cand + off + wlo;
    uint32_t cnt = 0;
    auto keep = [&](uint32_t u, int64_t i, bool in) {
      const uint32_t key = order_key(u);
      const bool take = in && (all || (key >> kShift1) >= d1);
      const uint32_t m = __ballot_sync(0xffffffffu, take);
      if (take) dst[cnt + __popc(m & lt)] = composite(key, static_cast<uint32_t>(i));
      cnt += __popc(m);
    };
    int64_t done = wlo;
    if (wlo < whi && (reinterpret_cast<uintptr_t>(base + wlo) & 15u) == 0) {
      // 16-byte loads, eight in flight per lane (the trip count is the warp's)
      const int64_t nv = (whi - wlo) >> 2;
      const uint4* b4 = reinterpret_cast<const uint4*>(base + wlo);
      constexpr int kV = 8;
      for (int64_t v0 = 0; v0 < nv; v0 += 32 * kV) {
        uint4 w[kV];
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          const int64_t v = v0 + j * 32 + lane;
          w[j] = v < nv ? __ldcg(b4 + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kV; ++j) {
          const int64_t v = v0 + j * 32 + lane;
          const bool in = v < nv;
          const int64_t i = wlo + 4 * v;
          keep(w[j].x, i, in);
          keep(w[j].y, i + 1, in);
          keep(w[j].z, i + 2, in);
          keep(w[j].w, i + 3, in);
        }
      }
      done = wlo + nv * 4;
    }
    for (int64_t i0 = done; i0 < whi; i0 += 32 * 8) {
      uint32_t u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = i0 + j * 32 + lane;
        u[j] = i < whi ? __ldcg(base + i) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t i = i0 + j * 32 + lane;
        keep(u[j], i, i < whi);
      }
    }
    if (lane == 0) ws.wcount[static_cast<int64_t>(blockIdx.x) * kWarps + warp] = cnt;
  }
  __threadfence();
  __syncthreads();
  if (t == 0) s_last = atomicAdd(&rs->done2, 1u) == npieces - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- the row's last CTA: gather the lists, finish the selection, write the result
  const uint32_t kk = static_cast<uint32_t>(n < k ? n : k);
  const int64_t first_blk = static_cast<int64_t>(blockIdx.x) - piece;
  const int64_t nl = npieces * kWarps;
  // visits every kept composite once, list by list (lists in kThreads-sized
  // groups: counts scanned into offsets), as fn(x, e) with e its rank in that order
  auto for_each_kept = [&](auto&& fn) {
    uint32_t carry = 0;
    for (int64_t l0 = 0; l0 < nl; l0 += kThreads) {
      const int64_t l = l0 + t;
      const uint32_t c = l < nl ? __ldcg(ws.wcount + first_blk * kWarps + l) : 0u;
      uint32_t tot;
      const uint32_t incl = block_inclusive_sum<uint32_t>(c, s_scan, &tot);
      s_hist[t] = incl - c;
      __syncthreads();
      const int nlc = static_cast<int>(nl - l0 < kThreads ? nl - l0 : kThreads);
      constexpr int kG = 4;  // composites per thread per round: their loads in flight together
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
            const int64_t lg = l0 + a;
            x[u] = __ldcg(ws.cand + off + (lg / kWarps) * chunk + (lg % kWarps) * wsub + (e - s_hist[a]));
          }
        }
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const uint32_t e = e0 + u * kThreads + t;
          fn(x[u], e < tot, carry + e);
        }
      }
      __syncthreads();  // s_hist and s_scan are reused by the next group
      carry += tot;
    }
  };
  if (t == 0) {
    s_count = 0;
    s_ccount = 0;
  }
  __syncthreads();
  for_each_kept([&](uint64_t x, bool in, uint32_t) {
    const uint32_t dig = static_cast<uint32_t>(x >> (32 + kShift1));
    const bool w = in && (all || dig > d1), c = in && !all && dig == d1;
    const uint32_t pw = warp_append(&s_count, w, 0xffffffffu);
    if (w && pw < static_cast<uint32_t>(kMaxK)) s_sel[pw] = x;
    const uint32_t pc = warp_append(&s_ccount, c, 0xffffffffu);
    if (c && pc < static_cast<uint32_t>(kSmemCand)) s_cand[pc] = x;
  });
  __syncthreads();
  const uint32_t n_win = s_count < kk ? s_count : kk;
  const uint32_t nc = s_ccount;
  const uint32_t kept = s_count + s_ccount;
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
        select_rest(s_cand, nc, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out, 53);
      }
    } else {
      // heavy ties: pack every kept composite to the front of the row's
      // workspace (each read lies at or after its write, and every read of a
      // group precedes its writes), then select among those in bin d1
      for_each_kept([&](uint64_t x, bool in, uint32_t e) {
        __syncthreads();
        if (in) ws.cand[off + e] = x;
      });
      select_rest(ws.cand + off, kept, need, s_sel, &s_count, kMaxK, s_hist, s_scan, s_out, 53,
                  static_cast<uint64_t>(d1) << 53, 0x7ffull << 53);
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
  if (!all) {
    uint32_t* gh = ws.hist + static_cast<int64_t>(row) * kBins;
    for (int i = t; i < kBins; i += kThreads) gh[i] = 0;
  }
  if (t == 0) {
    rs->done2 = 0;
    rs->digit = 0;
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

int64_t topk_chunk(int64_t total_rows) {
  // about one chunk per SM (a single wave of both passes), 4,096 to 65,536 scores
  const int64_t want = total_rows / static_cast<int64_t>(device_sms());
  int64_t c = kMinChunk;
  while (c * 2 <= want && c < 65536) c *= 2;
  return c;
}

int topk_launch_count(int64_t total_rows, int64_t max_row) {
  return (max_row > 0 && max_row <= kClMax) || total_rows <= kClMax ? 1 : 2;
}

cudaError_t launch_topk(const float* scores, Spans sp, int B, int64_t total_rows, int k,
                        int32_t* idx, float* vals, void* ws, uint32_t* status,
                        cudaStream_t stream, int64_t max_row, bool pdl) {
  Ws w = ws_view(ws, B, total_rows, k, status);
  if (topk_launch_count(total_rows, max_row) == 1) {
    // every row fits one cluster: a single launch
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kClDynSmem));
    if (e != cudaSuccess) return e;
    return launch_k(topk_cluster_kernel, dim3(static_cast<unsigned>(B) * kCl), dim3(kThreads),
                    kClDynSmem, stream, pdl, scores, sp, k, w, idx, vals);
  }
  const int64_t chunk = topk_chunk(total_rows);
  const unsigned grid = static_cast<unsigned>((total_rows + chunk - 1) / chunk + B);  // >= chunks
  cudaError_t e = launch_k(topk_hist_kernel, dim3(grid), dim3(kThreads), 0, stream, pdl, scores, sp,
                           B, k, chunk, w);
  if (e != cudaSuccess) return e;
  return launch_k(topk_select_kernel, dim3(grid), dim3(kThreads), 0, stream, true, scores, sp, B, k,
                  chunk, w, idx, vals);
}

}  // namespace hsa
