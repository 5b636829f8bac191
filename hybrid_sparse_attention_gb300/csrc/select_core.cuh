// Device helpers of exact top-k selection on order-preserving keys, shared by
// the standalone top-k kernels and the layer's fused selection.
//
// A score's key is order_key(bits) (common.cuh); the composite
// (key << 32) | (0xffffffff - index) is unique per element and orders
// elements by value descending, lower index first among equal values, so
// selection and sorting work on composites.
#pragma once

#include "common.cuh"

namespace hsa {

HSA_DEVINL bool is_nan_bits(uint32_t u) { return (u & 0x7fffffffu) > 0x7f800000u; }

// max(a, b), NaN when either is NaN.
HSA_DEVINL float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// A float bound for a key bound: for every non-NaN score f and every bar,
// order_key(f) >= bar <=> f >= bar_float(bar).  A non-negative score's key is
// its bits with the top bit set, a negative score's key its bits inverted
// (both orders agree with the values'); every non-NaN key is at least the key
// of -inf (0x007fffff), so lower bars admit every score.
HSA_DEVINL float bar_float(uint32_t bar) {
  if (bar >= 0x80000000u) return __uint_as_float(bar ^ 0x80000000u);
  if (bar < 0x00800000u) return -INFINITY;
  return __uint_as_float(~bar);
}

HSA_DEVINL uint64_t composite(uint32_t key, uint32_t j) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(0xffffffffu - j);
}

// Warp-aggregated append: lanes with `take` get consecutive slots of *counter.
HSA_DEVINL uint32_t warp_append(uint32_t* counter, bool take, uint32_t active) {
  const uint32_t mask = __ballot_sync(active, take);
  if (!mask) return 0;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(mask));
  base = __shfl_sync(active, base, leader);
  return base + __popc(mask & ((1u << lane) - 1u));
}

// Finds digit d with (#above d) < need <= (#above d) + hist[d] among nb <=
// kPer * blockDim.x bins of a shared histogram, scanned from the top; returns d
// and *above.  All threads call; returns synchronised.
template <int kPer = 4>
HSA_DEVINL uint32_t find_digit(const uint32_t* hist, uint32_t nb, uint32_t need, uint32_t* above,
                               uint32_t* s_scan, uint32_t* s_out) {
  const uint32_t per = (nb + blockDim.x - 1) / blockDim.x;
  const uint32_t first = threadIdx.x * per;  // bins counted from the top
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t bb = first + i;
    c[i] = (static_cast<uint32_t>(i) < per && bb < nb) ? hist[nb - 1 - bb] : 0u;
    sum += c[i];
  }
  uint32_t total;
  uint32_t a = block_inclusive_sum<uint32_t>(sum, s_scan, &total) - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t bb = first + i;
    if (static_cast<uint32_t>(i) < per && bb < nb && a < need && a + c[i] >= need) {
      s_out[0] = nb - 1 - bb;
      s_out[1] = a;
    }
    a += c[i];
  }
  __syncthreads();
  *above = s_out[1];
  const uint32_t d = s_out[0];
  __syncthreads();
  return d;
}

// Bitonic sort (descending) of n (a power of two) composites in shared memory;
// every thread of the block calls it.
HSA_DEVINL void bitonic_sort_desc(uint64_t* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < n / 2; t += blockDim.x) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = a[lo], y = a[hi];
        if ((x < y) == desc) {
          a[lo] = y;
          a[hi] = x;
        }
      }
    }
  }
  __syncthreads();
}

// Rank of this thread's composite among the (at most blockDim.x = 32 * kRunWarps) composites
// a[0..n) when sorted descending; x receives the composite (0, below every
// real composite, for threads past n).  Each warp sorts its 32 composites by
// a bitonic network in registers (shuffles only); the sorted runs go to
// shared memory and each composite's rank is the number of larger
// composites in every run, found by a branchless binary search per run.
// Composites are unique, so the ranks of the n real ones are 0..n-1.
template <int kRunWarps>
HSA_DEVINL uint32_t rank_desc(const uint64_t* a, int n, uint64_t* s_run, uint64_t* x_out) {
  const int t = threadIdx.x, lane = t & 31;
  uint64_t x = t < n ? a[t] : 0ull;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t y = __shfl_xor_sync(0xffffffffu, x, stride);
      const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
      const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
      x = (lower == desc) ? hi : lo;
    }
  }
  s_run[t] = x;
  __syncthreads();
  uint32_t rank = 0;
#pragma unroll
  for (int s = 0; s < kRunWarps; ++s) {  // unrolled: the searches overlap their load latencies
    const uint64_t* r = s_run + 32 * s;
    uint32_t c = 0;
#pragma unroll
    for (int st = 16; st >= 1; st >>= 1) c += r[c + st - 1] > x ? st : 0;
    c += r[c] > x ? 1 : 0;
    rank += c;
  }
  *x_out = x;
  return rank;
}

// Bitonic sort (descending) of one composite per lane across the warp, in
// registers (shuffles only); returns this lane's element of the sorted run.
// The loops stay rolled: code that runs once per launch costs more in
// instruction fetches than in loop overhead.
HSA_DEVINL uint64_t warp_sort_desc(uint64_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t y = __shfl_xor_sync(0xffffffffu, x, stride);
      const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
      const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
      x = (lower == desc) ? hi : lo;
    }
  }
  return x;
}

// Sorts a[0..n) descending; a and b each hold P entries (P a power of two,
// 32 <= P <= 4 * blockDim.x, n <= P); entries n..P-1 of a are padded with 0,
// which sorts last; b is scratch.  The result ends in a.  Runs of 32 are
// sorted in registers (one warp each), then merged level by level: an entry
// of the left run of a pair goes after the right run's entries greater than
// it, an entry of the right run after the left run's entries greater than or
// equal to it, so every entry gets a distinct place (padding zeros included).
// Every thread of the block calls it.
template <int kMaxPer>
HSA_DEVINL void merge_sort_desc(uint64_t* a, uint64_t* b, int n, int P) {
  const int t = threadIdx.x, T = blockDim.x, lane = t & 31, warp = t >> 5, W = T >> 5;
  for (int i = n + t; i < P; i += T) a[i] = 0ull;
  __syncthreads();
#pragma unroll 1
  for (int r = warp; r < P / 32; r += W) a[32 * r + lane] = warp_sort_desc(a[32 * r + lane]);
  __syncthreads();
  uint64_t* src = a;
  uint64_t* dst = b;
#pragma unroll 1
  for (int lw = 5; (1 << lw) < P; ++lw) {  // runs of width 2^lw merged pairwise
    const int width = 1 << lw;
    uint64_t x[kMaxPer];
    int c[kMaxPer], other[kMaxPer];  // rank within the other run; that run's start
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) {
      const int i = t + q * T;
      x[q] = i < P ? src[i] : 0ull;
      c[q] = 0;
      other[q] = (((i >> lw) ^ 1) << lw) - 1;
    }
#pragma unroll 1
    for (int st = width >> 1; st >= 1; st >>= 1) {
#pragma unroll
      for (int q = 0; q < kMaxPer; ++q) {  // the entries' searches step together
        const int i = t + q * T;
        if (i >= P) continue;
        const uint64_t y = src[other[q] + c[q] + st];
        c[q] += (((i >> lw) & 1) ? y >= x[q] : y > x[q]) ? st : 0;
      }
    }
#pragma unroll
    for (int q = 0; q < kMaxPer; ++q) {
      const int i = t + q * T;
      if (i >= P) continue;
      const uint64_t y = src[other[q] + c[q] + 1];
      c[q] += (((i >> lw) & 1) ? y >= x[q] : y > x[q]) ? 1 : 0;
      dst[(((i >> lw) & ~1) << lw) + (i & (width - 1)) + c[q]] = x[q];
    }
    __syncthreads();
    uint64_t* tmp = src;
    src = dst;
    dst = tmp;
  }
  if (src != a) {
    for (int i = t; i < P; i += T) a[i] = src[i];
    __syncthreads();
  }
}

// Appends to out[*count ...] the `need` largest of the composites cand[0..n)
// that match prefix on mask and all agree above their low `low_bits` bits:
// radix select with 11-bit digits from the top.  Composites are unique, so
// the boundary is exact.
template <int kPer = 4>
HSA_DEVINL void select_rest(const uint64_t* cand, uint32_t n, uint32_t need, uint64_t* out,
                            uint32_t* count, uint32_t cap, uint32_t* s_hist, uint32_t* s_scan,
                            uint32_t* s_out, int low_bits, uint64_t prefix = 0, uint64_t mask = 0) {
  // (composites not matching prefix on mask are not candidates and are skipped)
  int rest = low_bits;
  while (need > 0 && rest > 0) {
    const int width = rest >= 11 ? 11 : rest;
    rest -= width;
    const int shift = rest;
    const uint32_t nb = 1u << width;
    for (uint32_t i = threadIdx.x; i < nb; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t x = cand[i];
      if ((x & mask) == prefix)
        atomicAdd(&s_hist[static_cast<uint32_t>(x >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    uint32_t above;
    const uint32_t d = find_digit<kPer>(s_hist, nb, need, &above, s_scan, s_out);
    const uint32_t in = s_hist[d];
    const bool take_bin = in == need - above;  // the whole bin fits
    for (uint32_t i0 = 0; i0 < n; i0 += blockDim.x) {
      const uint32_t i = i0 + threadIdx.x;
      bool take = false;
      uint64_t x = 0;
      if (i < n) {
        x = cand[i];
        if ((x & mask) == prefix) {
          const uint32_t dig = static_cast<uint32_t>(x >> shift) & (nb - 1);
          take = dig > d || (take_bin && dig == d);
        }
      }
      const uint32_t pos = warp_append(count, take, 0xffffffffu);
      if (take && pos < cap) out[pos] = x;
    }
    __syncthreads();
    if (take_bin) break;
    need -= above;
    prefix |= static_cast<uint64_t>(d) << shift;
    mask |= static_cast<uint64_t>(nb - 1) << shift;
  }
}

}  // namespace hsa
