// Plain CPU oracle for the decode-time hybrid sparse-attention path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
// this file; it exists so that tests/, the smoke check and the benchmark's CPU
// baseline can check the CUDA kernels against an independent, obviously
// correct implementation.  It shares no code, header, table or helper with the
// CUDA library.
//
// Every function is the plain definition of one stage, computed in double
// precision from exactly-converted inputs, with no blocking, fusion or
// reordering beyond what the definition states.  The sources are three web
// pages on DeepSeek-V4 serving:
//   [KD] kerneldigest.dev, "DeepSeek-V4: optimización de inferencia y RL para
//        modelos con atención híbrida y FP4"
//   [LH] lehuy.net, "DeepSeek-V4: SGLang và Miles mang đến hỗ trợ Day-0 cho suy
//        luận nhanh và Học tăng cường"
//   [WK] AI-KOL wiki, "与 SGLang 团队聊 DeepSeek V4:混合注意力的推理与 RL 训练适配"
// The pages name the stages but print no formula; the formulas below are the
// ones this library fixes for them (stated at each function).
//
// Parity pins (what each function is checked against, in tests/):
//   oracle_compress        hand-worked blocks, r=1 identity, constant-gate mean,
//                          shift invariance, convexity, linearity, long-double
//                          brute force
//   oracle_compress_overlap  hand-worked windows, -inf bias on the previous
//                          block reduces to oracle_compress, first block,
//                          constant-gate window mean, scipy softmax
//   oracle_indexer_scores  hand-worked example, one-hot reduction, w-linearity,
//                          non-negativity, long-double brute force
//   oracle_topk            hand-worked example, full sort of (value, index),
//                          nth_element cross-check, all-equal / reversed rows
//   oracle_decode_attn     hand-worked example, single row, equal logits,
//                          split + log-sum-exp recombination, dense equivalence
//   oracle_e4m3_to_double  every code against torch's float8_e4m3fn decoding,
//                          the format's named values
//   oracle_quantize_e4m3   encodings against torch's float8_e4m3fn rounding,
//                          saturation, amax -> 448, zero rows, error bound
//   oracle_indexer_scores_e4m3  hand-worked example, numpy float64 brute force
//                          on the dequantized operands, one-hot keys
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

// bfloat16 is the upper half of an IEEE binary32: widening is exact.
double bf16_to_double(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// binary32 -> bfloat16, round to nearest, ties to even (format definition:
// keep the top 16 bits, rounding on the 16 dropped bits).
uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);  // quiet NaN
  uint32_t dropped = u & 0xffffu;
  uint32_t kept = u >> 16;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1;
  return static_cast<uint16_t>(kept);
}

// FP8 E4M3 (the 8-bit "e4m3fn" interchange format): a sign bit, 4 exponent
// bits with bias 7 and 3 mantissa bits; exponent field 0 holds the subnormals
// m * 2^-9; the pattern s.1111.111 is NaN and there is no infinity, so the
// largest finite magnitude is 1.75 * 2^8 = 448.  The library's reading of the
// pages' FP8 KV storage ([LH] §Hỗ trợ Học tăng cường: FP8 rollout; [WK]
// 新架构: a 1M-token KV cache under 10 GB) for the indexer-key pool.
double e4m3_to_double(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double v = e == 0 ? std::ldexp(static_cast<double>(m), -9)
                          : std::ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -v : v;
}

// binary32 -> E4M3: the nearest finite code (the even code on a tie), finite
// magnitudes beyond 448 saturating to 448 and infinities too; NaN -> 0x7f.
// The non-negative finite codes 0x00..0x7e are increasing in value, so the
// nearest is one of the two neighbours a binary search finds.
uint8_t float_to_e4m3_sat(float f) {
  if (std::isnan(f)) return 0x7f;
  static const std::vector<double> values = [] {
    std::vector<double> v(0x7f);
    for (int c = 0; c < 0x7f; ++c) v[c] = e4m3_to_double(static_cast<uint8_t>(c));
    return v;
  }();
  const double a = std::fabs(static_cast<double>(f));
  const uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  const size_t i = std::lower_bound(values.begin(), values.end(), a) - values.begin();
  int c;
  if (i == 0) {
    c = 0;
  } else if (i == values.size()) {
    c = 0x7e;
  } else {
    const double dlo = a - values[i - 1], dhi = values[i] - a;
    if (dlo < dhi) c = static_cast<int>(i - 1);
    else if (dhi < dlo) c = static_cast<int>(i);
    else c = ((i - 1) & 1) == 0 ? static_cast<int>(i - 1) : static_cast<int>(i);
  }
  return static_cast<uint8_t>(c) | sign;
}

// One row of C binary32 values -> E4M3 codes and a binary32 scale, every step
// rounded to binary32 as the stored result is: amax = max |x|, scale = amax /
// 448, code[d] = e4m3(x[d] * (448 / amax)); a row of zeros gets scale 0 and
// zero codes.  Dequantized value: scale * e4m3_to_double(code).
void quantize_row_e4m3(const float* x, int64_t C, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int64_t d = 0; d < C; ++d) amax = std::max(amax, std::fabs(x[d]));
  if (amax == 0.0f) {
    for (int64_t d = 0; d < C; ++d) codes[d] = 0;
    *scale = 0.0f;
    return;
  }
  const float inv = 448.0f / amax;
  *scale = amax / 448.0f;
  for (int64_t d = 0; d < C; ++d) {
    const float y = x[d] * inv;
    codes[d] = float_to_e4m3_sat(y);
  }
}

// Runs fn(i) for i in [0, n) on up to `threads` std::threads (contiguous
// ranges).  threads <= 1 runs inline.
void parallel_for(int64_t n, int threads, const std::function<void(int64_t)>& fn) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  int64_t t = std::min<int64_t>(threads, n);
  std::vector<std::thread> pool;
  for (int64_t w = 0; w < t; ++w) {
    int64_t lo = n * w / t, hi = n * (w + 1) / t;
    pool.emplace_back([lo, hi, &fn] {
      for (int64_t i = lo; i < hi; ++i) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int oracle_hardware_threads() {
  unsigned n = std::thread::hardware_concurrency();
  return n == 0 ? 1 : static_cast<int>(n);
}

void oracle_float_to_bf16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne(x[i]);
}

void oracle_bf16_to_double(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_double(x[i]);
}

// Flash Compressor ([KD] §Arquitectura del Sistema: the 5-stage compression
// chain fused into one on-chip pass; [WK] 推理侧优化, "Kernel fusion": read ->
// add -> softmax -> dot -> write).  The library fixes the chain as, for every
// complete block n of r consecutive tokens and every channel ch,
//     c[n, ch] = sum_i softmax_i(z[n*r+i, ch] + b[i, ch]) * kv[n*r+i, ch],
// the softmax running over the r positions of the block, per channel; b is a
// per-(position-in-block, channel) bias.  Block n covers tokens [n*r, n*r+r);
// a trailing partial block is not compressed.
//   kv, z : bf16 [S, T, C]   b : fp32 [r, C]   out : fp64 [S, T/r, C]
int oracle_compress(const uint16_t* kv, const uint16_t* z, const float* b, int64_t S,
                    int64_t T, int64_t C, int64_t r, double* out, int threads) {
  if (r <= 0 || S < 0 || T < 0 || C <= 0) return 1;
  const int64_t nblk = T / r;
  parallel_for(S * nblk, threads, [&](int64_t sn) {
    const int64_t s = sn / nblk, n = sn % nblk;
    for (int64_t ch = 0; ch < C; ++ch) {
      // add: logits of the block's r positions
      std::vector<double> logit(r), val(r);
      for (int64_t i = 0; i < r; ++i) {
        const int64_t t = n * r + i;
        logit[i] = bf16_to_double(z[(s * T + t) * C + ch]) + static_cast<double>(b[i * C + ch]);
        val[i] = bf16_to_double(kv[(s * T + t) * C + ch]);
      }
      // softmax (max-subtracted), then dot with kv
      double m = logit[0];
      for (int64_t i = 1; i < r; ++i) m = std::max(m, logit[i]);
      double num = 0.0, den = 0.0;
      for (int64_t i = 0; i < r; ++i) {
        const double e = std::exp(logit[i] - m);
        num += e * val[i];
        den += e;
      }
      out[(s * nblk + n) * C + ch] = num / den;
    }
  });
  return 0;
}

// C4 overlap transform ([WK] §RL 训练侧 ①: C4's "overlap transform", under
// which neighbouring compressed entries share tokens, so a context-parallel
// split cannot compress its first block without its neighbour's tokens).  The
// pages name it without defining it; the library's reading: entry n is the
// gated softmax average over a window of 2r tokens with stride r — block n's
// own r tokens and the r tokens of block n-1 before them —
//     c[n, ch] = sum_{i in window} softmax_i(z[n*r-r+i, ch] + b[i, ch]) * kv[n*r-r+i, ch],
// window i in [0, 2r), positions before the sequence's start absent (entry 0
// uses i in [r, 2r) only); b is per (position in the window, channel).
//   kv, z : bf16 [S, T, C]   b : fp32 [2r, C]   out : fp64 [S, T/r, C]
int oracle_compress_overlap(const uint16_t* kv, const uint16_t* z, const float* b, int64_t S,
                            int64_t T, int64_t C, int64_t r, double* out, int threads) {
  if (r <= 0 || S < 0 || T < 0 || C <= 0) return 1;
  const int64_t nblk = T / r;
  parallel_for(S * nblk, threads, [&](int64_t sn) {
    const int64_t s = sn / nblk, n = sn % nblk;
    const int64_t i0 = n == 0 ? r : 0;  // the window's first present position
    for (int64_t ch = 0; ch < C; ++ch) {
      std::vector<double> logit, val;
      for (int64_t i = i0; i < 2 * r; ++i) {
        const int64_t t = n * r - r + i;
        logit.push_back(bf16_to_double(z[(s * T + t) * C + ch]) + static_cast<double>(b[i * C + ch]));
        val.push_back(bf16_to_double(kv[(s * T + t) * C + ch]));
      }
      double m = logit[0];
      for (double l : logit) m = std::max(m, l);
      double num = 0.0, den = 0.0;
      for (size_t i = 0; i < logit.size(); ++i) {
        const double e = std::exp(logit[i] - m);
        num += e * val[i];
        den += e;
      }
      out[(s * nblk + n) * C + ch] = num / den;
    }
  });
  return 0;
}

// Indexer scores ([KD] §Arquitectura del Sistema: top-k selection "in the
// indexer"; [KD] flow step 6; [WK] RL ③, the attention indexer acts like an MoE
// router).  The library fixes the score of compressed entry j of sequence b as
//     s[b, j] = sum_h w[b, h] * max(0, sum_d q[b, h, d] * k[off_b + j, d]).
//   iq : bf16 [B, Hi, Di]   w : fp32 [B, Hi]   keys : bf16 [sum N_b, Di]
//   offsets : int64 [B+1], N_b = offsets[b+1] - offsets[b]
//   scores : fp64 [sum N_b], same offsets as keys
int oracle_indexer_scores(const uint16_t* iq, const float* w, const uint16_t* keys,
                          const int64_t* offsets, int64_t B, int64_t Hi, int64_t Di,
                          double* scores, int threads) {
  if (B < 0 || Hi <= 0 || Di <= 0) return 1;
  for (int64_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return 1;
  // every entry is independent: the entries of all sequences are shared out
  // among the threads in contiguous ranges; entry j belongs to the sequence b
  // whose range [offsets[b], offsets[b+1]) holds it
  const int64_t first = offsets[0], total = offsets[B] - offsets[0];
  parallel_for(total, threads, [&](int64_t e) {
    const int64_t j = first + e;
    const int64_t b = (std::upper_bound(offsets, offsets + B + 1, j) - offsets) - 1;
    double s = 0.0;
    for (int64_t h = 0; h < Hi; ++h) {
      double dot = 0.0;
      for (int64_t d = 0; d < Di; ++d)
        dot += bf16_to_double(iq[(b * Hi + h) * Di + d]) * bf16_to_double(keys[j * Di + d]);
      s += static_cast<double>(w[b * Hi + h]) * std::max(0.0, dot);
    }
    scores[j] = s;
  });
  return 0;
}

// Lightning TopK ([KD] §Arquitectura del Sistema: radix-select reduction in
// place of a global sort; [WK] 推理侧优化, "Lightning topk").  The result is
// defined by a sort, whatever algorithm reaches it: per row, the first
// min(k, N) entries of the row's (value, index) pairs ordered by value
// descending, lower row-local index first among equal values; -0.0 equals
// +0.0 (IEEE comparison); +-inf are ordinary extremes.  Unused slots hold -1
// (indices) and -inf (values).  A NaN anywhere is a precondition violation:
// the function returns 2 and writes nothing for that row.
//   scores : fp32 [sum N_b]   offsets : int64 [B+1]
//   idx : int32 [B, k] row-local   vals : fp32 [B, k] or null
int oracle_topk(const float* scores, const int64_t* offsets, int64_t B, int64_t k,
                int32_t* idx, float* vals, int threads) {
  if (B < 0 || k <= 0) return 1;
  for (int64_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return 1;
  std::vector<int> status(B, 0);
  parallel_for(B, threads, [&](int64_t b) {
    const int64_t n = offsets[b + 1] - offsets[b];
    const float* row = scores + offsets[b];
    std::vector<std::pair<float, int64_t>> pairs(n);
    for (int64_t j = 0; j < n; ++j) {
      if (std::isnan(row[j])) {
        status[b] = 2;
        return;
      }
      pairs[j] = {row[j], j};
    }
    std::sort(pairs.begin(), pairs.end(), [](const auto& a, const auto& c) {
      if (a.first != c.first) return a.first > c.first;
      return a.second < c.second;
    });
    for (int64_t i = 0; i < k; ++i) {
      const bool live = i < n;
      idx[b * k + i] = live ? static_cast<int32_t>(pairs[i].second) : -1;
      if (vals) vals[b * k + i] = live ? pairs[i].first : -std::numeric_limits<float>::infinity();
    }
  });
  for (int64_t b = 0; b < B; ++b)
    if (status[b]) return status[b];
  return 0;
}

// Fused hybrid attention ([KD] flow step 5 and the technology table: SWA and
// the extra C4/C128 attention in one kernel; [LH] §Tích hợp Kernel: FlashMLA
// path combining SWA with the extra attention in one call; [WK] 核心观点: SWA
// sees the most recent tokens, C4 attends its top-k, C128 attends everything).
// For query token b and head h, the attended set T_b is
//   - the SWA rows of positions p in [max(0, L_b - W), L_b), stored at ring
//     slot p mod W, and
//   - the compressed rows extra[off_b + j] for every j listed in idx[b, 0..k)
//     with j >= 0 (one term per listed entry), or, when idx is null, every j
//     in [0, N_b).
// Keys are full Dqk-wide rows and values are their first Dv channels (one
// shared latent KV head).  One softmax runs over the whole set:
//     l_t = scale * q[b,h,:] . K_t,  m = max_t l_t,
//     o[b,h,:] = sum_t exp(l_t - m) V_t / sum_t exp(l_t - m),
//     lse[b,h] = m + log sum_t exp(l_t - m).
// An empty set gives o = 0 and lse = -inf.  An index j >= N_b returns 3.
//   q : bf16 [B, Hq, Dqk]   swa : bf16 [B, W, Dqk]   seq_len : int32 [B]
//   extra : bf16 [sum N_b, Dqk]   extra_offsets : int64 [B+1]
//   extra_idx : int32 [B, k] or null   out : fp64 [B, Hq, Dv]   lse : fp64 [B, Hq]
int oracle_decode_attn(const uint16_t* q, const uint16_t* swa, const int32_t* seq_len,
                       int64_t W, const uint16_t* extra, const int64_t* extra_offsets,
                       const int32_t* extra_idx, int64_t k, int64_t B, int64_t Hq,
                       int64_t Dqk, int64_t Dv, double scale, double* out, double* lse,
                       int threads) {
  if (B < 0 || Hq <= 0 || Dqk <= 0 || Dv <= 0 || Dv > Dqk || W < 0) return 1;
  for (int64_t b = 0; b < B; ++b) {
    if (extra_offsets && extra_offsets[b + 1] < extra_offsets[b]) return 1;
    if (seq_len[b] < 0) return 1;
    if (extra_idx) {
      const int64_t n = extra_offsets ? extra_offsets[b + 1] - extra_offsets[b] : 0;
      for (int64_t i = 0; i < k; ++i)
        if (extra_idx[b * k + i] >= n) return 3;
    }
  }
  // the attended rows of each sequence (pointers into the pools)
  std::vector<std::vector<const uint16_t*>> rows(B);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = seq_len[b];
    for (int64_t p = std::max<int64_t>(0, L - W); p < L; ++p)
      rows[b].push_back(swa + (b * W + p % W) * Dqk);
    if (extra_offsets) {
      const int64_t off = extra_offsets[b], n = extra_offsets[b + 1] - off;
      if (extra_idx) {
        for (int64_t i = 0; i < k; ++i) {
          const int32_t j = extra_idx[b * k + i];
          if (j >= 0) rows[b].push_back(extra + (off + j) * Dqk);
        }
      } else {
        for (int64_t j = 0; j < n; ++j) rows[b].push_back(extra + (off + j) * Dqk);
      }
    }
  }
  // every (sequence, head) pair is independent
  parallel_for(B * Hq, threads, [&](int64_t bh) {
    const int64_t b = bh / Hq, h = bh % Hq;
    const std::vector<const uint16_t*>& rb = rows[b];
    const int64_t nt = static_cast<int64_t>(rb.size());
    double* o = out + (b * Hq + h) * Dv;
    if (nt == 0) {
      for (int64_t d = 0; d < Dv; ++d) o[d] = 0.0;
      if (lse) lse[b * Hq + h] = -std::numeric_limits<double>::infinity();
      return;
    }
    const uint16_t* qh = q + (b * Hq + h) * Dqk;
    std::vector<double> logit(nt);
    for (int64_t t = 0; t < nt; ++t) {
      double dot = 0.0;
      for (int64_t d = 0; d < Dqk; ++d) dot += bf16_to_double(qh[d]) * bf16_to_double(rb[t][d]);
      logit[t] = scale * dot;
    }
    double m = logit[0];
    for (int64_t t = 1; t < nt; ++t) m = std::max(m, logit[t]);
    double den = 0.0;
    std::vector<double> num(Dv, 0.0);
    for (int64_t t = 0; t < nt; ++t) {
      const double e = std::exp(logit[t] - m);
      den += e;
      for (int64_t d = 0; d < Dv; ++d) num[d] += e * bf16_to_double(rb[t][d]);
    }
    for (int64_t d = 0; d < Dv; ++d) o[d] = num[d] / den;
    if (lse) lse[b * Hq + h] = m + std::log(den);
  });
  return 0;
}

void oracle_e4m3_to_double(const uint8_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(x[i]);
}

void oracle_float_to_e4m3(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_to_e4m3_sat(x[i]);
}

// Per-row E4M3 quantization (quantize_row_e4m3 on each of `rows` rows of C).
//   x : fp32 [rows, C]   codes : u8 [rows, C]   scales : fp32 [rows]
int oracle_quantize_e4m3(const float* x, int64_t rows, int64_t C, uint8_t* codes, float* scales,
                         int threads) {
  if (rows < 0 || C <= 0) return 1;
  parallel_for(rows, threads, [&](int64_t i) {
    quantize_row_e4m3(x + i * C, C, codes + i * C, scales + i);
  });
  return 0;
}

// Indexer scores over an E4M3 key pool: the score of oracle_indexer_scores on
// the dequantized operands,
//     s[b, j] = sum_h w[b, h] * max(0, sum_d qhat[b, h, d] * khat[j, d]),
//     khat[j, d] = kscale[j] * e4m3(keys[j, d]),
//     qhat[b, h, d] = qscale[b, h] * e4m3(qcode[b, h, d]),
// where each query row iq[b, h, :] (bf16, widened exactly) is quantized as
// oracle_quantize_e4m3 quantizes a row.
//   iq : bf16 [B, Hi, Di]   w : fp32 [B, Hi]   keys : u8 [sum N_b, Di]
//   kscale : fp32 [sum N_b]   offsets : int64 [B+1]   scores : fp64 [sum N_b]
int oracle_indexer_scores_e4m3(const uint16_t* iq, const float* w, const uint8_t* keys,
                               const float* kscale, const int64_t* offsets, int64_t B,
                               int64_t Hi, int64_t Di, double* scores, int threads) {
  if (B < 0 || Hi <= 0 || Di <= 0) return 1;
  for (int64_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return 1;
  // the quantized, then dequantized, query rows
  std::vector<double> qhat(static_cast<size_t>(B * Hi * Di));
  {
    std::vector<float> row(Di);
    std::vector<uint8_t> code(Di);
    for (int64_t bh = 0; bh < B * Hi; ++bh) {
      for (int64_t d = 0; d < Di; ++d) row[d] = static_cast<float>(bf16_to_double(iq[bh * Di + d]));
      float sq;
      quantize_row_e4m3(row.data(), Di, code.data(), &sq);
      for (int64_t d = 0; d < Di; ++d)
        qhat[bh * Di + d] = static_cast<double>(sq) * e4m3_to_double(code[d]);
    }
  }
  const int64_t first = offsets[0], total = offsets[B] - offsets[0];
  parallel_for(total, threads, [&](int64_t e) {
    const int64_t j = first + e;
    const int64_t b = (std::upper_bound(offsets, offsets + B + 1, j) - offsets) - 1;
    double s = 0.0;
    for (int64_t h = 0; h < Hi; ++h) {
      double dot = 0.0;
      for (int64_t d = 0; d < Di; ++d)
        dot += qhat[(b * Hi + h) * Di + d] *
               (static_cast<double>(kscale[j]) * e4m3_to_double(keys[j * Di + d]));
      s += static_cast<double>(w[b * Hi + h]) * std::max(0.0, dot);
    }
    scores[j] = s;
  });
  return 0;
}

}  // extern "C"
