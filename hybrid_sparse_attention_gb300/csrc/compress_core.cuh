// Softmax-gated block compression of one 8-channel chunk, shared by the
// standalone compressor and the decode-time block update.
//
// For rows i of a block: c[ch] = sum_i softmax_i(z[i,ch] + b[i,ch]) kv[i,ch].
// A thread reduces a contiguous range of the block's rows into an online-
// softmax partial (running max m, denominator l, numerator acc); partials of
// disjoint row ranges merge exactly, so a long block can be cut across lanes.
#pragma once

#include "common.cuh"

namespace hsa {

struct GatePartial {
  float m[8], l[8], acc[8];
};

HSA_DEVINL void partial_init(GatePartial& p) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    p.m[c] = -INFINITY;
    p.l[c] = 0.f;
    p.acc[c] = 0.f;
  }
}

// Rows [i0, i1) of one chunk; rows(i, &kv, &z) gives row i's two 16-byte
// chunks; bias(i, b0, b1) loads the 8 fp32 biases of row i.  kMasked:
// a logit may be -inf (a masked position, weight 0); without it every logit
// is finite (the guards cost about a fifth of the compressor's time).
// kGroup rows share one maximum and one rescale: larger groups take fewer
// exponentials, smaller ones fewer registers (1 = one rescale per row).
template <bool kMasked = false, int kGroup = 4, typename RowFn, typename BiasFn>
HSA_DEVINL void partial_rows_at(RowFn rows, int i0, int i1, BiasFn bias, GatePartial& p) {
  for (int r0 = i0; r0 < i1; r0 += kGroup) {
    const int g = min(kGroup, i1 - r0);
    uint4 kraw[kGroup], zraw[kGroup];
    float4 b0[kGroup], b1[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (j < g) {
        const uint4 *kp, *zp;
        rows(r0 + j, &kp, &zp);
        kraw[j] = ld_stream_u4(kp);
        zraw[j] = ld_stream_u4(zp);
        bias(r0 + j, &b0[j], &b1[j]);
      }
    }
    float x[kGroup][8], v[kGroup][8], gm[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) gm[c] = -INFINITY;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (j < g) {
        bf16x8_to_f32(zraw[j], x[j]);
        bf16x8_to_f32(kraw[j], v[j]);
        const float bb[8] = {b0[j].x, b0[j].y, b0[j].z, b0[j].w, b1[j].x, b1[j].y, b1[j].z, b1[j].w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          x[j][c] += bb[c];  // add
          gm[c] = fmaxf(gm[c], x[j][c]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float mn = fmaxf(p.m[c], gm[c]);
      // (masked: 0 while nothing finite has been seen, m = -inf, so that a
      // -inf logit weighs 0 and never makes -inf - -inf; otherwise
      // exp(-inf) = 0 on the first group)
      const float alpha = kMasked && p.m[c] == -INFINITY ? 0.f : __expf(p.m[c] - mn);
      p.l[c] *= alpha;
      p.acc[c] *= alpha;
      p.m[c] = mn;
    }
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if (j < g) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float e = kMasked && x[j][c] == -INFINITY ? 0.f : __expf(x[j][c] - p.m[c]);  // numerator
          p.l[c] += e;
          p.acc[c] = fmaf(e, v[j][c], p.acc[c]);    // dot
        }
      }
    }
  }
}

// The same over rows at kv[i * stride] / z[i * stride].
template <bool kMasked = false, int kGroup = 4, typename BiasFn>
HSA_DEVINL void partial_rows(const uint4* kv, const uint4* z, int64_t stride, int i0, int i1,
                             BiasFn bias, GatePartial& p) {
  partial_rows_at<kMasked, kGroup>(
      [&](int i, const uint4** kp, const uint4** zp) {
        *kp = kv + i * stride;
        *zp = z + i * stride;
      },
      i0, i1, bias, p);
}

// Merges the partials of `width` adjacent lanes (width a power of two <= 32;
// all 32 lanes of the warp must call it).
HSA_DEVINL void partial_merge_lanes(GatePartial& p, int width) {
  for (int o = 1; o < width; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float m2 = __shfl_xor_sync(0xffffffffu, p.m[c], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, p.l[c], o);
      const float a2 = __shfl_xor_sync(0xffffffffu, p.acc[c], o);
      const float mn = fmaxf(p.m[c], m2);
      const float s1 = p.m[c] == -INFINITY ? 0.f : __expf(p.m[c] - mn);
      const float s2 = m2 == -INFINITY ? 0.f : __expf(m2 - mn);
      p.l[c] = p.l[c] * s1 + l2 * s2;
      p.acc[c] = p.acc[c] * s1 + a2 * s2;
      p.m[c] = mn;
    }
  }
}

HSA_DEVINL void partial_result(const GatePartial& p, float out[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) out[c] = p.acc[c] / p.l[c];
}

}  // namespace hsa
