// Top-k expert gate of one token, run by one warp: shared by the gate kernel
// and the single-CTA small-batch routing kernel, so both select bit-identically.
//
// "Add deepseek_v3 fused gate" (sglang) describes a fused gate whose output
// order was unstable and whose host code synchronised; this code orders ids by
// key (descending, equal keys to the lower index) with a shuffle reduction that
// is the same total order on every run, and never touches the host.  Softmax
// top-k (Mixtral / Qwen2 shapes) selects on the raw logits; the sigmoid gate
// (DeepSeek-V3 shape) selects on sigmoid(logit) + bias inside the topk_group
// best groups, each group scored by the sum of its two best keys.
#pragma once

#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace gate_detail {

constexpr int kMaxTopK = 32;

struct Cand {
  float key;
  int idx;
  float val;  // softmax: exp(logit - max); sigmoid: sigmoid score (the weight before scaling)
};

__device__ __forceinline__ bool better(float k1, int i1, float k2, int i2) {
  return (k1 > k2) || (k1 == k2 && i1 < i2);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, c.key, off);
    const int oi = __shfl_xor_sync(0xffffffffu, c.idx, off);
    const float ov = __shfl_xor_sync(0xffffffffu, c.val, off);
    if (better(ok, oi, c.key, c.idx)) {
      c.key = ok;
      c.idx = oi;
      c.val = ov;
    }
  }
  return c;
}

// Selects the top-k experts of token t and writes ids[t, :] and w[t, :]; run by
// one full warp (lane = its lane).  `skeys` is 32 * EPL floats of shared memory
// private to the warp (group scores of the sigmoid gate).
template <int EPL>  // experts per lane; E <= 32 * EPL
__device__ __forceinline__ void gate_token(const GateArgs& a, int t, int lane, float* skeys) {
  const float* lrow = a.logits + static_cast<size_t>(t) * a.E;
  float key[EPL], val[EPL];
  uint32_t taken = 0;  // bit i: expert lane + 32 i is out of the running

  // Expert e = lane + 32 i (strided so the loads coalesce).
  float lmax = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float l = -INFINITY;
    if (e < a.E) {
      l = lrow[e];
      if (l != l) l = -INFINITY;  // a NaN logit is read as -inf
    } else {
      taken |= 1u << i;
    }
    val[i] = l;
    lmax = fmaxf(lmax, l);
  }
  float zsum = 0.f;
  if (!a.sigmoid) {
    // rank on the logits; carry exp(logit - max), the softmax numerator, as the value
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      key[i] = val[i];
      const float ev = ((taken >> i) & 1u) ? 0.f : expf(val[i] - lmax);
      zsum += ev;
      val[i] = ev;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
  } else {
    const bool raw_keys = (a.n_group == 0) && (a.bias == nullptr);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      const float l = val[i];
      const float s = 1.0f / (1.0f + expf(-l));
      float kk = raw_keys ? l : s;
      if (a.bias != nullptr && e < a.E) kk = s + a.bias[e];
      key[i] = kk;
      val[i] = s;
    }
  }

  if (a.n_group > 0) {
    // Group scores: sum of the two largest keys of each contiguous group.  The
    // keys are stored transposed (member j of group g at j * n_group + g), so
    // the lanes that score the groups read consecutive words, free of bank
    // conflicts, in the same member order.
    const int gs = a.E / a.n_group;
    const bool pow2 = (gs & (gs - 1)) == 0;
    const int gshift = __ffs(gs) - 1;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E) {
        const int g = pow2 ? (e >> gshift) : e / gs;
        skeys[(e - g * gs) * a.n_group + g] = key[i];
      }
    }
    __syncwarp();
    float gscore = -INFINITY;
    if (lane < a.n_group) {
      float m1 = -INFINITY, m2 = -INFINITY;
      const float* g = &skeys[lane];
      for (int j = 0; j < gs; ++j) {
        const float v = g[j * a.n_group];
        if (v > m1) {
          m2 = m1;
          m1 = v;
        } else if (v > m2) {
          m2 = v;
        }
      }
      gscore = (gs >= 2) ? (m1 + m2) : m1;
    }
    uint32_t gmask = 0;
    for (int j = 0; j < a.topk_group; ++j) {
      Cand c;
      const bool live = lane < a.n_group && !((gmask >> lane) & 1u);
      c.key = live ? gscore : -INFINITY;
      c.idx = live ? lane : INT_MAX;
      c.val = 0.f;
      c = warp_best(c);
      gmask |= 1u << c.idx;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((gmask >> (e / gs)) & 1u)) taken |= 1u << i;
    }
  }

  // k rounds of warp arg-max; the winner's owner lane retires it and lane j
  // keeps the j-th selection.
  const float inv_z = a.sigmoid ? 1.0f : 1.0f / zsum;
  int my_idx = 0;
  float my_val = 0.f;
  float total = 0.f;
#pragma unroll 1
  for (int j = 0; j < a.k; ++j) {
    Cand c{-INFINITY, INT_MAX, 0.f};
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!((taken >> i) & 1u)) {
        const int e = lane + 32 * i;
        if (better(key[i], e, c.key, c.idx)) {
          c.key = key[i];
          c.idx = e;
          c.val = val[i];
        }
      }
    }
    c = warp_best(c);
    if ((c.idx & 31) == lane) taken |= 1u << (c.idx >> 5);
    const float wv = c.val * inv_z;  // softmax: exp / sum; sigmoid: the score
    if (lane == j) {
      my_idx = c.idx;
      my_val = wv;
    }
    total += wv;
  }
  if (lane < a.k) {
    // selected scores that are all zero (every selected logit NaN) give zero
    // weights instead of 0 / 0
    const float inv = a.renormalize ? (total > 0.f ? 1.0f / total : 0.f) : 1.0f;
    const size_t o = static_cast<size_t>(t) * a.k + lane;
    a.ids[o] = my_idx;
    a.w[o] = a.renormalize ? (my_val * inv) * a.scale : my_val * a.scale;
  }
}

}  // namespace gate_detail
}  // namespace moe
