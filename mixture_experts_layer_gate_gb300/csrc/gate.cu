// Stage 1: top-k expert gate, one warp per token.
//
// "Add deepseek_v3 fused gate" (sglang) describes a fused gate whose output
// order was unstable and whose host code synchronised; this kernel orders ids
// by key (descending, equal keys to the lower index) with a shuffle reduction
// that is the same total order on every run, and never touches the host.
// Softmax top-k (Mixtral / Qwen2 shapes) selects on the raw logits; the sigmoid
// gate (DeepSeek-V3 shape) selects on sigmoid(logit) + bias inside the
// topk_group best groups, each group scored by the sum of its two best keys.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kGateWarps = 8;
constexpr int kMaxTopK = 32;

struct Cand {
  float key;
  int idx;
  float val;  // softmax: logit; sigmoid: sigmoid score (the weight before scaling)
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

template <int EPL>  // experts per lane; E <= 32 * EPL
__global__ void __launch_bounds__(kGateWarps * 32) gate_topk_kernel(GateArgs a) {
  __shared__ float skeys[kGateWarps][32 * EPL];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kGateWarps + warp;
  pdl_wait();
  pdl_trigger();
  if (t >= a.T) return;  // whole warp leaves together

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
      if (l != l) l = -INFINITY;  // NaN ranks lowest
    } else {
      taken |= 1u << i;
    }
    val[i] = l;
    lmax = fmaxf(lmax, l);
  }
  float zsum = 0.f;
  if (!a.sigmoid) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      key[i] = val[i];
      if (!((taken >> i) & 1u)) zsum += expf(val[i] - lmax);
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
    // Group scores: sum of the two largest keys of each contiguous group.
    const int gs = a.E / a.n_group;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E) skeys[warp][e] = key[i];
    }
    __syncwarp();
    float gscore = -INFINITY;
    if (lane < a.n_group) {
      float m1 = -INFINITY, m2 = -INFINITY;
      const float* g = &skeys[warp][lane * gs];
      for (int j = 0; j < gs; ++j) {
        const float v = g[j];
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

  // k rounds of warp arg-max; the winner's owner lane retires it.
  int sel_idx[kMaxTopK];
  float sel_val[kMaxTopK];
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
    const float wv = a.sigmoid ? c.val : expf(c.val - lmax) / zsum;
    if (lane == 0) {
      sel_idx[j] = c.idx;
      sel_val[j] = wv;
    }
    total += wv;
  }
  if (lane == 0) {
    int32_t* ids = a.ids + static_cast<size_t>(t) * a.k;
    float* w = a.w + static_cast<size_t>(t) * a.k;
    const float inv = a.renormalize ? 1.0f / total : 1.0f;
#pragma unroll 1
    for (int j = 0; j < a.k; ++j) {
      ids[j] = sel_idx[j];
      w[j] = a.renormalize ? (sel_val[j] * inv) * a.scale : sel_val[j] * a.scale;
    }
  }
}

}  // namespace

cudaError_t launch_gate(const GateArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const dim3 grid((a.T + kGateWarps - 1) / kGateWarps);
  const dim3 block(kGateWarps * 32);
  if (a.E <= 64) return launch_pdl(gate_topk_kernel<2>, grid, block, 0, s, a);
  if (a.E <= 256) return launch_pdl(gate_topk_kernel<8>, grid, block, 0, s, a);
  return launch_pdl(gate_topk_kernel<32>, grid, block, 0, s, a);
}

}  // namespace moe
