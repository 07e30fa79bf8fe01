// Copy of one token row to the k permuted rows its slots landed on, shared by
// the gather kernel and the small-batch routing kernel (so both write
// bit-identical x_perm rows): the row is read once and, for fp8, quantised
// once (e4m3 of x / a1, float32 division, round to nearest even, saturating).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// rows[j] = permuted row of slot t*k + j; run by `nthreads` threads, thread
// `tid`, over the 8-element column groups [c0, c1) of the row (0 .. H / 8 for
// the whole row).
template <bool FP8>
__device__ __forceinline__ void gather_token(const AlignArgs& a, int t, const int* rows, int c0, int c1, int tid,
                                             int nthreads) {
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                    static_cast<size_t>(t) * a.H);
  if (!FP8) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.x_perm);
    for (int c = c0 + tid; c < c1; c += nthreads) {
      const uint4 v = __ldg(src + c);
      for (int j = 0; j < a.k; ++j)
        reinterpret_cast<uint4*>(dst + static_cast<size_t>(rows[j]) * a.H)[c] = v;
    }
  } else {
    const float s = a.a1[0];
    uint8_t* dst = static_cast<uint8_t*>(a.x_perm);
    for (int c = c0 + tid; c < c1; c += nthreads) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t q[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h]), s),
                                            __fdiv_rn(bf16_hi(w[2 * h]), s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[2 * h + 1]), s),
                                            __fdiv_rn(bf16_hi(w[2 * h + 1]), s));
        q[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      const uint2 qv = make_uint2(q[0], q[1]);
      for (int j = 0; j < a.k; ++j)
        reinterpret_cast<uint2*>(dst + static_cast<size_t>(rows[j]) * a.H)[c] = qv;
    }
  }
}

}  // namespace moe
