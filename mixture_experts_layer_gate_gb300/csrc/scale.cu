// Dynamic per-tensor fp8 activation scales (the W8A8 path with scales computed
// per batch instead of given): scale = max |v| / 448 over a whole bf16 tensor,
// so its largest magnitude maps to the e4m3 maximum, then v -> e4m3(v / scale).
//
// "[kernel] introduce fused_moe_triton_splitk to sglang" and the FBGEMM
// grouped-GEMM blog run fp8 W8A8 with per-tensor activation scales; the scale
// of the SwiGLU output is taken over the output as stored in bf16, and the
// quantisation is a separate pass, as the pages' fused-MoE code keeps that
// output in the model dtype between the two GEMMs.
//
// absmax_scale_kernel (token rows): each CTA takes the maximum bf16 magnitude
// of its share (the magnitude bits of a non-NaN bf16 order like its value),
// folds it into one word with atomicMax (exact, so the result is the same on
// every run), and the last CTA to finish (ticket counter) turns the word into
// the scale and clears word and counter for the next call.  The SwiGLU output
// gets its maximum from the epilogue that stores it, so its pass only
// quantises.  Inputs are assumed finite.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kScaleThreads = 256;
constexpr int kScaleMaxCtas = 1216;  // 8 per SM of a 152-SM part; grid-stride beyond

__global__ void __launch_bounds__(kScaleThreads)
    absmax_scale_kernel(const uint4* __restrict__ x, int64_t nvec, DynScales* d, int which) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t wmax[kScaleThreads / 32];
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kScaleThreads + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kScaleThreads) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
#pragma unroll
    for (int i = 0; i < kScaleThreads / 32; ++i) b = max(b, wmax[i]);
    atomicMax(&d->amax[which], b);
    __threadfence();
    if (atomicAdd(&d->ticket[which], 1u) == gridDim.x - 1) {
      __threadfence();
      const float a = __uint_as_float(atomicExch(&d->amax[which], 0u) << 16);
      atomicExch(&d->ticket[which], 0u);
      d->scale[which] = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
    }
  }
}

// The SwiGLU output's pass: the gate_up GEMM (or its split-K finish) folded the
// magnitude bits of every bf16 value it stored into amax[which]; each CTA
// derives the same scale from that word, quantises its share, and the last CTA
// publishes the scale for the down GEMM and clears the word and the counter.
__global__ void __launch_bounds__(kScaleThreads)
    quantize_e4m3_dynamic_kernel(const uint4* __restrict__ x, int64_t nvec, DynScales* d, int which,
                                 uint2* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const float a = __uint_as_float(*reinterpret_cast<volatile uint32_t*>(&d->amax[which]) << 16);
  const float s = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
  // times the reciprocal, as the static requantisation in the GEMM epilogue does
  // (an IEEE division per element made this pass instruction-bound)
  const float rs = __fdiv_rn(1.0f, s);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kScaleThreads + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kScaleThreads) {
    const uint4 v = __ldg(x + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t lo = f32x2_to_e4m3x2(bf16_lo(w[2 * h]) * rs, bf16_hi(w[2 * h]) * rs);
      const uint16_t hi = f32x2_to_e4m3x2(bf16_lo(w[2 * h + 1]) * rs, bf16_hi(w[2 * h + 1]) * rs);
      q[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    out[i] = make_uint2(q[0], q[1]);
  }
  __syncthreads();  // every thread of the CTA has read amax before the CTA counts itself
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&d->ticket[which], 1u) == gridDim.x - 1) {
      d->scale[which] = s;
      atomicExch(&d->amax[which], 0u);
      atomicExch(&d->ticket[which], 0u);
    }
  }
}

int scale_grid(int64_t nvec) {
  const int64_t g = (nvec + kScaleThreads - 1) / kScaleThreads;
  return static_cast<int>(g < 1 ? 1 : (g > kScaleMaxCtas ? kScaleMaxCtas : g));
}

}  // namespace

cudaError_t launch_absmax_scale(const void* x, int64_t n, DynScales* d, int which, cudaStream_t s) {
  const int64_t nvec = n / 8;
  return launch_pdl(absmax_scale_kernel, dim3(scale_grid(nvec)), dim3(kScaleThreads), 0, s,
                    static_cast<const uint4*>(x), nvec, d, which);
}

cudaError_t launch_quantize_e4m3_dynamic(const void* x, int64_t n, DynScales* d, int which, void* out,
                                         cudaStream_t s) {
  const int64_t nvec = n / 8;
  return launch_pdl(quantize_e4m3_dynamic_kernel, dim3(scale_grid(nvec)), dim3(kScaleThreads), 0, s,
                    static_cast<const uint4*>(x), nvec, d, which, static_cast<uint2*>(out));
}

}  // namespace moe
