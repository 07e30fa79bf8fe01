// Stage 4: unpermute and top-k weighted reduction, plus the split-K finishing
// passes of the grouped GEMMs.
//
// "Add deepseek_v3 fused gate" (sglang) names TensorRT-LLM's
// unpermute_and_reduce; "[kernel] introduce fused_moe_triton_splitk to sglang"
// reports that split-K partials added with atomics gave random values.  Every
// sum here runs in a fixed order in fp32 (j = 0..k-1; slice p = 0..P-1), so the
// result is the same on every run.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kReduceMaxK = 32;  // top_k limit of the problem checks

// Loads token t's k (row, weight) pairs into shared memory once, so the row
// loads of different j depend on no global load and can be in flight together
// (a small batch is otherwise a chain of k dependent round trips).
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ inv, const float* __restrict__ w,
                                           int t, int k, int* s_inv, float* s_w) {
  if (threadIdx.x < k) {
    s_inv[threadIdx.x] = inv[static_cast<size_t>(t) * k + threadIdx.x];
    s_w[threadIdx.x] = w[static_cast<size_t>(t) * k + threadIdx.x];
  }
  __syncthreads();
}

// grid (ceil(H / 2048), T); each thread owns 8 consecutive elements of a row.
__global__ void __launch_bounds__(256)
    unpermute_reduce_kernel(const __nv_bfloat16* __restrict__ y, const int32_t* __restrict__ inv,
                            const float* __restrict__ w, int H, int k, __nv_bfloat16* out) {
  __shared__ int s_inv[kReduceMaxK];
  __shared__ float s_w[kReduceMaxK];
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  load_slots(inv, w, t, k, s_inv, s_w);
  if (c * 8 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int j = 0; j < k; ++j) {
    const int r = s_inv[j];
    const float wj = s_w[j];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + static_cast<size_t>(r) * H) + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wj, bf16_lo(u[i]), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj, bf16_hi(u[i]), acc[2 * i + 1]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
}

// out[t, h] = sum_j w[t, j] * bf16(sum_p part[p][inv[t, j]][h]): the down
// GEMM's split-K finish folded into the reduce.  The slice sum, its bf16
// rounding and the weighted sum run in the same order and precision as
// down_finish followed by unpermute_reduce, so the result is bit-identical to
// that pair (and the permuted expert outputs never go through memory).
__global__ void __launch_bounds__(256)
    unpermute_reduce_splitk_kernel(const float* __restrict__ part, int P, int64_t pstride,
                                   const int32_t* __restrict__ inv, const float* __restrict__ w, int H,
                                   int k, __nv_bfloat16* out) {
  __shared__ int s_inv[kReduceMaxK];
  __shared__ float s_w[kReduceMaxK];
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  load_slots(inv, w, t, k, s_inv, s_w);
  if (c * 8 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int j = 0; j < k; ++j) {
    const int r = s_inv[j];
    const float wj = s_w[j];
    const float* row = part + static_cast<size_t>(r) * H;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
#pragma unroll 4
    for (int q = 0; q < P; ++q) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(row + q * pstride) + 2 * c);
      const float4 b = __ldg(reinterpret_cast<const float4*>(row + q * pstride) + 2 * c + 1);
      s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
      s1.x += b.x; s1.y += b.y; s1.z += b.z; s1.w += b.w;
    }
    const uint32_t u[4] = {pack_bf16x2(s0.x, s0.y), pack_bf16x2(s0.z, s0.w), pack_bf16x2(s1.x, s1.y),
                           pack_bf16x2(s1.z, s1.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wj, bf16_lo(u[i]), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj, bf16_hi(u[i]), acc[2 * i + 1]);
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H)[c] = o;
}

// The same result for small batches, with the work spread over the slots too:
// block (64, kSplitSlotThreads), a CTA owns 256 columns of one token.  First
// every (slot j, 4 columns) pair sums its P slices (threads along y take the
// slots, so a decode step's few tokens still spread over many warps with many
// loads in flight), rounds to bf16 and parks the result in shared memory; then
// the 64 threads of row y = 0 form the weighted sum in j order.  (At large
// batches the idle slot rows cost more than the extra parallelism gains.)
constexpr int kSplitSlotThreads = 8;

__global__ void __launch_bounds__(64 * kSplitSlotThreads)
    unpermute_reduce_splitk_slots_kernel(const float* __restrict__ part, int P, int64_t pstride,
                                   const int32_t* __restrict__ inv, const float* __restrict__ w, int H,
                                   int k, __nv_bfloat16* out) {
  __shared__ int s_inv[kReduceMaxK];
  __shared__ float s_w[kReduceMaxK];
  __shared__ uint2 s_y[kReduceMaxK][64];  // bf16 slice sums: slot j, 4 columns per entry
  const int t = blockIdx.y;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * 64 + tx;
  const int c = blockIdx.x * 64 + tx;  // float4 column index
  pdl_wait();
  pdl_trigger();
  if (tid < k) {
    s_inv[tid] = inv[static_cast<size_t>(t) * k + tid];
    s_w[tid] = w[static_cast<size_t>(t) * k + tid];
  }
  __syncthreads();
  const bool live = c * 4 < H;
  if (live) {
    for (int j = ty; j < k; j += kSplitSlotThreads) {
      const float* row = part + static_cast<size_t>(s_inv[j]) * H;
      float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int q = 0; q < P; ++q) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(row + q * pstride) + c);
        s0.x += a.x; s0.y += a.y; s0.z += a.z; s0.w += a.w;
      }
      s_y[j][tx] = make_uint2(pack_bf16x2(s0.x, s0.y), pack_bf16x2(s0.z, s0.w));
    }
  }
  __syncthreads();
  if (ty != 0 || !live) return;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    const float wj = s_w[j];
    const uint2 u = s_y[j][tx];
    acc[0] = fmaf(wj, bf16_lo(u.x), acc[0]);
    acc[1] = fmaf(wj, bf16_hi(u.x), acc[1]);
    acc[2] = fmaf(wj, bf16_lo(u.y), acc[2]);
    acc[3] = fmaf(wj, bf16_hi(u.y), acc[3]);
  }
  reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H)[c] =
      make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
}

// act[r, i] = silu(sum_p part[p][r][i]) * sum_p part[p][r][I + i]; 4 columns per thread.
// amax (bf16 output only, may be null): running max of the stored |act| bits.
template <bool FP8>
__global__ void __launch_bounds__(256)
    swiglu_finish_kernel(const float* __restrict__ part, int P, int64_t pstride, int I,
                         const float* __restrict__ a2, void* act, uint32_t* amax) {
  const int r = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  uint32_t mx = 0;
  if (c * 4 < I) {
    const float* row = part + static_cast<size_t>(r) * (2 * static_cast<size_t>(I));
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
#pragma unroll 4
    for (int p = 0; p < P; ++p) {
      const float4 gg = __ldg(reinterpret_cast<const float4*>(row + p * pstride) + c);
      const float4 uu = __ldg(reinterpret_cast<const float4*>(row + p * pstride + I) + c);
      g.x += gg.x; g.y += gg.y; g.z += gg.z; g.w += gg.w;
      u.x += uu.x; u.y += uu.y; u.z += uu.z; u.w += uu.w;
    }
    const float a0 = silu_f32(g.x) * u.x, a1 = silu_f32(g.y) * u.y;
    const float a2v = silu_f32(g.z) * u.z, a3 = silu_f32(g.w) * u.w;
    if (!FP8) {
      const uint2 o = make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(a2v, a3));
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(act) + static_cast<size_t>(r) * I)[c] = o;
      mx = max(max(o.x & 0x7FFFu, (o.x >> 16) & 0x7FFFu), max(o.y & 0x7FFFu, (o.y >> 16) & 0x7FFFu));
    } else {
      const float s = a2[0];
      const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(a0, s), __fdiv_rn(a1, s));
      const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(a2v, s), __fdiv_rn(a3, s));
      reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(act) + static_cast<size_t>(r) * I)[c] =
          lo | (hi << 16);
    }
  }
  if (amax != nullptr) {  // uniform over the grid: every thread of the warp takes part
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((threadIdx.x & 31) == 0 && mx != 0u) atomicMax(amax, mx);
  }
}

// y[r, h] = sum_p part[p][r][h] (bf16 out); 4 columns per thread.
__global__ void __launch_bounds__(256)
    down_finish_kernel(const float* __restrict__ part, int P, int64_t pstride, int H,
                       __nv_bfloat16* y) {
  const int r = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (c * 4 >= H) return;
  const float* row = part + static_cast<size_t>(r) * H;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int p = 0; p < P; ++p) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row + p * pstride) + c);
    s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
  }
  reinterpret_cast<uint2*>(y + static_cast<size_t>(r) * H)[c] =
      make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
}

}  // namespace

cudaError_t launch_unpermute_reduce(const void* y_perm, const int32_t* inv, const float* w, int T,
                                    int H, int k, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((H / 8 + 255) / 256, T);
  return launch_pdl(unpermute_reduce_kernel, grid, dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(y_perm), inv, w, H, k,
                    static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_unpermute_reduce_splitk(const float* part, int P, int64_t pstride, const int32_t* inv,
                                           const float* w, int T, int H, int k, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int col_blocks = (H / 4 + 63) / 64;
  if (static_cast<long long>(T) * col_blocks <= 1024)  // a few waves at most: spread the slots too
    return launch_pdl(unpermute_reduce_splitk_slots_kernel, dim3(col_blocks, T), dim3(64, kSplitSlotThreads), 0, s,
                      part, P, pstride, inv, w, H, k, static_cast<__nv_bfloat16*>(out));
  const dim3 grid((H / 8 + 255) / 256, T);
  return launch_pdl(unpermute_reduce_splitk_kernel, grid, dim3(256), 0, s, part, P, pstride, inv, w, H, k,
                    static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_swiglu_finish(const float* part, int P, int64_t pstride, int S, int I,
                                 const float* a2, int fp8, void* act, uint32_t* amax, cudaStream_t s) {
  if (S == 0) return cudaSuccess;
  const dim3 grid((I / 4 + 255) / 256, S);
  if (fp8)
    return launch_pdl(swiglu_finish_kernel<true>, grid, dim3(256), 0, s, part, P, pstride, I, a2, act,
                      static_cast<uint32_t*>(nullptr));
  return launch_pdl(swiglu_finish_kernel<false>, grid, dim3(256), 0, s, part, P, pstride, I, a2, act, amax);
}

cudaError_t launch_down_finish(const float* part, int P, int64_t pstride, int S, int H, void* y,
                               cudaStream_t s) {
  if (S == 0) return cudaSuccess;
  const dim3 grid((H / 4 + 255) / 256, S);
  return launch_pdl(down_finish_kernel, grid, dim3(256), 0, s, part, P, pstride, H,
                    static_cast<__nv_bfloat16*>(y));
}

}  // namespace moe
