// Stage 4: unpermute and top-k weighted reduction, with or without the down
// GEMM's split-K slices folded in.
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
// the down GEMM's own split-K finish (slice sum in slice order, bf16 y) followed
// by unpermute_reduce, so the result is bit-identical to that pair (and the
// permuted expert outputs never go through memory).
// Block (64, kSplitSlotThreads): a CTA owns 256 columns of one token.  First
// every (slot j, 4 columns) pair sums its P slices (threads along y take the
// slots, so a decode step's few tokens still spread over many warps with many
// loads in flight), rounds to bf16 and parks the result in shared memory; then
// the 64 threads of row y = 0 form the weighted sum in j order.
constexpr int kSplitSlotThreads = 8;

__global__ void __launch_bounds__(64 * kSplitSlotThreads)
    unpermute_reduce_splitk_kernel(const float* __restrict__ part, int P, int64_t pstride,
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
  const dim3 grid((H / 4 + 63) / 64, T);
  return launch_pdl(unpermute_reduce_splitk_kernel, grid, dim3(64, kSplitSlotThreads), 0, s, part, P, pstride,
                    inv, w, H, k, static_cast<__nv_bfloat16*>(out));
}

}  // namespace moe
