// Stage 2: align and permute.
//
// "[Kernel] add triton fused moe kernel for gptq/awq" (vLLM), note 1: the
// shared-memory moe_align_block_size made DeepSeek-V3 (E = 256) usable under
// CUDA graphs; "Add deepseek_v3 fused gate" (sglang): TensorRT-LLM's
// expand_and_permute lays the token rows out expert-contiguous with no padding.
//
// A stable counting sort of the S = T*k slots by expert, with no host sync:
//   align_count   : per CTA of 1024 slots, a shared-memory histogram.
//   align_scatter : per CTA, expert totals and its own base (sum over earlier
//                   CTAs) from the histograms, an exclusive scan for offsets,
//                   then a rank for each slot that keeps ascending slot order
//                   inside an expert (warp match + per-warp prefix counts).
//   gather_rows   : x_perm[inv[t*k + j]] = x[t] for each of token t's k slots
//                   (fp8: e4m3 of x / a1, quantised once per token).
#include "common.cuh"
#include "gather_token.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kScatterThreads = 512;
constexpr int kGatherThreads = 256;
constexpr int kGatherMaxK = 32;  // top_k limit of the problem checks
constexpr int kScatterWarps = kScatterThreads / 32;

__global__ void __launch_bounds__(512) align_count_kernel(AlignArgs a) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) hist[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int base = blockIdx.x * kAlignSlotsPerCta;
  const int end = min(a.S, base + kAlignSlotsPerCta);
  for (int f = base + threadIdx.x; f < end; f += blockDim.x) {
    int e = a.ids[f];
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(a.E)) {
      record_error(a.err, kErrBadIndex, static_cast<uint32_t>(f));
      e = 0;
    }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x)
    a.block_counts[static_cast<size_t>(blockIdx.x) * a.E + e] = hist[e];
}

// Exclusive scan of v[0..n) in place (n <= 1024) by a block of 512 threads.
__device__ void block_exclusive_scan(int* v, int n, int* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kScatterThreads - 1) / kScatterThreads;  // <= 2
  const int i0 = tid * per;
  int local[2] = {0, 0};
  int s = 0;
  for (int j = 0; j < per; ++j) {
    const int i = i0 + j;
    local[j] = (i < n) ? v[i] : 0;
    s += local[j];
  }
  int incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = (lane < kScatterWarps) ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kScatterWarps) warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  int run = warp_sums[warp] + incl - s;
  for (int j = 0; j < per; ++j) {
    const int i = i0 + j;
    if (i < n) v[i] = run;
    run += local[j];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kScatterThreads) align_scatter_kernel(AlignArgs a, int nblk) {
  extern __shared__ int smem[];
  const int E = a.E;
  int* run = smem;                      // [E] next row for each expert in this CTA
  int* off = run + E;                   // [E] expert offsets
  int* ctot = off + E;                  // [E] per-chunk totals
  int* warp_sums = ctot + E;            // [32]
  uint16_t* wc = reinterpret_cast<uint16_t*>(warp_sums + 32);  // [warps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();

  for (int e = tid; e < E; e += kScatterThreads) {
    int tot = 0, before = 0;
    for (int b = 0; b < nblk; ++b) {
      const int c = a.block_counts[static_cast<size_t>(b) * E + e];
      if (b < static_cast<int>(blockIdx.x)) before += c;
      tot += c;
    }
    off[e] = tot;
    run[e] = before;
    for (int w = 0; w < kScatterWarps; ++w) wc[w * E + e] = 0;
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e < E; e += kScatterThreads) a.counts[e] = off[e];
  block_exclusive_scan(off, E, warp_sums);
  for (int e = tid; e < E; e += kScatterThreads) {
    run[e] += off[e];
    if (blockIdx.x == 0) a.offsets[e] = off[e];
  }
  if (blockIdx.x == 0 && tid == 0) a.offsets[E] = a.S;
  __syncthreads();

  const int base = blockIdx.x * kAlignSlotsPerCta;
  const int end = min(a.S, base + kAlignSlotsPerCta);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = base; c0 < end; c0 += kScatterThreads) {
    const int f = c0 + tid;
    const bool valid = f < end;
    int e = -1;
    if (valid) {
      e = a.ids[f];
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = 0;  // recorded by count
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    if (valid && rank == 0) wc[warp * E + e] = static_cast<uint16_t>(__popc(same));
    __syncthreads();
    for (int x = tid; x < E; x += kScatterThreads) {
      int acc = 0;
      for (int w = 0; w < kScatterWarps; ++w) {
        const int v = wc[w * E + x];
        wc[w * E + x] = static_cast<uint16_t>(acc);
        acc += v;
      }
      ctot[x] = acc;
    }
    __syncthreads();
    if (valid) {
      const int pos = run[e] + wc[warp * E + e] + rank;
      a.perm[pos] = f;
      a.inv[f] = pos;
    }
    __syncthreads();
    for (int x = tid; x < E; x += kScatterThreads) {
      run[x] += ctot[x];
      for (int w = 0; w < kScatterWarps; ++w) wc[w * E + x] = 0;
    }
    __syncthreads();
  }
}

// One CTA per token: its row is read once, quantised once (fp8), and written to
// the k permuted rows its slots landed on (inv).  A CTA per permuted row read
// and quantised each token row k times; the divisions of the fp8 path made
// that instruction-bound.
template <bool FP8>
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(AlignArgs a) {
  __shared__ int rows[kGatherMaxK];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < a.k) rows[threadIdx.x] = a.inv[static_cast<size_t>(t) * a.k + threadIdx.x];
  __syncthreads();
  gather_token<FP8>(a, t, rows, 0, a.H / 8, threadIdx.x, kGatherThreads);
}

__global__ void __launch_bounds__(256)
    align_block_size_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
                            int E, int S, int block, int32_t* sorted_ids, int32_t* block_expert,
                            int32_t* total_out) {
  extern __shared__ int poff[];  // [E + 1]
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      poff[e] = acc;
      const int c = offsets[e + 1] - offsets[e];
      acc += ((c + block - 1) / block) * block;
    }
    poff[E] = acc;
    if (blockIdx.x == 0) *total_out = acc;
  }
  __syncthreads();
  const int total = poff[E];
  for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < total; q += gridDim.x * blockDim.x) {
    int lo = 0, hi = E;  // largest e with poff[e] <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (poff[mid] <= q) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int r = q - poff[e];
    const int c = offsets[e + 1] - offsets[e];
    sorted_ids[q] = (r < c) ? perm[offsets[e] + r] : S;
    if (r % block == 0) block_expert[q / block] = e;
  }
}

}  // namespace

cudaError_t launch_align(const AlignArgs& a, cudaStream_t s) {
  if (a.S == 0) {
    cudaError_t err = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.E, s);
    if (err != cudaSuccess) return err;
    return cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.E + 1), s);
  }
  const int nblk = align_blocks(a.S);
  cudaError_t err = launch_pdl(align_count_kernel, dim3(nblk), dim3(512), sizeof(int) * a.E, s, a);
  if (err != cudaSuccess) return err;
  const size_t scatter_smem = sizeof(int) * (3 * a.E + 32) + sizeof(uint16_t) * kScatterWarps * a.E;
  err = launch_pdl(align_scatter_kernel, dim3(nblk), dim3(kScatterThreads), scatter_smem, s, a, nblk);
  if (err != cudaSuccess) return err;
  return launch_gather(a, s);
}

cudaError_t launch_gather(const AlignArgs& a, cudaStream_t s) {
  if (a.S == 0) return cudaSuccess;
  const int T = a.S / a.k;
  if (a.fp8) return launch_pdl(gather_rows_kernel<true>, dim3(T), dim3(kGatherThreads), 0, s, a);
  return launch_pdl(gather_rows_kernel<false>, dim3(T), dim3(kGatherThreads), 0, s, a);
}

cudaError_t launch_align_block_size(const int32_t* offsets, const int32_t* perm, int E, int S,
                                    int block, size_t capacity, int32_t* sorted_ids,
                                    int32_t* block_expert, int32_t* total, cudaStream_t s) {
  int grid = static_cast<int>((capacity + 255) / 256);
  if (grid < 1) grid = 1;
  if (grid > 1024) grid = 1024;
  return launch_pdl(align_block_size_kernel, dim3(grid), dim3(256), sizeof(int) * (E + 1), s, offsets,
                    perm, E, S, block, sorted_ids, block_expert, total);
}

}  // namespace moe
