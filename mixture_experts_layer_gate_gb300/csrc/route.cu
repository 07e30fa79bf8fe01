// Stages 1 + 2 for small batches in one CTA: the gate (one warp per token), the
// per-expert histogram, the offsets scan and the stable ranking of the (token,
// expert) slots, with no kernel boundary in between.  A decode step would
// otherwise pay three dependent launches for a few microseconds of work.  The
// gate is the same per-token routine as gate_topk_kernel and the ranking gives
// the same unique stable order as align_count + align_scatter, so the results
// are bit-identical to that path.
#include "gate_token.cuh"

namespace moe {

namespace {

constexpr int kRouteThreads = 1024;  // one thread per slot (S <= kRouteMaxSlots)
constexpr int kRouteWarps = kRouteThreads / 32;
static_assert(kRouteThreads >= kRouteMaxSlots, "one slot per thread");

template <int EPL>
__global__ void __launch_bounds__(kRouteThreads, 1) route_small_kernel(GateArgs g, AlignArgs a) {
  extern __shared__ __align__(16) unsigned char route_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  pdl_wait();
  pdl_trigger();

  // gate: warp w takes tokens w, w + 32, ...; ids go to global memory
  float* skeys = reinterpret_cast<float*>(route_smem) + warp * (32 * EPL);
  for (int t = warp; t < g.T; t += kRouteWarps) gate_detail::gate_token<EPL>(g, t, lane, skeys);
  __syncthreads();  // the block's ids writes are visible to the block from here on

  // the gate's shared memory is reused for the histogram and rank tables
  int* hist = reinterpret_cast<int*>(route_smem);        // [E]
  int* off = hist + E;                                    // [E]
  int* warp_sums = off + E;                               // [32]
  uint16_t* wc = reinterpret_cast<uint16_t*>(warp_sums + 32);  // [32][E]
  for (int e = tid; e < E; e += kRouteThreads) hist[e] = 0;
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wc[i] = 0;
  __syncthreads();
  const int f = tid;
  const bool valid = f < a.S;
  int e = -1;
  if (valid) {
    e = __ldcg(a.ids + f);  // L2 load: written by this block above
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      record_error(a.err, kErrBadIndex, static_cast<uint32_t>(f));
      e = 0;
    }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();

  // exclusive scan of the histogram (E <= 1024 entries, one per thread)
  const int v = (tid < E) ? hist[tid] : 0;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  if (tid < E) {
    const int o0 = warp_sums[warp] + incl - v;
    off[tid] = o0;
    a.counts[tid] = v;
    a.offsets[tid] = o0;
  }
  if (tid == 0) a.offsets[E] = a.S;

  // stable rank: slots of one expert in ascending slot order
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(same & ((1u << lane) - 1u));
  if (valid && rank == 0) wc[warp * E + e] = static_cast<uint16_t>(__popc(same));
  __syncthreads();
  for (int x = tid; x < E; x += kRouteThreads) {
    int acc = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = wc[w * E + x];
      wc[w * E + x] = static_cast<uint16_t>(acc);
      acc += c;
    }
  }
  __syncthreads();
  if (valid) {
    const int pos = off[e] + wc[warp * E + e] + rank;
    a.perm[pos] = f;
    a.inv[f] = pos;
  }
}

template <int EPL>
cudaError_t launch_route(const GateArgs& g, const AlignArgs& a, cudaStream_t s) {
  const size_t gate_bytes = sizeof(float) * kRouteWarps * 32 * EPL;
  const size_t align_bytes = sizeof(int) * (2 * a.E + 32) + sizeof(uint16_t) * kRouteWarps * a.E;
  const size_t smem = gate_bytes > align_bytes ? gate_bytes : align_bytes;
  static int configured = -1;  // attribute set once per device (single-device processes)
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured != dev) {
    err = cudaFuncSetAttribute(route_small_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(float) * kRouteWarps * 32 * 32));
    if (err != cudaSuccess) return err;
    configured = dev;
  }
  return launch_pdl(route_small_kernel<EPL>, dim3(1), dim3(kRouteThreads), smem, s, g, a);
}

}  // namespace

cudaError_t launch_route_small(const GateArgs& g, const AlignArgs& a, cudaStream_t s) {
  if (a.S == 0 || a.S > kRouteMaxSlots || a.E > 1024) return cudaErrorInvalidValue;
  if (a.E <= 64) return launch_route<2>(g, a, s);
  if (a.E <= 256) return launch_route<8>(g, a, s);
  return launch_route<32>(g, a, s);
}

}  // namespace moe
