// Stages 1 + 2 for small batches in one kernel: the gate (one warp per token),
// the per-expert histogram, the offsets scan, the stable ranking of the
// (token, expert) slots and the row gather, with no kernel boundary in between.
// A decode step would otherwise pay four dependent launches for a few
// microseconds of work.  Every CTA computes the whole routing in its own shared
// memory (at most kRouteMaxSlots slots: cheaper than waiting for another CTA),
// CTA 0 alone writes ids, weights, counts, offsets, perm and inv, and the
// gather is split into T x `chunks` pieces (a token's row in `chunks` column
// ranges, so a batch of a few tokens still spreads its k row copies over many
// SMs), CTA b taking pieces b, b + G, ...  The gate is the same per-token routine as
// gate_topk_kernel, the ranking gives the same unique stable order as
// align_count + align_scatter and the gather is the same per-token copy, so the
// results are bit-identical to that path.
#include "gate_token.cuh"
#include "gather_token.cuh"

namespace moe {

namespace {

constexpr int kRouteThreads = 1024;  // one thread per slot (S <= kRouteMaxSlots)
constexpr int kRouteWarps = kRouteThreads / 32;
static_assert(kRouteThreads >= kRouteMaxSlots, "one slot per thread");

template <int EPL, bool FP8>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_small_kernel(GateArgs g, AlignArgs a, int scratch_bytes, int chunks) {
  extern __shared__ __align__(16) unsigned char route_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  const bool writer = blockIdx.x == 0;
  // per-slot ids, weights and permuted rows, private to this CTA
  int32_t* s_ids = reinterpret_cast<int32_t*>(route_smem + scratch_bytes);
  float* s_w = reinterpret_cast<float*>(s_ids + kRouteMaxSlots);
  int* s_pos = reinterpret_cast<int*>(s_w + kRouteMaxSlots);
  pdl_wait();
  pdl_trigger();

  // gate: warp w takes tokens w, w + 32, ...; ids and weights into shared memory
  GateArgs gl = g;
  gl.ids = s_ids;
  gl.w = s_w;
  float* skeys = reinterpret_cast<float*>(route_smem) + warp * (32 * EPL);
  for (int t = warp; t < g.T; t += kRouteWarps) gate_detail::gate_token<EPL>(gl, t, lane, skeys);
  __syncthreads();
  if (writer) {
    for (int i = tid; i < a.S; i += kRouteThreads) {
      g.ids[i] = s_ids[i];
      g.w[i] = s_w[i];
    }
  }

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
    e = s_ids[f];
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      if (writer) record_error(a.err, kErrBadIndex, static_cast<uint32_t>(f));
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
    if (writer) {
      a.counts[tid] = v;
      a.offsets[tid] = o0;
    }
  }
  if (writer && tid == 0) a.offsets[E] = a.S;

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
    s_pos[f] = pos;
    if (writer) {
      a.perm[pos] = f;
      a.inv[f] = pos;
    }
  }
  __syncthreads();

  // gather: this CTA's pieces (token, column range), each to the rows its k
  // slots landed on
  const int nvec = a.H / 8;
  for (int w = blockIdx.x; w < g.T * chunks; w += gridDim.x) {
    const int t = w / chunks, c = w - t * chunks;
    gather_token<FP8>(a, t, s_pos + static_cast<size_t>(t) * a.k, c * nvec / chunks, (c + 1) * nvec / chunks, tid,
                      kRouteThreads);
  }
}

template <int EPL>
cudaError_t launch_route(const GateArgs& g, const AlignArgs& a, cudaStream_t s) {
  const size_t gate_bytes = sizeof(float) * kRouteWarps * 32 * EPL;
  const size_t align_bytes = sizeof(int) * (2 * a.E + 32) + sizeof(uint16_t) * kRouteWarps * a.E;
  const size_t scratch = ((gate_bytes > align_bytes ? gate_bytes : align_bytes) + 15) & ~static_cast<size_t>(15);
  const size_t slots = 3 * sizeof(int32_t) * kRouteMaxSlots;
  const size_t smem = scratch + slots;
  static int configured = -1;  // attribute set once per device (single-device processes)
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured != dev) {
    const int most = static_cast<int>(sizeof(float) * kRouteWarps * 32 * 32 + slots);
    err = cudaFuncSetAttribute(route_small_kernel<EPL, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(route_small_kernel<EPL, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (err != cudaSuccess) return err;
    configured = dev;
  }
  // up to one CTA per SM: every CTA repeats the routing, so more CTAs only
  // shorten the gather.  Batches of <= 4 tokens split a token's row into
  // column ranges of at least 64 x 8 elements until the pieces fill the SMs
  // (DeepSeek-V3 shapes, T = 1-4: 1-3% faster layer); larger ones keep one
  // piece per token, since routing CTAs beyond the tokens' count hold SMs the
  // next GEMM's prologue could use (TP8 slice, T = 64: 1.3% slower split).
  int sms = 0;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  int chunks = g.T <= 4 ? sms / g.T : 1;
  const int max_chunks = a.H / (8 * 64);
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  const int pieces = g.T * chunks;
  const int grid = pieces < sms ? pieces : sms;
  if (a.fp8)
    return launch_pdl(route_small_kernel<EPL, true>, dim3(grid), dim3(kRouteThreads), smem, s, g, a,
                      static_cast<int>(scratch), chunks);
  return launch_pdl(route_small_kernel<EPL, false>, dim3(grid), dim3(kRouteThreads), smem, s, g, a,
                    static_cast<int>(scratch), chunks);
}

}  // namespace

cudaError_t launch_route_small(const GateArgs& g, const AlignArgs& a, cudaStream_t s) {
  if (a.S == 0 || a.S > kRouteMaxSlots || a.E > 1024) return cudaErrorInvalidValue;
  if (a.E <= 64) return launch_route<2>(g, a, s);
  if (a.E <= 256) return launch_route<8>(g, a, s);
  return launch_route<32>(g, a, s);
}

}  // namespace moe
