// Stage 1: top-k expert gate, one warp per token (the per-token selection is in
// gate_token.cuh).
#include "gate_token.cuh"

namespace moe {

namespace {

constexpr int kGateWarps = 8;

template <int EPL>
__global__ void __launch_bounds__(kGateWarps * 32) gate_topk_kernel(GateArgs a) {
  __shared__ float skeys[kGateWarps][32 * EPL];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kGateWarps + warp;
  pdl_wait();
  pdl_trigger();
  if (t >= a.T) return;  // whole warp leaves together
  gate_detail::gate_token<EPL>(a, t, lane, skeys[warp]);
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
