// moe_align_permute_noalloc: the align/permute stage for callers that cannot
// allocate device memory.  Same kernels and results as moe_align_permute; the
// per-CTA expert histograms it needs between its two passes live in a
// fixed-size array that is part of the library's own device image instead of
// a caller-provided workspace.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Room for 65 536 int32 per-CTA expert counts: ceil(T*k / 1024) * E <= 65 536,
// e.g. E = 256 experts up to T*k = 262 144 slots, or E = 1024 up to 65 536.
constexpr size_t kNoAllocScratchBytes = 256 * 1024;

// One copy per device that loads the library; it stays allocated until the
// process exits.  Host code must not pass this symbol to a kernel: on the host
// it names a host-side shadow, so its device address is looked up below.
static __device__ __align__(256) unsigned char g_align_scratch[kNoAllocScratchBytes];

// The array's device address is cached per CUDA context (the address belongs to
// the module as loaded into one context: another context on the same device,
// or the primary context re-created after a device reset, has its own copy).
constexpr int kMaxContexts = 64;
std::mutex g_mu;
struct CachedAddress {
  CUcontext ctx;
  void* addr;
};
CachedAddress g_cache[kMaxContexts] = {};
int g_cached = 0;

PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Device address of g_align_scratch in the current context, looked up with
// cudaGetSymbolAddress the first time a context calls (the runtime makes the
// device's primary context current if none is) and cached for it.
cudaError_t scratch_address(void** out) {
  auto get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  void* fresh = nullptr;
  if (ctx == nullptr) {
    // no context bound to this thread yet: the symbol lookup binds the current
    // device's primary context, which is then the one to key the address by
    const cudaError_t err = cudaGetSymbolAddress(&fresh, g_align_scratch);
    if (err != cudaSuccess) return err;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_cached; ++i) {
    if (g_cache[i].ctx == ctx) {
      *out = g_cache[i].addr;
      return cudaSuccess;
    }
  }
  if (g_cached == kMaxContexts) return cudaErrorNotSupported;  // cache full: refuse, never guess
  if (fresh == nullptr) {
    const cudaError_t err = cudaGetSymbolAddress(&fresh, g_align_scratch);
    if (err != cudaSuccess) return err;
  }
  g_cache[g_cached++] = CachedAddress{ctx, fresh};
  *out = fresh;
  return cudaSuccess;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" moe_status_t moe_align_permute_noalloc(const moe_problem_t* p, const int32_t* topk_ids,
                                                  const void* x, const float* a1_scale,
                                                  int32_t* counts, int32_t* offsets, int32_t* perm,
                                                  int32_t* inv, void* x_perm,
                                                  moe_stream_t stream) {
  // Same problem checks and statuses as every other entry point.
  const moe_status_t st = moe::validate_problem(p);
  if (st != MOE_OK) return st;
  const long long S = static_cast<long long>(p->T) * p->top_k;
  const long long need = static_cast<long long>(moe::align_blocks(static_cast<int>(S))) * p->E * 4;
  if (need > static_cast<long long>(kNoAllocScratchBytes)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4)) return MOE_ERR_INVALID_ARG;
  if (p->T > 0) {
    if (!topk_ids || !x || !perm || !inv || !x_perm || !aligned(x, 16) || !aligned(x_perm, 16) ||
        !aligned(perm, 4) || !aligned(inv, 4) || !aligned(topk_ids, 4))
      return MOE_ERR_INVALID_ARG;
    if (p->wdtype == MOE_W_FP8_E4M3 && !a1_scale) return MOE_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  moe::AlignArgs a;
  a.ids = topk_ids;
  a.S = static_cast<int>(S);
  a.E = p->E;
  a.k = p->top_k;
  a.H = p->H;
  // Every histogram entry the scatter pass reads is written by the count pass
  // of the same call, so nothing in the array has to start at zero.
  a.block_counts = static_cast<int32_t*>(scratch);
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.x = x;
  a.x_perm = x_perm;
  a.a1 = a1_scale;
  a.fp8 = p->wdtype == MOE_W_FP8_E4M3;
  a.err = nullptr;  // no workspace header to report bad ids into
  return moe::launch_align(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK
                                                                                     : MOE_ERR_CUDA;
}
