// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace layout, launch planning (token tile, split-K, pipeline depth),
// TMA descriptor encoding and the stage launches.  No call here synchronises
// with the host except moe_get_device_error.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void moe::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxSplits = 16;
constexpr int kMaxStages = 8;  // bf16 / fp8 operand ring (12 measured no better)
constexpr int kMaxStagesInt4 = 8;
constexpr int kMaxSlotsInt4 = 7;  // int4 / int8: converted weight tiles in TMEM
constexpr int kSuper = kInt4StageKb;  // int4 / int8: k-blocks per ring stage
constexpr int kSmsForSizing = 160;  // upper bound on SMs used when sizing split-K scratch
constexpr size_t kMaxDynSmem = 232448;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int roundup16(int x) { return (x + 15) & ~15; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

moe_status_t moe::validate_problem(const moe_problem_t* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->H <= 0 || p->I <= 0 || p->E <= 0 || p->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (p->H % 128 != 0 || p->I % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (p->top_k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->E > kMaxE || p->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (p->T > 65535) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(p->T) * p->top_k > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (p->scoring != MOE_SCORE_SOFTMAX && p->scoring != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (p->renormalize != 0 && p->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(p->routed_scaling_factor)) return MOE_ERR_INVALID_ARG;
  if (p->n_group < 0 || p->topk_group < 0) return MOE_ERR_INVALID_ARG;
  if (p->n_group > 0) {
    if (p->scoring != MOE_SCORE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    if (p->n_group > 32 || p->E % p->n_group != 0) return MOE_ERR_INVALID_ARG;
    if (p->topk_group < 1 || p->topk_group > p->n_group) return MOE_ERR_INVALID_ARG;
    if (p->top_k > p->topk_group * (p->E / p->n_group)) return MOE_ERR_INVALID_ARG;
  } else if (p->topk_group != 0) {
    return MOE_ERR_INVALID_ARG;
  }
  if (p->wdtype != MOE_W_BF16 && p->wdtype != MOE_W_FP8_E4M3 && p->wdtype != MOE_W_INT4_G128 &&
      p->wdtype != MOE_W_INT8_G128 && p->wdtype != MOE_W_INT4_G128_PAIRED)
    return MOE_ERR_INVALID_ARG;
  if ((p->wdtype == MOE_W_INT4_G128 || p->wdtype == MOE_W_INT4_G128_PAIRED || p->wdtype == MOE_W_INT8_G128) &&
      p->group_size != 128)
    return MOE_ERR_UNSUPPORTED;
  if (p->act_scale != MOE_ACT_SCALE_STATIC && p->act_scale != MOE_ACT_SCALE_DYNAMIC) return MOE_ERR_INVALID_ARG;
  if (p->act_scale == MOE_ACT_SCALE_DYNAMIC && p->wdtype != MOE_W_FP8_E4M3) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

namespace {

// ------------------------------------------------------------ device facts

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

cudaError_t device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  *out = cache[dev];
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr),
                  reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides_bytes),
                  reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- planning

struct GemmPlan {
  int bn_max, P, stages, astages, slot_kb, conv_groups, ksplit, acc_cols, acc_bufs, pair, dual, full_box, FB, KB;
  int epi_warps;
  size_t smem;
};

// Planner overrides set through moe_set_tuning (tests and benchmarks only; a
// field of -1 leaves the planner's choice).  Nothing is read from the
// environment: a process gets these only by calling moe_set_tuning.
std::mutex g_tuning_mu;
moe_tuning_t g_tuning = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};

moe_tuning_t current_tuning() {
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  return g_tuning;
}

// The override of one knob, or `dflt` when it is unset.
inline int knob(int32_t v, int dflt) { return v < 0 ? dflt : v; }

int wkind_of(const moe_problem_t& p) {
  switch (p.wdtype) {
    case MOE_W_FP8_E4M3: return kW_FP8;
    case MOE_W_INT4_G128: return kW_INT4;
    case MOE_W_INT4_G128_PAIRED: return kW_INT4;
    case MOE_W_INT8_G128: return kW_INT8;
    default: return kW_BF16;
  }
}

// Token tile limit: generous enough that one tile usually holds all of an
// expert's tokens (each extra token block re-reads the expert's weights).
// int4 / int8 keep the converted weight tiles in TMEM beside the accumulators:
// up to 128 columns with two accumulator buffers (and two MMA issuers), above
// that (CTA pairs only) one buffer and one issuer.  Each tile converts the
// weights once, so many rows per expert favour wide tiles: measured on the
// DeepSeek-V3 int4 shape (T = 4096, 128 rows per expert on average: 192-token
// tiles 4% faster than 128, 256 slower: its 80 KB ring stages leave two) and
// the Mixtral int8 shape (T = 1024 and 4096, 256 and 1024 rows per expert:
// 256-token tiles 18-25% faster).
int plan_bn_max(const moe_problem_t& p) {
  const long long S = static_cast<long long>(p.T) * p.top_k;
  if (S <= 0) return 16;
  const long long touched = std::max(1ll, std::min<long long>(p.E, S));
  const long long m_avg = (S + touched - 1) / touched;
  long long bn = std::max(3 * m_avg, m_avg + 24);
  long long cap = 256;
  if (wkind_of(p) == kW_INT4) cap = m_avg >= 128 ? 192 : 128;
  if (p.wdtype == MOE_W_INT8_G128) cap = m_avg >= 192 ? 256 : 128;
  bn = std::min<long long>(cap, std::max<long long>(16, bn));
  return roundup16(static_cast<int>(bn));
}

long long plan_tiles(const moe_problem_t& p, bool up, int bn_max) {
  const long long S = static_cast<long long>(p.T) * p.top_k;
  const long long touched = std::max(1ll, std::min<long long>(p.E, S));
  const long long m_avg = (S + touched - 1) / touched;
  const int FB = up ? p.I / 64 : p.H / 128;
  return touched * ((m_avg + bn_max - 1) / bn_max) * FB;
}

// Split-K factor: the smallest P whose units fill their waves of the SM count
// to min_eff.  int4 / int8 units carry more fixed cost (converter pipeline,
// group scales), so they accept emptier waves before splitting: the DeepSeek-V3
// int4 gate_up at T = 1 took 51.8 us unsplit (84% of one wave's SMs busy) and
// 58.1 us in four slices.
int plan_splits(const moe_problem_t& p, bool up, int bn_max, int KB, int sms) {
  const long long tiles = plan_tiles(p, up, bn_max);
  if (tiles >= 4ll * sms) return 1;
  const double min_eff = converts(wkind_of(p)) ? 0.8 : 0.9;
  const int pmax = std::max(1, std::min(kMaxSplits, KB / 4));
  int best = 1;
  double best_eff = 0.0;
  for (int P = 1; P <= pmax; ++P) {
    const long long units = tiles * P;
    const long long waves = (units + sms - 1) / sms;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * sms);
    if (eff >= min_eff) return P;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = P;
    }
  }
  return best;
}

GemmPlan plan_gemm(const moe_problem_t& p, bool up, int sms) {
  GemmPlan g;
  const int wk = wkind_of(p);
  g.bn_max = plan_bn_max(p);
  const moe_tuning_t tu = current_tuning();
  const int bn_env = knob(tu.bn_max, 0);
  if (bn_env >= 16 && bn_env <= 256 && bn_env % 16 == 0) g.bn_max = bn_env;
  g.FB = up ? p.I / 64 : p.H / 128;
  const int K = up ? p.H : p.I;
  g.KB = K / (wk == kW_FP8 ? 128 : 64);
  g.P = plan_splits(p, up, g.bn_max, g.KB, std::min(sms, kSmsForSizing));
  const int p_env = knob(tu.splits, 0);
  if (p_env >= 1 && p_env <= kMaxSplits && p_env <= std::max(1, g.KB / 4)) g.P = p_env;
  size_t per_stage;
  int cap;
  g.conv_groups = 0;
  g.ksplit = 0;
  g.dual = 0;
  g.acc_bufs = 2;
  // int4 / int8: one CTA per 128 weight rows for small token tiles (<= 32
  // tokens), CTA pairs (M = 256 per MMA) above that, as for bf16 / fp8 whenever
  // the weight blocks pair up.  Two MMA-issuing threads for every int4 GEMM and
  // for int8 tiles of <= 32 tokens.  Measured on DeepSeek-V3 int4 (T = 1 to
  // 4096: two issuers 8-20% faster up to T = 1024, 2% at 4096) and Mixtral int8
  // (T = 1 to 4096: 8-11% faster at <= 32 tokens, neutral to 1.6% slower above;
  // one CTA at 64 tokens leaves int8's larger stages a shallow ring).
  // Converting kernels load whole token tiles too: one TMA per stage keeps the
  // producer thread, which shares its SM sub-partition with integer-bound
  // converter warps, short of instructions.
  const bool small_tile = converts(wk) && g.bn_max <= 32;
  const bool dual_fit = wk == kW_INT4 || (wk == kW_INT8 && small_tile);
  g.pair = 0;
  const int pair_env = knob(tu.pair, -1);
  // Small int4 / int8 tiles whose units carry <= 8 k-blocks (the DeepSeek-V3
  // TP8 down GEMM, K = 256) pair up too once a batch has >= 64 rows: a unit
  // then covers two weight blocks for the same fixed cost per unit (down GEMM
  // 9-22% faster at T = 16-256; within 3% at T = 4-8; 4-5% slower at T <= 2,
  // and long-K GEMMs 6% slower, which keep one CTA per weight block).
  const long long S_rows = static_cast<long long>(p.T) * p.top_k;
  const bool short_units = g.KB / g.P <= 8 && S_rows >= 64;
  if (g.FB % 2 == 0 && (pair_env == 1 || (pair_env != 0 && (!small_tile || short_units)))) {
    g.pair = 1;
    g.bn_max = std::max(32, (g.bn_max + 31) / 32 * 32);
  }
  // int4 / int8 on one CTA stage all of a tile's token rows for four k-blocks
  // per ring stage: above 128 rows no second stage fits in shared memory
  if (converts(wk) && !g.pair) g.bn_max = std::min(g.bn_max, 128);
  // Token tiles always load as one box of the full tile height (rows past a
  // short tile are loaded and ignored): on CTA pairs this measured 16% faster
  // for the Mixtral T = 4096 layer (gate_up 1.33 -> 1.17 ms) and 2-11 points of
  // roofline better for Mixtral, Qwen2 and Scout at 64-4096 tokens, with no
  // batch size slower, against 64- and 16-row boxes for an expert's last tile.
  g.full_box = knob(tu.full_box, 1) != 0 ? 1 : 0;
  bool one_slot = false;  // int4 / int8: two wide accumulators beside one converted slot
  if (converts(wk)) {
    // TMEM: two accumulators of acc_cols columns, then converted slots of
    // slot_kb k-blocks (32 columns each).  A converter group that fills the
    // 4 / slot_kb slots of its stage jumps (groups - 1) * 4 / slot_kb slots
    // ahead, so the slot ring needs one more than that (parity-wait rule).
    // Whole-stage slots (one wait and one commit per 16 MMAs) when TMEM holds
    // one per group; else two-k-block slots.
    g.acc_cols = (g.bn_max + 31) / 32 * 32;
    // Two MMA-issuing threads (whole-stage slots): each keeps its own partial
    // accumulators, two buffers of them where that leaves room for two
    // whole-stage slots (<= 64 columns), else one buffer (<= 128 columns; the
    // epilogue of a unit then no longer overlaps the next unit's MMAs).
    // Tiles of more than 128 tokens (CTA pairs only): one issuer and one
    // accumulator of up to 256 columns beside two whole-stage slots.  Each
    // converted weight tile then serves up to 256 tokens, so an expert with
    // 129..256 rows is converted once instead of twice, and the MMAs of a
    // stage (M = 256, N up to 256) outlast its conversion.
    // A second issuer that costs the second accumulator buffer (tiles of 65-128
    // tokens) only where units carry >= 16 k-blocks: with fewer, a unit's MMAs
    // are shorter than its epilogue, which must then overlap the next unit's
    // MMAs (DeepSeek-V3 TP8 slice, down GEMM with K = 256, T = 2048: 0.446 ms
    // with two issuers and one buffer, 0.365 ms with one issuer and two).
    // Tiles of 129-192 tokens can instead take two accumulator buffers beside a
    // single whole-stage slot that both converter groups fill (k-split; tuning
    // only): each stage's conversion then waits for the previous stage's MMAs.
    // On short-K units (the DeepSeek-V3 TP8 down GEMM, K = 256, T = 4096) it
    // measured no faster (0.471 vs 0.467 ms), on long ones far slower.
    const bool dual_pays = g.acc_cols <= 64 || g.KB / g.P >= 16;
    const int dual_env = knob(tu.dual, -1);
    const int ab_env = knob(tu.acc_bufs, 0);
    if (g.acc_cols > 128) {
      g.acc_bufs = 1;
      if (g.acc_cols <= 192 && ab_env == 2) {
        g.acc_bufs = 2;
        one_slot = true;
      }
    } else if (dual_env == 1 || (dual_env != 0 && dual_fit && dual_pays)) {
      g.dual = 1;
      g.acc_bufs = g.acc_cols <= 64 ? 2 : 1;
    }
    const int free_cols = 512 - (g.dual ? 2 : 1) * g.acc_bufs * g.acc_cols;
    const int cg_env = knob(tu.conv_groups, 0);
    const int sk_env = knob(tu.slot_kb, 0);
    // Converter groups: three for int4 tiles of <= 32 tokens on one CTA with two
    // MMA issuers, where TMEM holds the third whole-stage slot beside two pairs of
    // 32-column partial accumulators (DeepSeek-V3 shape, T = 8 to 64: 4-9% faster
    // than two; 608 threads leave 96 registers, a few spilled outside the dequant
    // loop).  Two elsewhere: with one issuer a third measured no faster (single-
    // thread issue, of TMA copies and of MMAs, set the pace); three remain
    // available with CTA pairs and one MMA issuer for tuning.
    g.conv_groups = 2;
    if (wk == kW_INT4 && !g.pair && g.dual && g.acc_cols <= 32 && cg_env != 2) g.conv_groups = 3;
    if (cg_env == 3 && g.pair && wk == kW_INT4 && !g.dual) g.conv_groups = 3;
    auto slots_needed = [&](int sk) { return (g.conv_groups - 1) * (kSuper / sk) + 1; };
    auto slots_fit = [&](int sk) { return std::min(kMaxSlotsInt4, free_cols / (32 * sk)); };
    g.slot_kb = (slots_fit(4) >= slots_needed(4)) ? 4 : 2;
    if ((sk_env == 2 || sk_env == 4) && !g.dual && slots_fit(sk_env) >= slots_needed(sk_env)) g.slot_kb = sk_env;
    if (slots_fit(g.slot_kb) < slots_needed(g.slot_kb)) g.conv_groups = 2;  // 3 groups do not fit
    g.astages = slots_fit(g.slot_kb);
    if (one_slot) {
      g.conv_groups = 2;
      g.slot_kb = kSuper;
      g.astages = 1;
    }
    per_stage = static_cast<size_t>(raw_stage_bytes(wk)) + 4 * static_cast<size_t>(g.pair ? g.bn_max / 2 : g.bn_max) * 128 + 16;
    cap = kMaxStagesInt4;
  } else {
    g.acc_cols = 256;
    g.astages = 0;
    g.slot_kb = 0;
    per_stage = 16384 + static_cast<size_t>(g.pair ? g.bn_max / 2 : g.bn_max) * 128 + 16;
    cap = kMaxStages;
  }
  // Epilogue warps: eight (two per TMEM lane quarter, alternate 32-token
  // columns) on bf16 / fp8 CTA pairs, where a short-K down GEMM otherwise waits
  // on its epilogue (Qwen2 tensor-parallel slice, I = 640, T = 4096: down GEMM
  // 0.130 -> 0.105 ms; no workload measured slower); four elsewhere.
  g.epi_warps = (!converts(wk) && g.pair) ? 8 : 4;
  const int ew_env = knob(tu.epi_warps, 0);
  if (ew_env == 4 || (ew_env == 8 && gemm_epi8_supported(wk, g.conv_groups, g.pair, g.slot_kb)))
    g.epi_warps = ew_env;
  // rows of token tile each CTA stages per K step
  const int brows = g.pair ? g.bn_max / 2 : g.bn_max;
  const size_t fixed = gemm_smem_bytes(wk, brows, 0, g.astages, p.E, g.epi_warps);
  g.stages = static_cast<int>(std::min<size_t>(cap, (kMaxDynSmem - fixed) / per_stage));
  const int st_env = knob(tu.stages, 0);
  if (st_env >= 2 && st_env < g.stages) g.stages = st_env;
  while (g.stages > 2 && gemm_smem_bytes(wk, brows, g.stages, g.astages, p.E, g.epi_warps) > kMaxDynSmem)
    --g.stages;
  if (converts(wk)) {
    // Converter groups alternating stages need a ring depth that is a multiple of
    // the group count (parity-wait rule: a stage's previous user was the same
    // group).  k-split (both groups convert every stage, each half its k-blocks)
    // has no such rule but more bookkeeping per stage (measured slower at equal
    // depth), so it is taken only where rounding down would leave a shallow ring
    // (int8 codes with 128-token tiles: three stages instead of two).
    const int alt = g.stages - g.stages % g.conv_groups;
    const int ks_env = knob(tu.ksplit, -1);
    const bool can_ks = g.conv_groups == 2 && g.slot_kb == kSuper;
    g.ksplit = (can_ks && (one_slot || ks_env == 1 || (ks_env != 0 && alt < 4 && g.stages > alt))) ? 1 : 0;
    if (!g.ksplit) g.stages = alt;
  }
  // whole-stage slots: converters wait on the stage ring for slot reuse, which
  // needs at least as many ring stages as slots (parity-wait rule)
  if (converts(wk) && g.slot_kb == kSuper && g.astages > g.stages) g.astages = g.stages;
  g.smem = gemm_smem_bytes(wk, brows, g.stages, g.astages, p.E, g.epi_warps);
  return g;
}

// ---------------------------------------------------------- workspace layout

struct Layout {
  size_t hdr, align_counts, partial, act_bf16, scratch_end;
  size_t ids, w, counts, offsets, perm, inv, x_perm, act, y_perm, total;
};

size_t partial_bytes(const moe_problem_t& p, bool up) {
  const int bn = plan_bn_max(p);
  const long long tiles = plan_tiles(p, up, bn);
  if (tiles >= 4ll * kSmsForSizing) return 0;
  const size_t S = static_cast<size_t>(p.T) * p.top_k;
  const size_t N = up ? 2 * static_cast<size_t>(p.I) : static_cast<size_t>(p.H);
  return static_cast<size_t>(kMaxSplits) * S * N * sizeof(float);
}

Layout layout_of(const moe_problem_t& p) {
  Layout L;
  const size_t S = static_cast<size_t>(p.T) * p.top_k;
  const size_t esz = (p.wdtype == MOE_W_FP8_E4M3) ? 1 : 2;
  size_t o = 0;
  L.hdr = o;
  o += kHeaderBytes;
  L.align_counts = o;
  o = align256(o + static_cast<size_t>(std::max(1, align_blocks(static_cast<int>(S)))) * p.E * 4);
  L.partial = o;
  o = align256(o + std::max(partial_bytes(p, true), partial_bytes(p, false)));
  // dynamic fp8 scales: the SwiGLU output in bf16 before its scale is known
  L.act_bf16 = o;
  if (p.act_scale == MOE_ACT_SCALE_DYNAMIC) o = align256(o + S * p.I * 2);
  L.scratch_end = o;
  L.ids = o;
  o = align256(o + S * 4);
  L.w = o;
  o = align256(o + S * 4);
  L.counts = o;
  o = align256(o + static_cast<size_t>(p.E) * 4);
  L.offsets = o;
  o = align256(o + static_cast<size_t>(p.E + 1) * 4);
  L.perm = o;
  o = align256(o + S * 4);
  L.inv = o;
  o = align256(o + S * 4);
  L.x_perm = o;
  o = align256(o + S * p.H * esz);
  L.act = o;
  o = align256(o + S * p.I * esz);
  L.y_perm = o;
  o = align256(o + S * p.H * 2);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool dynamic_scales(const moe_problem_t& p) { return p.act_scale == MOE_ACT_SCALE_DYNAMIC; }
DynScales* dyn_of(void* ws) { return at<DynScales>(ws, kDynScalesOffset); }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ----------------------------------------------------------------- stages

GateArgs gate_args(const moe_problem_t& p, const float* logits, const float* bias, int32_t* ids,
                   float* w) {
  GateArgs a;
  a.logits = logits;
  a.bias = (p.scoring == MOE_SCORE_SIGMOID) ? bias : nullptr;
  a.ids = ids;
  a.w = w;
  a.T = p.T;
  a.E = p.E;
  a.k = p.top_k;
  a.sigmoid = p.scoring == MOE_SCORE_SIGMOID;
  a.renormalize = p.renormalize;
  a.n_group = p.n_group;
  a.topk_group = p.topk_group;
  a.scale = p.routed_scaling_factor;
  return a;
}

moe_status_t run_gate(const moe_problem_t& p, const float* logits, const float* bias, int32_t* ids,
                      float* w, cudaStream_t s) {
  return cuda_status(launch_gate(gate_args(p, logits, bias, ids, w), s));
}

AlignArgs align_args(const moe_problem_t& p, const int32_t* ids, const void* x, const float* a1,
                     int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                     void* ws) {
  const Layout L = layout_of(p);
  AlignArgs a;
  a.ids = ids;
  a.S = p.T * p.top_k;
  a.E = p.E;
  a.k = p.top_k;
  a.H = p.H;
  a.block_counts = at<int32_t>(ws, L.align_counts);
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.x = x;
  a.x_perm = x_perm;
  a.a1 = a1;
  a.fp8 = p.wdtype == MOE_W_FP8_E4M3;
  a.err = at<uint32_t>(ws, L.hdr);
  return a;
}

moe_status_t run_align(const moe_problem_t& p, const int32_t* ids, const void* x, const float* a1,
                       int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                       void* x_perm, void* ws, cudaStream_t s) {
  return cuda_status(
      launch_align(align_args(p, ids, x, a1, counts, offsets, perm, inv, x_perm, ws), s));
}

// Split-K partials of the down GEMM left for the caller's reduce to finish.
struct DeferredFinish {
  const float* part = nullptr;
  int P = 1;
  int64_t pstride = 0;
};

moe_status_t run_gemm(const moe_problem_t& p, const moe_weights_t& wt, bool up, const void* in,
                      const int32_t* offsets, void* out, void* ws, cudaStream_t s,
                      DeferredFinish* defer = nullptr) {
  const int S = p.T * p.top_k;
  if (S == 0) return MOE_OK;
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
  const GemmPlan g = plan_gemm(p, up, di.sms);
  const Layout L = layout_of(p);
  const int wk = wkind_of(p);
  const uint64_t E = p.E, H = p.H, I = p.I;

  GemmMaps maps;
  // A: expert weights.
  bool ok;
  if (up) {
    // [E][2][I/16][16][K] viewed as dims (K, 16, 2, I/16, E): one box = 4 blocks
    // of 16 rows of gate followed by the 16 matching rows of up.
    const uint64_t Kb = (wk == kW_INT4) ? H / 2 : (wk == kW_BF16 ? H * 2 : H);  // bytes per row
    const uint64_t dimK = (wk == kW_BF16) ? H : Kb;
    uint64_t dims[5] = {dimK, 16, 2, I / 16, E};
    uint64_t str[4] = {Kb, I * Kb, 16 * Kb, 2 * I * Kb};
    // 128 bytes of each row per box: 64 bf16, 128 e4m3 / int8, or 256 int4 codes
    uint32_t box[5] = {wk == kW_BF16 ? 64u : 128u, 16, 2, 4, 1};
    ok = encode_map(&maps.a, wk == kW_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                    5, wt.w13, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t Kb = (wk == kW_INT4) ? I / 2 : (wk == kW_BF16 ? I * 2 : I);
    const uint64_t dimK = (wk == kW_BF16) ? I : Kb;
    uint64_t dims[3] = {dimK, H, E};
    uint64_t str[2] = {Kb, H * Kb};
    uint32_t box[3] = {wk == kW_BF16 ? 64u : 128u, 128, 1};
    ok = encode_map(&maps.a, wk == kW_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                    3, wt.w2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return MOE_ERR_CUDA;
  {
    // B: permuted token rows [S, K] (bf16, or e4m3 for the fp8 path), three box heights.
    const uint64_t K = up ? H : I;
    const bool f8 = wk == kW_FP8;
    uint64_t dims[2] = {K, static_cast<uint64_t>(S)};
    uint64_t str[1] = {K * (f8 ? 1 : 2)};
    const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap* dst[3] = {&maps.b, &maps.b64, &maps.b16};
    const uint32_t rows[3] = {static_cast<uint32_t>(g.pair ? g.bn_max / 2 : g.bn_max), 64u, 16u};
    for (int i = 0; i < 3; ++i) {
      uint32_t box[2] = {f8 ? 128u : 64u, rows[i]};
      if (!encode_map(dst[i], dt, 2, in, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MOE_ERR_CUDA;
    }
    if (converts(wk)) {
      // full tiles: the token rows of 4 consecutive k-blocks in one box, viewed
      // as [K/64][S][64] so each k-block lands as its own 128-byte-swizzled tile
      uint64_t d3[3] = {64, static_cast<uint64_t>(S), K / 64};
      uint64_t s3[2] = {K * 2, 128};
      uint32_t b3[3] = {64, static_cast<uint32_t>(g.pair ? g.bn_max / 2 : g.bn_max), 4};
      if (!encode_map(&maps.b, dt, 3, in, d3, s3, b3, CU_TENSOR_MAP_SWIZZLE_128B)) return MOE_ERR_CUDA;
    }
  }

  GemmParams gp;
  gp.offsets = offsets;
  gp.err = at<uint32_t>(ws, L.hdr);
  const bool dyn = dynamic_scales(p);
  DynScales* ds = dyn_of(ws);
  // dynamic scales: a1 comes from the align stage, a2 from this gate_up call,
  // whose GEMM then writes bf16 to scratch for a separate quantisation pass
  const float* a1 = dyn ? &ds->scale[0] : wt.a1_scale;
  const float* a2 = dyn ? &ds->scale[1] : wt.a2_scale;
  void* const final_out = out;
  if (dyn && up) out = at<void>(ws, L.act_bf16);
  gp.a_scale = up ? a1 : a2;
  gp.w_scale = static_cast<const float*>(up ? wt.w13_scale : wt.w2_scale);
  gp.q_scale = dyn ? nullptr : wt.a2_scale;
  gp.amax = (dyn && up) ? &ds->amax[1] : nullptr;
  gp.w4_scale = up ? wt.w13_scale : wt.w2_scale;
  gp.w4_zero = static_cast<const uint8_t*>(up ? wt.w13_zero : wt.w2_zero);
  gp.w4_paired = p.wdtype == MOE_W_INT4_G128_PAIRED ? 1 : 0;
  gp.E = p.E;
  gp.S = S;
  gp.I = p.I;
  gp.FB = g.pair ? g.FB / 2 : g.FB;
  gp.pair = g.pair;
  {
    // weights are streamed (read once) when one token tile is expected to hold
    // all of an expert's rows; otherwise several tiles reuse them through L2
    const long long Sl = static_cast<long long>(p.T) * p.top_k;
    const long long touched = std::max(1ll, std::min<long long>(p.E, Sl));
    const long long m_avg = (Sl + touched - 1) / touched;
    gp.w_stream = (m_avg <= g.bn_max) ? 1 : 0;
    const int ws_env = knob(current_tuning().w_stream, -1);
    if (ws_env == 0 || ws_env == 1) gp.w_stream = ws_env;
  }
  // work-unit order: experts with more than one token tile interleaved with the
  // others whenever both kinds occur (decided on the device from the counts)
  gp.unit_order = knob(current_tuning().unit_order, 2);
  gp.KB = g.KB;
  gp.P = g.P;
  gp.bn_max = g.bn_max;
  gp.stages = g.stages;
  gp.astages = g.astages;
  gp.slot_kb = g.slot_kb;
  gp.conv_groups = g.conv_groups;
  gp.dual = g.dual;
  gp.acc_bufs = g.acc_bufs;
  gp.epi_warps = g.epi_warps;
  gp.ksplit = g.ksplit;
  gp.acc_cols = g.acc_cols;
  gp.full_box = g.full_box;
  gp.is_up = up ? 1 : 0;
  gp.R = up ? 2 * p.I : p.H;
  gp.G = up ? p.H / 128 : p.I / 128;
  float* part = at<float>(ws, L.partial);
  {
    const size_t N = up ? 2 * static_cast<size_t>(p.I) : static_cast<size_t>(p.H);
    const size_t need = static_cast<size_t>(g.P) * S * N * sizeof(float);
    if (g.P > 1 && need > L.scratch_end - L.partial) return MOE_ERR_UNSUPPORTED;  // plan/size mismatch
  }
  if (g.P == 1) {
    gp.epi = up ? kEpiSwiglu : kEpiStore;
    gp.out = out;
    gp.out_ld = up ? p.I : p.H;
    gp.part_stride = 0;
  } else {
    gp.epi = kEpiPartial;
    gp.out = part;
    gp.out_ld = up ? 2 * static_cast<int64_t>(p.I) : p.H;
    gp.part_stride = static_cast<int64_t>(S) * gp.out_ld;
  }
  cudaError_t err = launch_grouped_gemm(wk, maps, gp, di.sms, g.smem, s);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  if (g.P > 1) {
    if (up) {
      err = launch_swiglu_finish(part, g.P, gp.part_stride, S, p.I, wt.a2_scale, wk == kW_FP8 && !dyn, out,
                                 gp.amax, s);
    } else if (defer != nullptr) {
      defer->part = part;  // the caller folds the slice sum into its reduce
      defer->P = g.P;
      defer->pstride = gp.part_stride;
    } else {
      err = launch_down_finish(part, g.P, gp.part_stride, S, p.H, out, s);
    }
  }
  if (err == cudaSuccess && dyn && up)
    err = launch_quantize_e4m3_dynamic(out, static_cast<int64_t>(S) * p.I, ds, 1, final_out, s);
  return cuda_status(err);
}

moe_status_t check_weights(const moe_problem_t& p, const moe_weights_t* w) {
  if (w == nullptr || w->w13 == nullptr || w->w2 == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned(w->w13, 16) || !aligned(w->w2, 16)) return MOE_ERR_INVALID_ARG;
  if (p.wdtype == MOE_W_FP8_E4M3) {
    if (!w->w13_scale || !w->w2_scale) return MOE_ERR_INVALID_ARG;
    // static: both activation scales given; dynamic: both computed, none given
    const bool given = w->a1_scale && w->a2_scale, none = !w->a1_scale && !w->a2_scale;
    if (dynamic_scales(p) ? !none : !given) return MOE_ERR_INVALID_ARG;
  }
  if (converts(wkind_of(p))) {
    if (!w->w13_scale || !w->w2_scale || !aligned(w->w13_scale, 2) || !aligned(w->w2_scale, 2))
      return MOE_ERR_INVALID_ARG;
    if ((w->w13_zero == nullptr) != (w->w2_zero == nullptr)) return MOE_ERR_INVALID_ARG;
  } else if (w->w13_zero || w->w2_zero) {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status_t check_ws(const moe_problem_t& p, void* ws, size_t ws_bytes, bool full) {
  if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  const Layout L = layout_of(p);
  if (ws_bytes < (full ? L.total : L.scratch_end)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define MOE_TRY(x)                       \
  do {                                   \
    const moe_status_t st__ = (x);       \
    if (st__ != MOE_OK) return st__;     \
  } while (0)

}  // namespace

extern "C" {

size_t moe_scratch_size(const moe_problem_t* p) {
  if (validate_problem(p) != MOE_OK) return 0;
  return layout_of(*p).scratch_end;
}

size_t moe_workspace_size(const moe_problem_t* p) {
  if (validate_problem(p) != MOE_OK) return 0;
  return layout_of(*p).total;
}

size_t moe_padded_capacity(const moe_problem_t* p, int32_t block) {
  if (validate_problem(p) != MOE_OK || block < 1) return 0;
  const size_t S = static_cast<size_t>(p->T) * p->top_k;
  const size_t cap = S + static_cast<size_t>(p->E) * (block - 1);
  return (cap + block - 1) / block * block;
}

moe_status_t moe_gate_topk(const moe_problem_t* p, const float* logits, const float* bias,
                           int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  if (p->T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w || !aligned(logits, 4) || !aligned(topk_ids, 4) ||
      !aligned(topk_w, 4) || (bias && !aligned(bias, 4)))
    return MOE_ERR_INVALID_ARG;
  return run_gate(*p, logits, bias, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_align_permute(const moe_problem_t* p, const int32_t* topk_ids, const void* x,
                               const float* a1_scale, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv, void* x_perm, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  MOE_TRY(check_ws(*p, ws, ws_bytes, false));
  if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4)) return MOE_ERR_INVALID_ARG;
  if (p->T > 0) {
    if (!topk_ids || !x || !perm || !inv || !x_perm || !aligned(x, 16) || !aligned(x_perm, 16) ||
        !aligned(perm, 4) || !aligned(inv, 4) || !aligned(topk_ids, 4))
      return MOE_ERR_INVALID_ARG;
    if (p->wdtype == MOE_W_FP8_E4M3 && !dynamic_scales(*p) && !a1_scale) return MOE_ERR_INVALID_ARG;
  }
  if (dynamic_scales(*p) && a1_scale) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dynamic_scales(*p) && p->T > 0) {
    MOE_TRY(cuda_status(launch_absmax_scale(x, static_cast<int64_t>(p->T) * p->H, dyn_of(ws), 0, s)));
    a1_scale = &dyn_of(ws)->scale[0];
  }
  return run_align(*p, topk_ids, x, a1_scale, counts, offsets, perm, inv, x_perm, ws, s);
}

moe_status_t moe_align_block_size(const moe_problem_t* p, const int32_t* offsets,
                                  const int32_t* perm, int32_t block, int32_t* sorted_ids,
                                  int32_t* block_expert, int32_t* total_padded,
                                  moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  if (block < 1 || block > 1024) return MOE_ERR_INVALID_ARG;
  if (!offsets || !total_padded || !sorted_ids || !block_expert) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && !perm) return MOE_ERR_INVALID_ARG;
  const size_t cap = moe_padded_capacity(p, block);
  return cuda_status(launch_align_block_size(offsets, perm, p->E, p->T * p->top_k, block, cap,
                                             sorted_ids, block_expert, total_padded,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_gemm_swiglu(const moe_problem_t* p, const moe_weights_t* w,
                                     const void* x_perm, const int32_t* offsets, void* act,
                                     void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  MOE_TRY(check_weights(*p, w));
  MOE_TRY(check_ws(*p, ws, ws_bytes, false));
  if (p->T == 0) return MOE_OK;
  if (!x_perm || !offsets || !act || !aligned(x_perm, 16) || !aligned(act, 16) || !aligned(offsets, 4))
    return MOE_ERR_INVALID_ARG;
  return run_gemm(*p, *w, true, x_perm, offsets, act, ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_gemm_down(const moe_problem_t* p, const moe_weights_t* w,
                                   const void* act, const int32_t* offsets, void* y_perm,
                                   void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  MOE_TRY(check_weights(*p, w));
  MOE_TRY(check_ws(*p, ws, ws_bytes, false));
  if (p->T == 0) return MOE_OK;
  if (!act || !offsets || !y_perm || !aligned(act, 16) || !aligned(y_perm, 16) || !aligned(offsets, 4))
    return MOE_ERR_INVALID_ARG;
  return run_gemm(*p, *w, false, act, offsets, y_perm, ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_unpermute_reduce(const moe_problem_t* p, const void* y_perm, const int32_t* inv,
                                  const float* topk_w, void* out, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  MOE_TRY(check_ws(*p, ws, ws_bytes, false));
  if (p->T == 0) return MOE_OK;
  if (!y_perm || !inv || !topk_w || !out || !aligned(y_perm, 16) || !aligned(out, 16) ||
      !aligned(inv, 4) || !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_unpermute_reduce(y_perm, inv, topk_w, p->T, p->H, p->top_k, out,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_forward(const moe_problem_t* p, const moe_weights_t* w, const void* x,
                         const float* logits, const float* bias, void* out, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(validate_problem(p));
  MOE_TRY(check_weights(*p, w));
  MOE_TRY(check_ws(*p, ws, ws_bytes, true));
  if (p->T == 0) return MOE_OK;
  if (!x || !logits || !out || !aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4) ||
      (bias && !aligned(bias, 4)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Layout L = layout_of(*p);
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* tw = at<float>(ws, L.w);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm = at<int32_t>(ws, L.perm);
  int32_t* inv = at<int32_t>(ws, L.inv);
  void* x_perm = at<void>(ws, L.x_perm);
  void* act = at<void>(ws, L.act);
  void* y_perm = at<void>(ws, L.y_perm);
  const float* a1 = w->a1_scale;
  if (dynamic_scales(*p)) {
    MOE_TRY(cuda_status(launch_absmax_scale(x, static_cast<int64_t>(p->T) * p->H, dyn_of(ws), 0, s)));
    a1 = &dyn_of(ws)->scale[0];
  }
  if (p->T * p->top_k <= kRouteMaxSlots) {
    // small batch: gate, histogram, offsets, permutation and row gather in one
    // kernel (results identical to the path below)
    const AlignArgs aa = align_args(*p, ids, x, a1, counts, offsets, perm, inv, x_perm, ws);
    MOE_TRY(cuda_status(launch_route_small(gate_args(*p, logits, bias, ids, tw), aa, s)));
  } else {
    MOE_TRY(run_gate(*p, logits, bias, ids, tw, s));
    MOE_TRY(run_align(*p, ids, x, a1, counts, offsets, perm, inv, x_perm, ws, s));
  }
  MOE_TRY(run_gemm(*p, *w, true, x_perm, offsets, act, ws, s));
  DeferredFinish df;
  MOE_TRY(run_gemm(*p, *w, false, act, offsets, y_perm, ws, s, &df));
  if (df.part != nullptr)
    return cuda_status(launch_unpermute_reduce_splitk(df.part, df.P, df.pstride, inv, tw, p->T, p->H,
                                                      p->top_k, out, s));
  return cuda_status(launch_unpermute_reduce(y_perm, inv, tw, p->T, p->H, p->top_k, out, s));
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_repack_int4(const void* codes, void* out, size_t n_bytes, moe_stream_t stream) {
  if (n_bytes == 0) return MOE_OK;
  if (codes == nullptr || out == nullptr || n_bytes % 4 != 0 || reinterpret_cast<uintptr_t>(codes) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return MOE_ERR_INVALID_ARG;
  const cudaError_t e = launch_repack_int4(static_cast<const uint32_t*>(codes), static_cast<uint32_t*>(out),
                                           n_bytes / 4, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

float* moe_dynamic_scales(void* ws) {
  if (ws == nullptr || !aligned(ws, 256)) return nullptr;
  return dyn_of(ws)->scale;
}

moe_status_t moe_get_device_error(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t h[2] = {0, 0};
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (h[0] != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(h), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return static_cast<moe_status_t>(h[0]);
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported problem";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE_BAD_INDEX: return "expert id outside [0, E) seen on the device";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

moe_status_t moe_get_plan_for_sms(const moe_problem_t* p, int32_t num_sms, moe_plan_t* plan) {
  MOE_TRY(validate_problem(p));
  if (plan == nullptr || num_sms < 1) return MOE_ERR_INVALID_ARG;
  const GemmPlan u = plan_gemm(*p, true, num_sms);
  const GemmPlan d = plan_gemm(*p, false, num_sms);
  plan->bn_max_up = u.bn_max;
  plan->splits_up = u.P;
  plan->stages_up = u.stages;
  plan->astages_up = u.astages;
  plan->smem_up = static_cast<int32_t>(u.smem);
  plan->bn_max_down = d.bn_max;
  plan->splits_down = d.P;
  plan->stages_down = d.stages;
  plan->astages_down = d.astages;
  plan->smem_down = static_cast<int32_t>(d.smem);
  plan->num_sms = num_sms;
  plan->slot_kb_up = u.slot_kb;
  plan->slot_kb_down = d.slot_kb;
  plan->pair_up = u.pair;
  plan->pair_down = d.pair;
  plan->issuers_up = u.dual ? 2 : 1;
  plan->issuers_down = d.dual ? 2 : 1;
  plan->conv_groups_up = u.conv_groups;
  plan->conv_groups_down = d.conv_groups;
  plan->epi_warps_up = u.epi_warps;
  plan->epi_warps_down = d.epi_warps;
  plan->acc_bufs_up = u.acc_bufs;
  plan->acc_bufs_down = d.acc_bufs;
  return MOE_OK;
}

moe_status_t moe_set_tuning(const moe_tuning_t* t) {
  moe_tuning_t v = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
  if (t != nullptr) {
    v = *t;
    auto ok = [](int32_t x, int32_t lo, int32_t hi) { return x == -1 || (x >= lo && x <= hi); };
    if (!ok(v.bn_max, 16, 256) || (v.bn_max > 0 && v.bn_max % 16 != 0) || !ok(v.stages, 2, kMaxStages) ||
        !ok(v.splits, 1, kMaxSplits) || !ok(v.pair, 0, 1) || !ok(v.conv_groups, 2, 3) ||
        !(v.slot_kb == -1 || v.slot_kb == 2 || v.slot_kb == 4) || !ok(v.ksplit, 0, 1) || !ok(v.dual, 0, 1) ||
        !ok(v.full_box, 0, 1) || !ok(v.w_stream, 0, 1) || !ok(v.unit_order, 0, 2) ||
        !(v.epi_warps == -1 || v.epi_warps == 4 || v.epi_warps == 8) || !ok(v.acc_bufs, 1, 2))
      return MOE_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  g_tuning = v;
  return MOE_OK;
}

moe_status_t moe_get_plan(const moe_problem_t* p, moe_plan_t* plan) {
  MOE_TRY(validate_problem(p));
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_get_plan_for_sms(p, di.sms, plan);
}

}  // extern "C"
