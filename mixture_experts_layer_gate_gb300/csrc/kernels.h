// Internal launchers of the MoE kernels (host side).  The C ABI in api.cu
// validates arguments and lays out the workspace; these functions only launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

#ifdef MOE_GB300_H
// Problem checks shared by every entry point: MOE_OK, MOE_ERR_INVALID_ARG for a
// malformed problem, MOE_ERR_UNSUPPORTED for one beyond the library's limits.
moe_status_t validate_problem(const moe_problem_t* p);
#endif

// ------------------------------------------------------------------- gate
struct GateArgs {
  const float* logits;  // [T, E]
  const float* bias;    // [E] or null
  int32_t* ids;         // [T, k]
  float* w;             // [T, k]
  int T, E, k;
  int sigmoid;          // 0 softmax, 1 sigmoid
  int renormalize;
  int n_group, topk_group;
  float scale;
};
cudaError_t launch_gate(const GateArgs& a, cudaStream_t s);

// ------------------------------------------------------------------ align
constexpr int kAlignSlotsPerCta = 1024;
inline int align_blocks(int S) { return (S + kAlignSlotsPerCta - 1) / kAlignSlotsPerCta; }

struct AlignArgs {
  const int32_t* ids;     // [S]
  int S, E, k, H;
  int32_t* block_counts;  // [nblk, E] scratch
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E + 1]
  int32_t* perm;          // [S]
  int32_t* inv;           // [S]
  const void* x;          // [T, H] bf16
  void* x_perm;           // [S, H] bf16 or e4m3
  const float* a1;        // fp8: [1]
  int fp8;
  uint32_t* err;
};
cudaError_t launch_align(const AlignArgs& a, cudaStream_t s);
// x_perm rows only (perm must be ready).
cudaError_t launch_gather(const AlignArgs& a, cudaStream_t s);

// Gate + histogram + offsets + stable permutation + row gather in one kernel,
// for batches of at most kRouteMaxSlots (token, expert) slots; ids / w /
// counts / offsets / perm / inv / x_perm are bit-identical to launch_gate
// followed by launch_align.
constexpr int kRouteMaxSlots = 1024;
cudaError_t launch_route_small(const GateArgs& g, const AlignArgs& a, cudaStream_t s);

cudaError_t launch_align_block_size(const int32_t* offsets, const int32_t* perm, int E, int S,
                                    int block, size_t capacity, int32_t* sorted_ids,
                                    int32_t* block_expert, int32_t* total, cudaStream_t s);

// ----------------------------------------------------------------- reduce
cudaError_t launch_unpermute_reduce(const void* y_perm, const int32_t* inv, const float* w,
                                    int T, int H, int k, void* out, cudaStream_t s);

// Split-K finishing passes (fixed summation order over the P slices).
// amax: dynamic fp8 scales only (bf16 act): running max of the stored |act| bits, else null.
cudaError_t launch_swiglu_finish(const float* part, int P, int64_t pstride, int S, int I,
                                 const float* a2, int fp8, void* act, uint32_t* amax, cudaStream_t s);
cudaError_t launch_down_finish(const float* part, int P, int64_t pstride, int S, int H,
                               void* y, cudaStream_t s);
// down_finish + unpermute_reduce in one pass, bit-identical to the pair.
cudaError_t launch_unpermute_reduce_splitk(const float* part, int P, int64_t pstride, const int32_t* inv,
                                           const float* w, int T, int H, int k, void* out, cudaStream_t s);

// ------------------------------------------------- dynamic fp8 scales
// Words in the workspace header (byte kDynScalesOffset) for dynamic per-tensor
// activation scales; index 0 = a1 (token rows), 1 = a2 (SwiGLU output).  amax
// and ticket are zero between calls (the last CTA of each pass clears them).
struct DynScales {
  uint32_t amax[2];    // largest bf16 magnitude bits seen so far
  uint32_t ticket[2];  // CTAs finished
  float scale[2];      // amax / 448 (1 for an all-zero tensor)
};
constexpr size_t kDynScalesOffset = 64;
// scale[which] = max |x[0..n)| / 448 over bf16 x (n a multiple of 8).
cudaError_t launch_absmax_scale(const void* x, int64_t n, DynScales* d, int which, cudaStream_t s);
// out[i] = e4m3(x[i] / s) (round to nearest even, saturating), n a multiple of 8, with
// s = amax[which] / 448 from the bits a producer folded in; the last CTA stores s in
// scale[which] and clears amax and ticket.
cudaError_t launch_quantize_e4m3_dynamic(const void* x, int64_t n, DynScales* d, int which, void* out,
                                         cudaStream_t s);

// ------------------------------------------------------------ grouped GEMM
// int4 / int8: k-blocks (64 reduction elements each) per operand ring stage.
constexpr int kInt4StageKb = 4;

enum WKind : int { kW_BF16 = 0, kW_FP8 = 1, kW_INT4 = 2, kW_INT8 = 3 };

// int4 / int8 weights are turned into bf16 by converter warps before the MMA.
__host__ __device__ constexpr bool converts(int wk) { return wk == kW_INT4 || wk == kW_INT8; }
// Packed weight codes per ring stage: 128 rows x kInt4StageKb k-blocks.
__host__ __device__ constexpr int raw_stage_bytes(int wk) {
  return wk == kW_INT8 ? 128 * kInt4StageKb * 64 : 128 * kInt4StageKb * 32;
}
enum EpiKind : int { kEpiSwiglu = 0, kEpiStore = 1, kEpiPartial = 2 };

struct GemmParams {
  const int32_t* offsets;  // [E + 1]
  uint32_t* err;
  void* out;
  const float* a_scale;    // fp8: activation scale of the B operand (a1 or a2)
  const float* w_scale;    // fp8: per-expert weight scale [E]
  const float* q_scale;    // fp8 gate_up: a2, the scale `act` is quantised with (null: store bf16)
  uint32_t* amax;          // dynamic fp8 gate_up: running max of the stored |bf16 act| bits, or null
  const void* w4_scale;    // int4 / int8: half [E, R, G]
  const uint8_t* w4_zero;  // int4 / int8: uint8 [E, R, G] zero points (unsigned codes), or null (signed)
  int w4_paired;           // int4: codes in the paired order of moe_repack_int4 (else the packed order)
  int64_t out_ld;          // elements per output row
  int64_t part_stride;     // elements between split-K slices
  int E, S, I;
  int FB;                  // feature blocks (I/64 for gate_up, H/128 for down)
  int KB;                  // k blocks of the reduction
  int P;                   // split-K factor
  int bn_max;              // token tile limit: multiple of 16, <= 256
  int stages;              // operand ring depth (int4 / int8: ring of packed A + token tiles)
  int astages;             // int4 / int8 only: ring of converted bf16 A tiles
  int slot_kb;             // int4 / int8 only: k-blocks per converted tile (2 or 4)
  int full_box;            // 1: always load bn_max token rows, one box per stage (int4 / int8 default)
  int conv_groups;         // int4 / int8 only: converter warp groups (2, or 3 with CTA pairs)
  int ksplit;              // int4 / int8, 2 groups, whole-stage slots: both groups convert every
                           // stage, group g its k-blocks 2g and 2g + 1 (else groups alternate stages)
  int acc_cols;            // TMEM columns per accumulator buffer
  int pair;                // 1: CTA-pair kernel (FB counts 256-row weight blocks)
  int dual;                // int4 / int8, whole-stage slots: two MMA-issuing threads, each its half
                           // of every stage's k-blocks into its own partial accumulator
  int acc_bufs;            // accumulator buffers in TMEM (2; 1 with two issuers and > 64 columns)
  int epi_warps;           // epilogue warps: 4 (one per TMEM lane quarter) or 8 (two per quarter)
  int w_stream;            // 1: each weight tile is read once (evict it from L2 first)
  int unit_order;          // 0 expert-major, 1 weight-block-major, 2 heavy / light interleave
  int epi;                 // EpiKind
  int is_up;
  int R;                   // weight rows per expert (2I or H)
  int G;                   // int4 / int8 groups per weight row
};

struct GemmMaps {
  CUtensorMap a;    // weights: bf16/e4m3 tile of 128 rows x 128 B, or for int4 128 rows x
                    // 128 B of packed codes (4 k-blocks), for int8 128 rows x 128 B of codes
                    // (2 k-blocks, two boxes per ring stage); 128-byte swizzle
  CUtensorMap b;    // token rows (x_perm or act), box of bn_max rows: one load per full tile
                    // (int4 / int8: 3-D view [k-block][row][64], box of 4 k-blocks)
  CUtensorMap b64;  // the same rows, 64-row box (ragged last tile of an expert)
  CUtensorMap b16;  // the same rows, 16-row box (ragged last tile of an expert)
};

constexpr int kMaxEpiWarps = 8;
size_t gemm_smem_bytes(int wkind, int bn_max, int stages, int astages, int E, int epi_warps);
int gemm_threads(int wkind, int conv_groups, int dual, int epi_warps);
// whether a kernel with eight epilogue warps exists for this configuration
bool gemm_epi8_supported(int wkind, int conv_groups, int pair, int slot_kb);
cudaError_t launch_grouped_gemm(int wkind, const GemmMaps& maps, const GemmParams& p, int grid,
                                size_t smem, cudaStream_t s);

// int4 codes from the packed order (low nibble = even K index) to the paired
// order (per 4-byte word: even K indices in the low 16 bits, odd in the high).
cudaError_t launch_repack_int4(const uint32_t* in, uint32_t* out, size_t n_words, cudaStream_t s);

}  // namespace moe
