/*
 * moe.h - C ABI of a fused Mixture-of-Experts layer forward pass for GB300
 * (sm_103a).  One library, plain pointers and sizes, no framework types.
 *
 * The layer (prose of the pages; none prints a formula):
 *   1. gate: router logits -> top-k expert ids and weights
 *      ("Add deepseek_v3 fused gate", the fused gate and its PyTorch reference;
 *       softmax top-k as in Mixtral on "Optimized fused MoE Kernel, take 2").
 *   2. align + permute: group the T*k token slots by expert
 *      ("[Kernel] add triton fused moe kernel for gptq/awq", note 1 on
 *       moe_align_block_size; "Add deepseek_v3 fused gate", TensorRT-LLM's
 *       expand_and_permute, which needs no padding).
 *   3. grouped GEMMs per expert: gate_up, SiLU-and-mul, down
 *      (Triton fused_moe on "Optimized fused MoE Kernel, take 2"; split-K on
 *       "[kernel] introduce fused_moe_triton_splitk to sglang"; the FBGEMM
 *       grouped GEMM blog; weight formats bf16, fp8 e4m3 per-tensor, int4
 *       group-128 from those pages).
 *   4. unpermute + top-k weighted reduction ("Add deepseek_v3 fused gate",
 *      TensorRT-LLM's unpermute_and_reduce).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, row-major, 16-byte aligned,
 *     owned by the caller.  The library allocates nothing and keeps no state
 *     between calls other than per-device constants (SM count, driver entry
 *     point) looked up on first use and the planner overrides a caller sets
 *     with moe_set_tuning.
 *   - Every call is asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).  No call synchronises with
 *     the host except moe_get_device_error.  Calls can be captured in a CUDA
 *     graph.
 *   - Argument errors are reported synchronously by the return value and
 *     nothing is launched.  Data-dependent errors found by the kernels (an
 *     expert id outside [0, E), a pipeline wait that ran out) are recorded in
 *     a sticky error word at the start of the workspace and read with
 *     moe_get_device_error; the kernels then finish their bounded work with
 *     memory-safe (but meaningless) results.
 *   - A workspace `ws` of at least moe_scratch_size() bytes (stage calls) or
 *     moe_workspace_size() bytes (moe_forward) is passed to the calls that
 *     need one.  Its first 256 bytes are the error header and must be zero
 *     when the workspace is first used (allocate it zeroed once).
 *
 * Shapes: T tokens, H hidden, I intermediate per expert, E experts, k = top_k,
 * S = T*k slots.  Requirements: H % 128 == 0, I % 128 == 0, 1 <= k <= E <= 1024,
 * T >= 0; grouped gating needs n_group <= 32, E % n_group == 0,
 * 1 <= topk_group <= n_group and k <= topk_group * E / n_group.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,      /* bad shape, null or misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. E > 1024) */
  MOE_ERR_WORKSPACE = 3,        /* workspace missing or too small */
  MOE_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_BAD_INDEX = 5, /* a kernel saw an expert id outside [0, E) */
  MOE_ERR_TIMEOUT = 6           /* a kernel pipeline wait ran out (about 1 s) */
} moe_status_t;

typedef enum {
  MOE_W_BF16 = 0,
  MOE_W_FP8_E4M3 = 1,
  MOE_W_INT4_G128 = 2,
  MOE_W_INT8_G128 = 3,
  MOE_W_INT4_G128_PAIRED = 4 /* int4 codes prepared by moe_repack_int4 */
} moe_wdtype_t;
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;
/* fp8 activation scales ("[kernel] introduce fused_moe_triton_splitk to
 * sglang" and the FBGEMM grouped-GEMM blog run fp8 W8A8 with per-tensor
 * activation scales).  STATIC: the caller passes a1 (token rows) and a2
 * (SwiGLU output).  DYNAMIC: the library computes them per call as
 * max |v| / 448 over the whole tensor (a1 over the T x H input rows, a2 over
 * the S x I SwiGLU output as stored in bf16), then quantises v / scale; the
 * SwiGLU output goes through a bf16 scratch buffer and a separate pass. */
typedef enum { MOE_ACT_SCALE_STATIC = 0, MOE_ACT_SCALE_DYNAMIC = 1 } moe_act_scale_t;

/* Problem description.  Enum-valued fields are stored as int32_t so the
 * struct layout is fixed: 13 four-byte fields, no padding. */
typedef struct {
  int32_t T, H, I, E, top_k;
  int32_t scoring;               /* moe_score_t */
  int32_t renormalize;           /* 1: divide the k selected scores by their sum */
  int32_t n_group, topk_group;   /* 0, 0 = ungrouped selection */
  float routed_scaling_factor;   /* multiplies the final weights (1.0f = none) */
  int32_t wdtype;                /* moe_wdtype_t */
  int32_t group_size;            /* int4 / int8 only: must be 128 */
  int32_t act_scale;             /* moe_act_scale_t; DYNAMIC only with fp8 */
} moe_problem_t;

/* Expert weights (device pointers).
 *   bf16 : w13 bf16 [E, 2I, H], w2 bf16 [E, H, I]; scales NULL.
 *   fp8  : w13 uint8 e4m3 [E, 2I, H], w2 uint8 e4m3 [E, H, I];
 *          w13_scale, w2_scale float [E] (value = e4m3(code) * scale[e]);
 *          a1_scale, a2_scale: float [1] static activation scales for the
 *          token rows entering gate_up and the activation entering down;
 *          both NULL with MOE_ACT_SCALE_DYNAMIC (see moe_dynamic_scales).
 *   int4 : w13 uint8 [E, 2I, H/2], w2 uint8 [E, H, I/2], two codes per
 *          byte, the low nibble holding the even K index; w13_scale half
 *          [E, 2I, H/128], w2_scale half [E, H, I/128].  With w13_zero and
 *          w2_zero NULL the codes are signed two's complement and
 *          value = code * scale (symmetric).  With both set (uint8
 *          [E, 2I, H/128] and [E, H, I/128], one zero point 0..15 per group,
 *          the shape of the scales) the codes are unsigned 0..15 and
 *          value = (code - zero) * scale (asymmetric, AWQ-style).  Setting
 *          only one of the two is MOE_ERR_INVALID_ARG.
 *   int4 paired (MOE_W_INT4_G128_PAIRED): the int4 tensors, scales and zero
 *          points above, with the codes of every 4-byte word (8 consecutive K
 *          indices k0..k7 of one row) reordered by moe_repack_int4: k0, k2,
 *          k4, k6 in the nibbles of the low 16 bits and k1, k3, k5, k7 in
 *          those of the high 16 bits, lowest first.  Results are those of the
 *          same weights in the packed order; the converters need fewer
 *          integer instructions per code.
 *   int8 : w13 uint8 [E, 2I, H], w2 uint8 [E, H, I], one code per byte;
 *          scales and zero points exactly as for int4 (zero points 0..255).
 *          Without zero points a byte is a signed two's-complement code
 *          (value = code * scale); with them an unsigned code
 *          (value = (code - zero) * scale).  Int4 and int8 weights are
 *          turned into bf16 (code - zero) * scale, rounded once, before the
 *          bf16 tensor-core product; activations stay bf16 (W4A16 / W8A16).
 * Zero points must be NULL for bf16 and fp8.
 * In w13, rows [0, I) are the gate projection (SiLU applied) and rows
 * [I, 2I) the up projection. */
typedef struct {
  const void* w13;
  const void* w2;
  const void* w13_scale;
  const void* w2_scale;
  const float* a1_scale;
  const float* a2_scale;
  const void* w13_zero;
  const void* w2_zero;
} moe_weights_t;

/* Bytes of workspace the stage calls need (error header, align scratch,
 * split-K partial sums).  Depends only on the problem.  Returns 0 for an
 * invalid problem. */
size_t moe_scratch_size(const moe_problem_t* p);

/* Bytes of workspace moe_forward needs: moe_scratch_size() plus every
 * intermediate (ids, weights, counts, offsets, perm, inv, x_perm, act,
 * y_perm).  Returns 0 for an invalid problem. */
size_t moe_workspace_size(const moe_problem_t* p);

/* Stage 1: top-k gate ("Add deepseek_v3 fused gate"; reading of the
 * selection rule below, the pages name the gate but print no formula).
 *   logits   float [T, E]
 *   bias     float [E] or NULL (sigmoid only; steers selection, not weights)
 *   topk_ids int32 [T, k]  out: ids ordered by selection key, descending,
 *                           equal keys to the lower expert index
 *   topk_w   float [T, k]  out
 * Softmax: key = logit; weight = softmax probability over all E, divided by
 * the sum of the k selected if renormalize, times routed_scaling_factor.
 * Sigmoid: s = sigmoid(logit); key = s + bias (raw logit when ungrouped and
 * bias is NULL); with n_group > 0 the experts form n_group contiguous groups,
 * each scored by the sum of its two largest keys, and only the topk_group best
 * groups (ties to the lower group) compete; weight = s, renormalised if asked,
 * times routed_scaling_factor.  A NaN logit is read as -inf: softmax
 * probability 0 (left out of the normalising sum), sigmoid score 0, and the
 * key of a -inf logit (with a bias, the bias alone), so it ranks after every
 * finite logit of equal bias.  Each softmax row needs one finite logit.  If
 * renormalisation meets selected scores that are all zero (every selected
 * logit NaN), the token's weights are zero. */
moe_status_t moe_gate_topk(const moe_problem_t* p, const float* logits, const float* bias,
                           int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* Stage 2: align and permute ("[Kernel] add triton fused moe kernel for
 * gptq/awq", note 1, moe_align_block_size; "Add deepseek_v3 fused gate",
 * expand_and_permute).  A stable counting sort of the flat slots f = t*k + j.
 *   topk_ids int32 [T, k]
 *   x        bf16 [T, H] token rows
 *   a1_scale float [1] (fp8 with static scales; NULL otherwise: with dynamic
 *            scales this call computes a1 from x into the workspace)
 *   counts   int32 [E]      out: slots per expert
 *   offsets  int32 [E + 1]  out: exclusive prefix sum, offsets[E] = S
 *   perm     int32 [S]      out: row -> slot; the r-th slot (ascending f)
 *                                routed to e is row offsets[e] + r
 *   inv      int32 [S]      out: slot -> row
 *   x_perm   [S, H]         out: x[perm[r] / k]; bf16, or for fp8 the e4m3
 *                                code of x / a1 (float32 division, round to
 *                                nearest even, saturating at 448)
 * Ids outside [0, E) set MOE_ERR_DEVICE_BAD_INDEX and are treated as 0. */
moe_status_t moe_align_permute(const moe_problem_t* p, const int32_t* topk_ids, const void* x,
                               const float* a1_scale, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv, void* x_perm, void* ws,
                               size_t ws_bytes, moe_stream_t stream);

/* moe_align_permute without a workspace, for callers that are not allowed to
 * allocate device memory: for instance a host framework that hands out no
 * scratch buffer to a custom operator, or a serving loop that forbids
 * cudaMalloc after start-up because it synchronises the device.  The pages
 * have no counterpart: it is a packaging variant of stage 2 only.
 *   Arguments and results are those of moe_align_permute minus ws/ws_bytes,
 *   except that fp8 always needs a1_scale (with dynamic scales too: there is
 *   no workspace to compute a1 in).
 *   Its scratch (per-CTA expert histograms) is a fixed 256 KiB array in the
 *   library's device image, one per device that loads the library, held until
 *   the process exits.  Limit: ceil(T*k / 1024) * E <= 65536 (e.g. E = 256 up
 *   to T*k = 262144); larger problems return MOE_ERR_UNSUPPORTED and launch
 *   nothing.  No cudaMalloc/cudaFree or other allocation happens.
 *   The first call in each CUDA context (e.g. the first per device, in its
 *   primary context) looks up the array's device address with that context
 *   current and caches it for the context; make that first call before any
 *   stream capture.  A context created later (another context on the device,
 *   or the primary context again after a device reset) gets its own lookup on
 *   its first call; at most 64 contexts per process are served, later ones get
 *   MOE_ERR_CUDA.
 *   All calls share the one array: calls whose GPU work can overlap (e.g. on
 *   two unsynchronised streams) race; order them.  Expert ids outside [0, E)
 *   are still routed to expert 0 but are not reported (there is no error
 *   header). */
moe_status_t moe_align_permute_noalloc(const moe_problem_t* p, const int32_t* topk_ids,
                                       const void* x, const float* a1_scale, int32_t* counts,
                                       int32_t* offsets, int32_t* perm, int32_t* inv,
                                       void* x_perm, moe_stream_t stream);

/* Padded view of the sorted slots for a GEMM row block of `block` rows (the
 * layout moe_align_block_size produces, "[Kernel] add triton fused moe kernel
 * for gptq/awq", note 1).  Each expert's segment is padded up to a multiple of
 * `block` with the sentinel S.
 *   offsets      int32 [E + 1], perm int32 [S]   (from moe_align_permute)
 *   sorted_ids   int32 [moe_padded_capacity(p, block)]             out
 *   block_expert int32 [moe_padded_capacity(p, block) / block]    out
 *   total_padded int32 [1]                                         out
 * Entries past total_padded are left untouched.  1 <= block <= 1024. */
moe_status_t moe_align_block_size(const moe_problem_t* p, const int32_t* offsets,
                                  const int32_t* perm, int32_t block, int32_t* sorted_ids,
                                  int32_t* block_expert, int32_t* total_padded,
                                  moe_stream_t stream);

/* Upper bound on total_padded: S + E * (block - 1), rounded up to a multiple
 * of block. */
size_t moe_padded_capacity(const moe_problem_t* p, int32_t block);

/* Stage 3a: grouped gate_up GEMM with SiLU-and-mul fused into its epilogue.
 * For every expert e and row r in [offsets[e], offsets[e+1]):
 *   h = W13[e] x_perm[r]  (fp32 accumulation; fp8: times a1 * w13_scale[e];
 *                          int4 / int8: weights (code - zero) * scale, each
 *                          rounded to bf16)
 *   act[r, i] = silu(h[i]) * h[I + i],  silu(z) = z / (1 + exp(-z))
 * act is bf16 [S, I], or for fp8 the e4m3 code of act / a2 (a2 static, or with
 * dynamic scales computed here from the bf16 act over all S rows).
 * Uses ws for split-K partial sums when the expert row counts are small.
 * offsets need not come from moe_align_permute: any nondecreasing int32
 * [E + 1] with offsets[0] = 0 and offsets[E] = S works, e.g. rows an
 * expert-parallel dispatch delivered for a rank's E local experts (then set
 * T = rows received and top_k = 1 in p).  Same for moe_grouped_gemm_down. */
moe_status_t moe_grouped_gemm_swiglu(const moe_problem_t* p, const moe_weights_t* w,
                                     const void* x_perm, const int32_t* offsets, void* act,
                                     void* ws, size_t ws_bytes, moe_stream_t stream);

/* Stage 3b: grouped down GEMM: y_perm[r] = W2[e] act[r] for rows of expert e
 * (fp8: times a2 * w2_scale[e]).  y_perm is bf16 [S, H].  Small row counts
 * split K across CTAs into fp32 partials in ws, summed in a fixed order
 * (no atomics; the result does not depend on scheduling). */
moe_status_t moe_grouped_gemm_down(const moe_problem_t* p, const moe_weights_t* w,
                                   const void* act, const int32_t* offsets, void* y_perm,
                                   void* ws, size_t ws_bytes, moe_stream_t stream);

/* Stage 4: unpermute and reduce ("Add deepseek_v3 fused gate",
 * unpermute_and_reduce):
 *   out[t] = sum_{j=0..k-1} topk_w[t, j] * y_perm[inv[t*k + j]]
 * accumulated in fp32 in j order (deterministic), stored bf16 [T, H]. */
moe_status_t moe_unpermute_reduce(const moe_problem_t* p, const void* y_perm, const int32_t* inv,
                                  const float* topk_w, void* out, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* The whole layer: gate, align/permute, gate_up+SwiGLU, down, unpermute and
 * reduce, all on `stream`, intermediates in ws (moe_workspace_size bytes).
 *   x bf16 [T, H], logits float [T, E], bias float [E] or NULL, out bf16 [T, H]. */
moe_status_t moe_forward(const moe_problem_t* p, const moe_weights_t* w, const void* x,
                         const float* logits, const float* bias, void* out, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* Kernel launches the library has issued in this process so far, counting
 * launches recorded into a CUDA graph once (at capture); for measurement, e.g.
 * the launches of one moe_forward = the count's change across one call. */
uint64_t moe_launch_count(void);

/* Weight preparation for int4 ("[Kernel] add triton fused moe kernel for
 * gptq/awq" streams group-quantised int4 codes packed two per byte; Marlin
 * reorders such codes once at load time for its own kernel).  Rewrites
 * n_bytes of int4 codes in the packed order (two codes per byte, the low
 * nibble holding the even K index: w13 or w2 of MOE_W_INT4_G128) into the
 * order of MOE_W_INT4_G128_PAIRED, a permutation inside every 4-byte word.
 * codes and out are device pointers, 4-byte aligned, either equal (in place)
 * or not overlapping at all (a partial overlap races); n_bytes is a multiple
 * of 4 (any int4 w13 / w2 tensor is).  Scales
 * and zero points are not touched.  Asynchronous on `stream`.  Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned pointer or a size that is not
 * a multiple of 4, MOE_OK for n_bytes == 0. */
moe_status_t moe_repack_int4(const void* codes, void* out, size_t n_bytes, moe_stream_t stream);

/* Dynamic fp8 scales (MOE_ACT_SCALE_DYNAMIC): device pointer to float [2]
 * inside the workspace ws, {a1, a2}.  moe_align_permute / moe_forward write
 * a1, moe_grouped_gemm_swiglu reads a1 and writes a2, moe_grouped_gemm_down
 * reads a2.  A caller that feeds the GEMMs with rows it quantised itself (an
 * expert-parallel dispatch) stores its a1 there before the gate_up call.
 * No work is launched; NULL for a NULL or misaligned ws. */
float* moe_dynamic_scales(void* ws);

/* Synchronises `stream`, returns the sticky device error recorded in ws (MOE_OK
 * if none) and clears it.  Debug/test use: it is the only blocking call. */
moe_status_t moe_get_device_error(void* ws, moe_stream_t stream);

/* Static, human-readable name of a status. */
const char* moe_status_string(moe_status_t s);

/* Launch plan the library makes for a problem (for tests and benchmarks): per
 * GEMM the token tile limit, split-K factor, operand ring depth, converted
 * weight ring depth (int4 / int8 only, else 0) and dynamic shared memory
 * bytes; then the SM count planned for; for int4 / int8 the k-blocks (64
 * reduction elements each) per converted weight slot in tensor memory (else
 * 0); per GEMM whether it runs as clusters of two CTAs sharing M = 256
 * MMAs (1) or one CTA per 128 weight rows (0); and per GEMM the threads that
 * issue its MMAs in a CTA (1, or for int4 / int8 tiles of at most 64 tokens
 * on one CTA 2, each its half of the reduction into its own accumulator); for
 * int4 / int8 the converter warp groups (2 or 3) per GEMM; per GEMM the warps
 * that drain its accumulators (4, or 8 taking alternate 32-token columns) and
 * the accumulator buffers in tensor memory (2 let a unit's epilogue overlap the
 * next unit's MMAs; 1 where the tile leaves no room for a second). */
typedef struct {
  int32_t bn_max_up, splits_up, stages_up, astages_up, smem_up;
  int32_t bn_max_down, splits_down, stages_down, astages_down, smem_down;
  int32_t num_sms;
  int32_t slot_kb_up, slot_kb_down;
  int32_t pair_up, pair_down;
  int32_t issuers_up, issuers_down;
  int32_t conv_groups_up, conv_groups_down;  /* int4 / int8: converter warp groups (else 0) */
  int32_t epi_warps_up, epi_warps_down;      /* epilogue warps per CTA (4 or 8) */
  int32_t acc_bufs_up, acc_bufs_down;        /* accumulator buffers (1 or 2) */
} moe_plan_t;

/* Planner overrides, for tests and benchmarks that want a kernel variant the
 * planner would not pick for a problem (results stay within the same
 * tolerances; only speed changes).  Each field is -1 for the planner's own
 * choice:
 *   bn_max      token tile limit, a multiple of 16 in [16, 256] (int4 / int8
 *               above 128 only on CTA pairs)
 *   stages      operand ring depth, 2..8 (only ever lowers the planner's)
 *   splits      split-K factor, 1..16 (at most K / 256; a workspace sized for
 *               fewer slices makes the GEMM call return MOE_ERR_UNSUPPORTED)
 *   pair        1: clusters of two CTAs sharing M = 256 MMAs, 0: one CTA per
 *               128 weight rows (pairs need an even number of weight blocks)
 *   conv_groups int4 with CTA pairs and one MMA issuer: 3 converter warp groups
 *   slot_kb     int4 / int8: k-blocks per converted weight slot, 2 or 4
 *   ksplit      int4 / int8: 1 = both converter groups convert every stage
 *   dual        int4 / int8: 1 = two MMA-issuing threads, 0 = one
 *   full_box    1 = every token tile loaded as one box of the full tile
 *               height (rows past the tile are loaded and not used), 0 = 64-
 *               and 16-row boxes for an expert's ragged last tile
 *   w_stream    1 = weights loaded with the L2 evict-first policy, 0 = normal
 *   unit_order  0 = GEMM work units expert by expert, 1 = weight block by
 *               weight block across experts, 2 = experts with more than one
 *               token tile interleaved with the others in proportion
 *   epi_warps   4 or 8 warps draining the accumulators (8: bf16 / fp8, and
 *               int4 / int8 on CTA pairs with two converter groups and
 *               four-k-block slots; elsewhere 4 is kept)
 *   acc_bufs    int4 / int8 tiles of 129-192 tokens: 2 = two accumulator
 *               buffers beside one converted-weight slot that both converter
 *               groups fill, 1 = one buffer beside two slots (the default)
 * The overrides apply to every later plan of the process (all threads) until
 * the next call; NULL restores the planner's choices.  Values outside those
 * ranges return MOE_ERR_INVALID_ARG and change nothing.  The library never
 * reads tuning from the environment. */
typedef struct {
  int32_t bn_max, stages, splits, pair, conv_groups, slot_kb, ksplit, dual, full_box, w_stream, unit_order;
  int32_t epi_warps, acc_bufs;
} moe_tuning_t;

moe_status_t moe_set_tuning(const moe_tuning_t* t);

/* Plan on the current device. */
moe_status_t moe_get_plan(const moe_problem_t* p, moe_plan_t* plan);

/* Plan for a device with `num_sms` SMs; pure host computation, needs no GPU. */
moe_status_t moe_get_plan_for_sms(const moe_problem_t* p, int32_t num_sms, moe_plan_t* plan);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
