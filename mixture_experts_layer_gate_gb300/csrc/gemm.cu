// Stage 3: persistent grouped GEMMs on the 5th-generation tensor cores.
//
// Prior art on the pages: Triton fused_moe tuned per batch size ("Optimized
// fused MoE Kernel, take 2"), split-K ("[kernel] introduce fused_moe_triton_
// splitk to sglang"), a persistent TMA grouped GEMM (FBGEMM grouped-GEMM blog),
// int4 dequantisation inside one launch instead of one launch per expert
// ("[Kernel] add triton fused moe kernel for gptq/awq") and TensorRT-LLM's
// grouped GEMM without padding ("Add deepseek_v3 fused gate").
//
// Design for sm_103a:
//   * Weights are the MMA's A operand (M = 128 weight rows) and the expert's
//     token rows are B (N = 16..256 tokens, sized per tile to the tokens the
//     expert actually has), so a decode step with 1..32 tokens per expert does
//     not pad to 128 tokens.  D = A * B^T lands in tensor memory (TMEM).
//   * One CTA per SM loops over work units (expert, 128-row weight block, token
//     block, K slice).  Units are derived on the device from the expert row
//     offsets, so no host synchronisation is needed and empty experts cost
//     nothing.
//   * Warp roles: warp 0 issues TMA loads into a ring of shared-memory stages,
//     warp 1 owns TMEM and issues tcgen05.mma from one thread, warps 2..5
//     (or 2..9, two per TMEM lane quarter) drain the double-buffered
//     accumulator (tcgen05.ld) and run the epilogue while the next unit
//     accumulates.
//   * int4 / int8 weights (grouped_gemm_wna16_kernel, W4A16 / W8A16): each
//     ring stage holds 4 k-blocks of codes (128 / 256 bytes per weight row)
//     plus the 4 matching token tiles; converter warp groups turn the codes,
//     fp16 group scales and optional zero points into bf16 and write them
//     straight into TMEM (tcgen05.st), and the MMA reads its A operand from
//     TMEM.  No converted tile passes through shared memory.
//   * gate_up: the A tile holds 64 gate rows and the 64 matching up rows,
//     interleaved in blocks of 16 (one 5-D TMA box), so SiLU(gate) * up pairs
//     lanes l and l + 16 of the same warp in the epilogue.
//   * Small token counts split K into P slices that write fp32 partial sums;
//     a separate pass adds them in slice order (no atomics).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kABytes = 16384;    // 128 rows x 128 B (bf16 / e4m3 weight tile)
constexpr int kSuper = kInt4StageKb;  // int4 / int8: k-blocks per ring stage
constexpr int kCodeBox = 16384;       // int4 / int8: one TMA box of codes, 128 rows x 128 B
constexpr int kStgBytesPerWarp = 2048;  // epilogue staging, per epilogue warp
constexpr uint32_t kTmemCols = 512;

// Shared-memory plan (offsets from a 1024-aligned base).
//   bf16 / fp8 : ring of `stages` x {A tile 16 KB} then `stages` x {B tile bn_max x 128 B}
//   int4 / int8: ring of `stages` x {codes 16 / 32 KB, 4 B tiles of bn_max x 128 B}
struct SmemLayout {
  uint32_t a, r, r_stride, stg, bars, misc, tiles, total;
};

__host__ __device__ inline SmemLayout smem_layout(int wk, int bn_max, int stages, int astages,
                                                  int E, int epi_warps) {
  SmemLayout L;
  uint32_t o = 0;
  const uint32_t bbytes = static_cast<uint32_t>(bn_max) * 128u;  // multiple of 2 KB
  if (converts(wk)) {
    L.a = 0;
    L.r = o;
    L.r_stride = static_cast<uint32_t>(raw_stage_bytes(wk)) + kSuper * bbytes;
    o += stages * L.r_stride;
  } else {
    L.a = o;
    o += stages * kABytes;
    L.r = o;
    L.r_stride = bbytes;
    o += stages * bbytes;
  }
  L.stg = o;
  o += static_cast<uint32_t>(epi_warps) * kStgBytesPerWarp;
  L.bars = o;
  o += (2 * stages + 2 * astages + 6) * 8;
  o = (o + 15u) & ~15u;
  L.misc = o;
  o += 16;
  L.tiles = o;
  o += (4 * (E + 1) + 1) * 4;  // tile_base, off, heavy and light prefixes, order in effect
  L.total = o + 1024;  // slack to align the dynamic base to 1024 B
  return L;
}

struct Unit {
  int e, fb, row0, nvalid, n, kb0, kb1, sp;
};

__device__ __forceinline__ Unit decode_unit(int u, const int* tile_base, const int* off,
                                            const GemmParams& p) {
  Unit t;
  const int tile = u / p.P;
  t.sp = u - tile * p.P;
  // Expert-major order: an expert's units are consecutive (weight block fb, then
  // its token tiles).  Weight-block-major order: for each fb, every expert's
  // token tiles; concurrent units then mix experts, e.g. one expert's
  // tensor-bound tiles with the weight streams of experts that have few rows.
  // Heavy / light interleave: experts with more than one token tile (their
  // weight tiles serve many rows: tensor-bound) and the rest (weight-bound)
  // are listed separately, and unit positions take from the two lists in
  // proportion to their sizes, so every stretch of concurrent units mixes
  // the two kinds instead of running them one after the other.
  int key = tile, fbm = 0;
  const int* base = tile_base;
  // order in effect (build_tile_table): the interleave only where both kinds exist
  const int order = off[3 * (p.E + 1)];
  if (order == 1) {
    const int nt = tile_base[p.E] / p.FB;  // token tiles over all experts
    fbm = tile / nt;
    key = (tile - fbm * nt) * p.FB;
  } else if (order == 2) {
    const int* hb = off + (p.E + 1);
    const long long H = hb[p.E], U = tile_base[p.E];
    const long long nh = (static_cast<long long>(tile) * H) / U;
    if (((static_cast<long long>(tile) + 1) * H) / U > nh) {
      base = hb;
      key = static_cast<int>(nh);
    } else {
      base = hb + (p.E + 1);
      key = tile - static_cast<int>(nh);
    }
  }
  int lo = 0, hi = p.E;  // largest e with base[e] <= key
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (base[mid] <= key) lo = mid; else hi = mid;
  }
  t.e = lo;
  const int cnt = off[lo + 1] - off[lo];
  const int nb = (cnt + p.bn_max - 1) / p.bn_max;
  const int local = key - base[lo];
  int tb;
  if (order == 1) {
    t.fb = fbm;
    tb = local / p.FB;
  } else {
    t.fb = local / nb;
    tb = local - t.fb * nb;
  }
  // full tiles of bn_max rows and a shorter last one (tiles of equal height
  // measured slower for bf16 / fp8: more, smaller token boxes per k-block)
  t.row0 = off[lo] + tb * p.bn_max;
  t.nvalid = min(p.bn_max, cnt - tb * p.bn_max);
  t.n = (t.nvalid + 15) & ~15;
  t.kb0 = static_cast<int>((static_cast<long long>(t.sp) * p.KB) / p.P);
  t.kb1 = static_cast<int>((static_cast<long long>(t.sp + 1) * p.KB) / p.P);
  return t;
}

// Work-unit prefix over experts (run by one full warp): expert e owns
// ceil(count_e / bn_max) * FB tiles; tile_base[E] is the total.  With the
// heavy / light order requested it also writes the prefixes of experts with
// more than one token tile (heavy) and of the others (light), and records the
// order in effect: the interleave only when both kinds are present.
__device__ void build_tile_table(const GemmParams& p, int lane, int* tile_base, int* off) {
  const int per = (p.E + 31) / 32;
  const int e0 = lane * per;
  int local = 0, lh = 0;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < p.E) {
      const int c = p.offsets[e + 1] - p.offsets[e];
      const int nb = (c + p.bn_max - 1) / p.bn_max;
      local += nb * p.FB;
      if (nb >= 2) lh += nb * p.FB;
    }
  }
  int incl = local, ih = lh;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int vh = __shfl_up_sync(0xffffffffu, ih, o);
    if (lane >= o) {
      incl += v;
      ih += vh;
    }
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const int heavy = __shfl_sync(0xffffffffu, ih, 31);
  const bool mixed = p.unit_order == 2 && heavy > 0 && heavy < total;
  int run = incl - local, rh = ih - lh, rl = run - rh;
  int* hb = off + (p.E + 1);
  int* lb = hb + (p.E + 1);
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < p.E) {
      const int o0 = p.offsets[e];
      const int c = p.offsets[e + 1] - o0;
      const int nt = ((c + p.bn_max - 1) / p.bn_max) * p.FB;
      tile_base[e] = run;
      off[e] = o0;
      run += nt;
      if (mixed) {
        hb[e] = rh;
        lb[e] = rl;
        if (nt >= 2 * p.FB) rh += nt; else rl += nt;
      }
    }
  }
  if (lane == 31) {
    tile_base[p.E] = incl;
    off[p.E] = p.offsets[p.E];
    if (mixed) {
      hb[p.E] = heavy;
      lb[p.E] = total - heavy;
    }
    off[3 * (p.E + 1)] = mixed ? 2 : (p.unit_order == 1 ? 1 : 0);
  }
}

// 8 packed int4 codes (low nibble first) -> 8 bf16 (code - zero) * scale in k
// order.  One byte permute of (x, x >> 4) puts the nibbles of k = 2i and
// 2i + 1 at the bottom of the low and high halves; masking them and OR-ing the
// bf16 pattern 0x4300 (= 128) makes each half the exact bf16 value 128 + q
// (bf16 steps by 1 on [128, 256)).  Signed two's-complement codes v are the
// unsigned codes q = v + 8 with zero point 8, which the same logic op reaches
// by also flipping bit 3 (`flip` = 0x43084308 instead of 0x43004300).
// Subtracting `off` = 128 + zero recovers q - zero exactly; the scale multiply
// rounds once.  Integer-pipe work is the cost that matters here (bf16x2
// arithmetic is far cheaper), hence 9 integer ops per 8 codes.
__device__ __forceinline__ uint4 dequant8(uint32_t x, uint32_t flip, __nv_bfloat162 off,
                                          __nv_bfloat162 s2) {
  const uint32_t xs = x >> 4;
  uint32_t o[4];
  o[0] = (__byte_perm(x, xs, 0x4400) & 0x000F000Fu) ^ flip;  // k0, k1
  o[1] = (__byte_perm(x, xs, 0x5511) & 0x000F000Fu) ^ flip;  // k2, k3
  o[2] = (__byte_perm(x, xs, 0x6622) & 0x000F000Fu) ^ flip;  // k4, k5
  o[3] = (__byte_perm(x, xs, 0x7733) & 0x000F000Fu) ^ flip;  // k6, k7
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&o[i]);
    v = __hmul2(__hsub2(v, off), s2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same for 8 codes in the paired order of moe_repack_int4 (nibbles of the
// low 16 bits: k0, k2, k4, k6; of the high 16 bits: k1, k3, k5, k7): a shift of
// the word by 4 i puts k 2i and 2i + 1 at the bottom of the two halves, so one
// masked XOR per pair forms 128 + q with no byte permute: 7 integer operations
// per 8 codes instead of 9, the bf16x2 subtract and scale unchanged.
__device__ __forceinline__ uint4 dequant8_paired(uint32_t x, uint32_t flip, __nv_bfloat162 off,
                                                 __nv_bfloat162 s2) {
  uint32_t o[4];
  o[0] = (x & 0x000F000Fu) ^ flip;          // k0, k1
  o[1] = ((x >> 4) & 0x000F000Fu) ^ flip;   // k2, k3
  o[2] = ((x >> 8) & 0x000F000Fu) ^ flip;   // k4, k5
  o[3] = ((x >> 12) & 0x000F000Fu) ^ flip;  // k6, k7
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&o[i]);
    v = __hmul2(__hsub2(v, off), s2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 4 unsigned 8-bit codes (byte i = k i) -> 4 bf16 (code - zero) * scale in k
// order.  A byte permute writes code q into the low byte of the float
// 2^23 (bit pattern 0x4B000000), giving exactly 2^23 + q; subtracting
// `zoff` = 2^23 + zero leaves q - zero exactly, the product with the fp16
// scale (at most 9 + 11 significant bits) is exact in fp32, and the bf16
// conversion rounds once.
__device__ __forceinline__ uint2 dequant4_i8(uint32_t x, float zoff, float s) {
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u + i)) - zoff) * s;
  return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}

// Moves a ring cursor to entry `target` (>= idx) of a ring of n entries:
// pos = target mod n, phase flips once per wrap.
__device__ __forceinline__ void ring_advance(int& pos, uint32_t& phase, int& idx, int target, int n) {
  int d = target - idx;
  idx = target;
  while (d >= n) {
    d -= n;
    phase ^= 1u;
  }
  pos += d;
  if (pos >= n) {
    pos -= n;
    phase ^= 1u;
  }
}

// `n` token rows (a multiple of 16) of one k-block as 64-row boxes and then
// 16-row ones.  (A decomposition into 128-, 64-, 32- and 16-row boxes issued
// the same copies for most tiles yet made the bf16 / fp8 GEMMs 15% slower at
// mid-size batches.)  PAIR: the completion is counted on the barrier at
// shared::cluster address `bar`, possibly in the peer CTA.
template <bool PAIR>
__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap* m, uint32_t bar, int kcoord, int row,
                                         uint64_t pol) {
  if (PAIR)
    tma_load_2d_pair(dst, m, bar, kcoord, row, pol);
  else
    tma_load_2d_hint(dst, m, bar, kcoord, row, pol);
}

template <bool PAIR>
__device__ __forceinline__ void load_rows_split(const GemmMaps& maps, uint32_t dst, uint32_t bar, int kcoord,
                                                int row0, int n, uint64_t pol) {
  int r = 0;
  for (; r + 64 <= n; r += 64) tma_rows<PAIR>(dst + static_cast<uint32_t>(r) * 128u, &maps.b64, bar, kcoord, row0 + r, pol);
  for (; r < n; r += 16) tma_rows<PAIR>(dst + static_cast<uint32_t>(r) * 128u, &maps.b16, bar, kcoord, row0 + r, pol);
}

// Token-row loads of one k-block into a B tile: a single box for a full tile,
// 64- and 16-row boxes for an expert's ragged last tile.
__device__ __forceinline__ void load_token_rows(const GemmMaps& maps, const GemmParams& p,
                                                const Unit& t, uint32_t dst, uint32_t bar, int kcoord,
                                                uint64_t pol) {
  if (t.n == p.bn_max || p.full_box)
    tma_load_2d_hint(dst, &maps.b, bar, kcoord, t.row0, pol);
  else
    load_rows_split<false>(maps, dst, bar, kcoord, t.row0, t.n, pol);
}

// Weight tile of k-block kb (bf16 / e4m3: 64 / 128 K), or the codes of the
// ring stage starting at k-block kb (int4: 256 K; int8: 128 K, the first of
// the stage's two boxes).  `kc` = byte column of the box within the row.
template <int WK>
__device__ __forceinline__ void load_weight_tile(const GemmMaps& maps, const GemmParams& p,
                                                 const Unit& t, uint32_t dst, uint32_t bar, int kb,
                                                 uint64_t pol) {
  const int kc = kb * (WK == kW_INT4 ? 32 : (WK == kW_FP8 ? 128 : 64));  // bf16: elements, else bytes
  if (p.is_up)
    tma_load_5d_hint(dst, &maps.a, bar, kc, 0, 0, t.fb * 4, t.e, pol);
  else
    tma_load_3d_hint(dst, &maps.a, bar, kc, t.fb * 128, t.e, pol);
}

// Epilogue role (warps 2 .. 2 + 4 * nsub - 1): drains each unit's accumulator
// from TMEM and writes act (SwiGLU), y_perm, or fp32 split-K partials.  A warp
// may read only the TMEM lane quarter warp % 4; with nsub = 2 (eight warps) the
// two warps of a quarter take alternate 32-token column blocks, which halves an
// epilogue that would otherwise outlast short-K units (a down GEMM of a
// tensor-parallel slice stores 128 x 256 outputs per 5-20 MMAs).
// Units are taken from `first` in steps of `stride`; `pair_rank` >= 0 marks a
// CTA-pair kernel (this CTA's rows are weight block 2*fb + rank); the arrival
// that frees an accumulator goes, one per warp, to the shared::cluster address
// `tempty_cl0` (+8 for buffer 1).  DUAL: buffer b is two partial accumulators
// (columns 2b and 2b + 1 times acc_cols) from two MMA-issuing threads, the
// second written only for units of more than two k-blocks; the epilogue adds them;
// the ring then has p.acc_bufs (1 or 2) buffers, else always 2.
// Byte offset of 16-token half `c` of row h (output column) of the staged
// 32 x 16 bf16 store tile: rows of 32 bytes, four to a 128-byte line, the
// line's eight 16-byte units permuted by a line-dependent XOR so that the
// rows' 16-byte stores (a quarter warp: 8 consecutive rows) and the transposing
// reads (rows 2j, 2j + 1, 8 + 2j, ... 25 + 2j) fall on distinct bank groups.
__device__ __forceinline__ uint32_t stg_swizzle(int h, int c) {
  const int L = h >> 2;
  const int g = (L & 1) ^ (4 * ((L >> 1) & 1)) ^ ((L >> 2) & 1);
  return static_cast<uint32_t>(L * 128 + (((2 * (h & 3) + c) ^ g) << 4));
}

template <int WK, bool DUAL = false>
__device__ __forceinline__ void run_epilogue(const GemmParams& p, const int* tile_base, const int* off,
                                             int units, int first, int stride, int pair_rank,
                                             uint32_t tmem_base, uint32_t tfull0, uint32_t tempty_cl0,
                                             volatile int* abort_flag, uint8_t* stg_all, int warp, int lane,
                                             int nsub) {
  const int q = warp & 3;            // TMEM lane quarter this warp may read
  const int sub = (warp - 2) >> 2;   // which of the quarter's nsub warps
  uint8_t* stg = stg_all + (warp - 2) * kStgBytesPerWarp;
  const uint32_t nbuf = static_cast<uint32_t>(p.acc_bufs);
  uint32_t acc = 0, accph = 0;
  for (int u = first; u < units; u += stride) {
    Unit t = decode_unit(u, tile_base, off, p);
    if (pair_rank >= 0) t.fb = 2 * t.fb + pair_rank;
    if (!mbar_wait(tfull0 + 8u * acc, accph, abort_flag, p.err, 0x300u)) break;
    tc_fence_after();
    float sc = 1.0f, inv_q = 1.0f;
    // e4m3 output (static a2); with dynamic scales the fp8 gate_up stores bf16
    const bool q8 = WK == kW_FP8 && p.q_scale != nullptr;
    if (WK == kW_FP8) {
      sc = p.a_scale[0] * p.w_scale[t.e];
      if (q8) inv_q = 1.0f / p.q_scale[0];
    }
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           (DUAL ? 2u * acc : acc) * static_cast<uint32_t>(p.acc_cols);
    const bool part1 = DUAL && t.kb1 - t.kb0 > 2;  // warp-uniform
    uint32_t mx = 0;  // dynamic scales: largest stored |act| (bf16 magnitude bits), valid tokens only
    for (int cb = 32 * sub; cb < t.nvalid; cb += 32 * nsub) {
      // two 16-column loads in flight, one wait
      uint32_t vv[2][16];
      const bool two = cb + 16 < t.nvalid;  // warp-uniform
      tmem_ld16(tbase + static_cast<uint32_t>(cb), vv[0]);
      if (two) tmem_ld16(tbase + static_cast<uint32_t>(cb + 16), vv[1]);
      if (DUAL && part1) {
        uint32_t ww[2][16];
        const uint32_t t1 = tbase + static_cast<uint32_t>(p.acc_cols);
        tmem_ld16(t1 + static_cast<uint32_t>(cb), ww[0]);
        if (two) tmem_ld16(t1 + static_cast<uint32_t>(cb + 16), ww[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          vv[0][c] = __float_as_uint(__uint_as_float(vv[0][c]) + __uint_as_float(ww[0][c]));
        if (two) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            vv[1][c] = __float_as_uint(__uint_as_float(vv[1][c]) + __uint_as_float(ww[1][c]));
        }
      } else {
        tmem_ld_wait();
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
      if (h == 1 && !two) break;
      const int c0 = cb + 16 * h;
      const uint32_t (&v)[16] = vv[h];
      const int ntok = min(16, t.nvalid - c0);
      const size_t row = static_cast<size_t>(t.row0 + c0);
      if (p.epi == kEpiSwiglu) {
        // lane l < 16: gate row of feature 16q + l; lane l + 16: its up row.
        // Columns go in pairs with every lane busy and no branch: the gate lane
        // sends its odd-column gate value and gets the even-column up value,
        // the up lane the reverse, so one exchange gives each lane the operands
        // of one output (even column on gate lanes, odd on up lanes).
        const bool upl = lane >= 16;
        const int f16 = lane & 15;
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const float x0 = __uint_as_float(v[c]) * sc;
          const float x1 = __uint_as_float(v[c + 1]) * sc;
          const float recv = __shfl_xor_sync(0xffffffffu, upl ? x0 : x1, 16);
          const float g = upl ? recv : x0;
          const float uu = upl ? x1 : recv;
          const float a = silu_f32(g) * uu;
          const int col = c + (upl ? 1 : 0);
          if (q8) {
            stg[col * 16 + f16] = static_cast<uint8_t>(f32x2_to_e4m3x2(a * inv_q, 0.f) & 0xFF);
          } else {
            const __nv_bfloat16 ab = __float2bfloat16_rn(a);
            reinterpret_cast<__nv_bfloat16*>(stg)[col * 16 + f16] = ab;
            if (WK == kW_FP8 && col < ntok)  // only the fp8 gate_up stores bf16 for a later scale
              mx = max(mx, static_cast<uint32_t>(__bfloat16_as_ushort(ab)) & 0x7FFFu);
          }
        }
        __syncwarp();
        const size_t col = static_cast<size_t>(t.fb) * 64 + q * 16;
        if (q8) {
          if (lane < ntok)
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (row + lane) * p.out_ld + col) =
                *reinterpret_cast<const uint4*>(stg + lane * 16);
        } else {
          const int tok = lane >> 1, half = lane & 1;
          if (tok < ntok)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (row + tok) * p.out_ld +
                                      col + half * 8) =
                *reinterpret_cast<const uint4*>(stg + tok * 32 + half * 16);
        }
      } else if (p.epi == kEpiStore) {
        // Lane h packs its column's token pairs to bf16x2 and stages them as
        // row h of a 32 x 16 bf16 tile (two 16-byte stores); a transposing
        // ldmatrix then hands lane l the 8 consecutive outputs 8 (l % 4) .. +7
        // of token l / 4 (and l / 4 + 8), one 16-byte store each.  The tile is
        // swizzled so that neither the stores nor the reads conflict on banks.
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * sc, __uint_as_float(v[2 * i + 1]) * sc);
        *reinterpret_cast<uint4*>(stg + stg_swizzle(lane, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(stg + stg_swizzle(lane, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        __syncwarp();
        // lane l addresses row l % 8 of matrix l / 8: output column hr
        const int mj = lane >> 3, mi = lane & 7;
        const int hr = (mi >> 1) * 8 + 2 * mj + (mi & 1);
        const size_t col = static_cast<size_t>(t.fb) * 128 + q * 32 + 8 * (lane & 3);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint4 r = ldmatrix_x4_trans(smem_u32(stg + stg_swizzle(hr, hf)));
          const int tok = hf * 8 + (lane >> 2);
          if (tok < ntok)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (row + tok) * p.out_ld + col) = r;
        }
      } else {  // fp32 split-K partials
#pragma unroll
        for (int c = 0; c < 16; ++c)
          reinterpret_cast<float*>(stg)[c * 32 + lane] = __uint_as_float(v[c]) * sc;
        __syncwarp();
        float* dst0 = static_cast<float*>(p.out) + static_cast<size_t>(t.sp) * p.part_stride;
#pragma unroll
        for (int i = lane; i < 128; i += 32) {
          const int tok = i >> 3, w8 = i & 7;
          if (tok < ntok) {
            size_t col;
            if (p.is_up)
              col = static_cast<size_t>((w8 >> 2) * p.I) + static_cast<size_t>(t.fb) * 64 + q * 16 +
                    (w8 & 3) * 4;
            else
              col = static_cast<size_t>(t.fb) * 128 + q * 32 + w8 * 4;
            *reinterpret_cast<float4*>(dst0 + (row + tok) * p.out_ld + col) =
                *reinterpret_cast<const float4*>(stg + tok * 128 + w8 * 16);
          }
        }
      }
      __syncwarp();
    }
    }
    if (WK == kW_FP8 && p.amax != nullptr) {
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0 && mx != 0u) atomicMax(p.amax, mx);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(tempty_cl0 + 8u * acc);
    if (++acc == nbuf) {
      acc = 0u;
      accph ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ bf16 / fp8

template <int WK>
__global__ void __launch_bounds__(64 + 32 * kMaxEpiWarps, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const int ns = p.stages;
  const SmemLayout L = smem_layout(WK, p.bn_max, ns, 0, p.E, p.epi_warps);
  const uint32_t sA = base_u32 + L.a;
  const uint32_t sR = base_u32 + L.r;
  const uint32_t bars = base_u32 + L.bars;
#define FULL(s) (bars + 8u * static_cast<uint32_t>(s))
#define EMPTY(s) (bars + 8u * static_cast<uint32_t>(ns + (s)))
  const uint32_t tfull0 = bars + 8u * static_cast<uint32_t>(2 * ns);
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tfull0 + 32u;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.misc + 4);
  int* tile_base = reinterpret_cast<int*>(base + L.tiles);
  int* off = tile_base + (p.E + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((p.epi_warps != 4 && p.epi_warps != 8) || blockDim.x != 64u + 32u * p.epi_warps) {
    if (threadIdx.x == 0) record_error(p.err, kErrTimeout, 0x501u);  // host plans never do this
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(FULL(s), 1u);
      mbar_init(EMPTY(s), 1u);
    }
    mbar_init(tfull0, 1u);
    mbar_init(tfull0 + 8u, 1u);
    mbar_init(tempty0, static_cast<uint32_t>(p.epi_warps));  // one arrival per epilogue warp
    mbar_init(tempty0 + 8u, static_cast<uint32_t>(p.epi_warps));
    mbar_init(drain_bar, 1u);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b);
    tma_prefetch_desc(&maps.b64);
    tma_prefetch_desc(&maps.b16);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();  // offsets, tokens and (for gate_up) x_perm come from earlier kernels
  if (warp == 2) build_tile_table(p, lane, tile_base, off);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int units = tile_base[p.E] * p.P;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int kelem_b = (WK == kW_FP8) ? 128 : 64;
      const uint64_t pol_w = p.w_stream ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_t = l2_policy_evict_last();
      int st = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, tile_base, off, p);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(EMPTY(st), ph ^ 1u, abort_flag, p.err, 0x100u)) {
            ok = false;
            break;
          }
          const uint32_t bbytes = static_cast<uint32_t>(p.full_box ? p.bn_max : t.n) * 128u;
          mbar_expect_tx(FULL(st), kABytes + bbytes);
          load_weight_tile<WK>(maps, p, t, sA + st * kABytes, FULL(st), kb, pol_w);
          load_token_rows(maps, p, t, sR + st * L.r_stride, FULL(st), kb * kelem_b, pol_t);
          issued |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (ph << st);
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let loads already in flight land before the CTA exits.
        for (int s = 0; s < ns; ++s)
          if ((issued >> s) & 1u) mbar_wait(FULL(s), (issued_par >> s) & 1u, nullptr, p.err, 0x180u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, acc = 0, accph = 0;
      bool ok = true, any = false;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, tile_base, off, p);
        if (!mbar_wait(tempty0 + 8u * acc, accph ^ 1u, abort_flag, p.err, 0x200u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * static_cast<uint32_t>(p.acc_cols);
        const uint32_t idesc = make_idesc(128u, static_cast<uint32_t>(t.n), WK == kW_FP8 ? 0u : 1u);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(FULL(st), ph, abort_flag, p.err, 0x210u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(sA + st * kABytes);
          const uint64_t bd = sw128_kmajor_desc(sR + st * L.r_stride);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > t.kb0 || kk > 0) ? 1u : 0u;
            if (WK == kW_FP8)
              mma_f8(d, ad + 2u * kk, bd + 2u * kk, idesc, accum);
            else
              mma_f16(d, ad + 2u * kk, bd + 2u * kk, idesc, accum);
          }
          mma_commit(EMPTY(st));
          any = true;
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8u * acc);
        acc ^= 1u;
        if (acc == 0u) accph ^= 1u;
      }
      if (!ok && any) {
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0u, nullptr, p.err, 0x280u);
      }
    }
  } else {
    run_epilogue<WK>(p, tile_base, off, units, blockIdx.x, gridDim.x, -1, tmem_base, tfull0,
                     map_to_rank(tempty0, cluster_ctarank()), abort_flag, base + L.stg, warp, lane,
                     p.epi_warps / 4);
  }
#undef FULL
#undef EMPTY

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------- bf16 / fp8, CTA pairs
//
// A cluster of two CTAs shares one tcgen05.mma.cta_group::2 per K step: each
// CTA stages its own 128 weight rows (A) and half of the tile's token rows (B),
// the leader (rank 0) issues M = 256 MMAs over both CTAs' shared memory, and
// each CTA's TMEM receives its 128 rows of the accumulator.  Per CTA the
// operand traffic per K step falls from 16 KB + N x 128 B to 16 KB + N x 64 B.
//   FULL (leader only): both CTAs' TMA loads count on the leader's barrier, the
//   leader's producer posts the expected bytes of both.
//   EMPTY (both): the leader's commit arrives on both CTAs' barrier.
//   tfull (both) / tempty (leader, one arrival per epilogue warp of each CTA).
template <int WK>
__global__ void __launch_bounds__(64 + 32 * kMaxEpiWarps, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const int ns = p.stages;
  const int half_max = p.bn_max / 2;  // token rows per CTA of a full tile
  const SmemLayout L = smem_layout(WK, half_max, ns, 0, p.E, p.epi_warps);
  const uint32_t sA = base_u32 + L.a;
  const uint32_t sR = base_u32 + L.r;
  const uint32_t bars = base_u32 + L.bars;
#define FULL(s) (bars + 8u * static_cast<uint32_t>(s))
#define EMPTY(s) (bars + 8u * static_cast<uint32_t>(ns + (s)))
  const uint32_t tfull0 = bars + 8u * static_cast<uint32_t>(2 * ns);
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tfull0 + 32u;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.misc + 4);
  int* tile_base = reinterpret_cast<int*>(base + L.tiles);
  int* off = tile_base + (p.E + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  if ((p.epi_warps != 4 && p.epi_warps != 8) || blockDim.x != 64u + 32u * p.epi_warps) {
    if (threadIdx.x == 0) record_error(p.err, kErrTimeout, 0x501u);  // host plans never do this
    return;  // (both CTAs of the pair see the same parameters and return)
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(FULL(s), 1u);
      mbar_init(EMPTY(s), 1u);
    }
    mbar_init(tfull0, 1u);
    mbar_init(tfull0 + 8u, 1u);
    // every epilogue warp of both CTAs of the pair
    mbar_init(tempty0, 2u * static_cast<uint32_t>(p.epi_warps));
    mbar_init(tempty0 + 8u, 2u * static_cast<uint32_t>(p.epi_warps));
    mbar_init(drain_bar, 1u);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b);
    tma_prefetch_desc(&maps.b64);
    tma_prefetch_desc(&maps.b16);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish_pair();
  }
  pdl_wait();
  if (warp == 2) build_tile_table(p, lane, tile_base, off);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before anyone signals them
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int units = tile_base[p.E] * p.P;
  const int first = static_cast<int>(cluster_id_x());
  const int stride = static_cast<int>(num_clusters_x());

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const int kelem = (WK == kW_FP8) ? 128 : 64;
      const uint64_t pol_w = p.w_stream ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_t = l2_policy_evict_last();
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = first; u < units && ok; u += stride) {
        Unit t = decode_unit(u, tile_base, off, p);
        const int fb = 2 * t.fb + static_cast<int>(rank);
        const int n = (t.nvalid + 31) & ~31;
        const int half = n >> 1;
        const int r0 = t.row0 + static_cast<int>(rank) * half;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(EMPTY(st), ph ^ 1u, abort_flag, p.err, 0x100u)) {
            ok = false;
            break;
          }
          const uint32_t full_cl = map_to_rank(FULL(st), 0);
          // full_box: every tile's token rows as one box of the full tile height
          // (rows past the tile are loaded and not used): one copy per k-block
          const bool fullb = half == half_max || p.full_box;
          const uint32_t brows = static_cast<uint32_t>(fullb ? half_max : half);
          if (leader) mbar_expect_tx(FULL(st), 2u * (kABytes + brows * 128u));
          const uint32_t adst = sA + st * kABytes;
          if (p.is_up)
            tma_load_5d_pair(adst, &maps.a, full_cl, kb * kelem, 0, 0, fb * 4, t.e, pol_w);
          else
            tma_load_3d_pair(adst, &maps.a, full_cl, kb * kelem, fb * 128, t.e, pol_w);
          const uint32_t bdst = sR + st * L.r_stride;
          if (fullb)
            tma_load_2d_pair(bdst, &maps.b, full_cl, kb * kelem, r0, pol_t);
          else
            load_rows_split<true>(maps, bdst, full_cl, kb * kelem, r0, half, pol_t);
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // (after an abort, loads already issued complete into this CTA's own
      // shared memory; the final cluster barrier keeps both CTAs resident)
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && leader) {
      int st = 0;
      uint32_t ph = 0, acc = 0, accph = 0;
      bool ok = true, any = false;
      for (int u = first; u < units && ok; u += stride) {
        const Unit t = decode_unit(u, tile_base, off, p);
        const int n = (t.nvalid + 31) & ~31;
        if (!mbar_wait(tempty0 + 8u * acc, accph ^ 1u, abort_flag, p.err, 0x200u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * static_cast<uint32_t>(p.acc_cols);
        const uint32_t idesc = make_idesc(256u, static_cast<uint32_t>(n), WK == kW_FP8 ? 0u : 1u);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(FULL(st), ph, abort_flag, p.err, 0x210u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(sA + st * kABytes);
          const uint64_t bd = sw128_kmajor_desc(sR + st * L.r_stride);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > t.kb0 || kk > 0) ? 1u : 0u;
            if (WK == kW_FP8)
              mma_f8_pair(d, ad + 2u * kk, bd + 2u * kk, idesc, accum);
            else
              mma_f16_pair(d, ad + 2u * kk, bd + 2u * kk, idesc, accum);
          }
          mma_commit_pair(EMPTY(st), 0x3);
          any = true;
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull0 + 8u * acc, 0x3);
        acc ^= 1u;
        if (acc == 0u) accph ^= 1u;
      }
      if (!ok && any) {
        mma_commit_pair(drain_bar, 0x1);
        mbar_wait(drain_bar, 0u, nullptr, p.err, 0x280u);
      }
    }
  } else {
    run_epilogue<WK>(p, tile_base, off, units, first, stride, static_cast<int>(rank), tmem_base, tfull0,
                     map_to_rank(tempty0, 0), abort_flag, base + L.stg, warp, lane, p.epi_warps / 4);
  }
#undef FULL
#undef EMPTY

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no signals into either CTA remain in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------ int4
//
// Rings and the parity-wait rules they obey (a parity wait is unambiguous only
// if the waiter is never two phases ahead of the barrier):
//   RFULL/REMPTY over `stages` ring stages of 4 k-blocks (packed codes + token
//   tiles).  Converter group g takes every CG-th stage; `stages` is a multiple
//   of CG, so the previous use of a slot was by the same group.  With k-split
//   (two groups, whole-stage slots) both groups take every stage instead,
//   group g converting its k-blocks 2g and 2g + 1, and AFULL counts all eight
//   warps: a stage is converted in half the time, which keeps the MMA fed when
//   TMEM holds only two whole-stage slots.
//   AFULL/AEMPTY over `astages` TMEM slots of slot_kb (2 or 4) converted
//   k-blocks, 128 rows x 32 * slot_kb columns each: one wait and one commit
//   per 4 * slot_kb MMAs.  A group fills the 4 / slot_kb slots of its stage
//   and jumps (CG - 1) * 4 / slot_kb slots ahead; astages is at least one more
//   than that jump, so a group is at most one phase ahead of any slot it
//   waits on.  With whole-stage slots (slot_kb = 4) slot i is ring stage i's,
//   so the MMA commits once per stage (REMPTY) and a converter about to refill
//   slot i mod astages waits for REMPTY of stage i - astages instead; stages >=
//   astages keeps that barrier from running a phase past the one awaited.
// PAIR: the kernel runs as clusters of two CTAs sharing M = 256 MMAs, each CTA
// converting its own 128 weight rows into its own TMEM and staging half of the
// token rows; converter groups of both CTAs report to the leader's AFULL, the
// leader's commits are multicast to both CTAs.
// DUAL (whole-stage slots): one thread issues MMAs at a fixed rate however idle
// the tensor pipe is, and the converters' integer work slows it further, so a
// second issuing thread (an extra warp; with PAIR, of the leader CTA) takes
// k-blocks 2 and 3 of every stage into its own partial accumulator while warp 1
// takes k-blocks 0 and 1.  Both wait for every stage and both report on its
// REMPTY (count 2) and on the accumulator's TFULL (count 2), in every CTA of the
// cluster; a thread with no k-block in a stage or unit (a short end of a K
// range) arrives without a commit.  Accumulator columns: p.acc_bufs buffers (2,
// or 1 when two pairs of partials do not fit beside two converted slots) of two
// partials each.
template <int BITS, int CG, bool PAIR, int SK, bool DUAL, int EW>
__global__ void __launch_bounds__(64 + 32 * EW + 128 * CG + (DUAL ? 32 : 0), 1)
    grouped_gemm_wna16_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  static_assert(!DUAL || SK == kSuper, "two issuers: whole-stage slots");
  constexpr int WKQ = BITS == 8 ? kW_INT8 : kW_INT4;
  constexpr uint32_t kRaw = static_cast<uint32_t>(raw_stage_bytes(WKQ));  // codes per ring stage
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const int ns = p.stages;
  const int na = p.astages;
  const int brows = PAIR ? p.bn_max / 2 : p.bn_max;  // token rows this CTA stages per k-block
  const SmemLayout L = smem_layout(WKQ, brows, ns, na, p.E, EW);
  const uint32_t sR = base_u32 + L.r;
  const uint32_t btile = static_cast<uint32_t>(brows) * 128u;
  const uint32_t bars = base_u32 + L.bars;
#define RFULL(s) (bars + 8u * static_cast<uint32_t>(s))
#define REMPTY(s) (bars + 8u * static_cast<uint32_t>(ns + (s)))
#define AFULL(s) (bars + 8u * static_cast<uint32_t>(2 * ns + (s)))
#define AEMPTY(s) (bars + 8u * static_cast<uint32_t>(2 * ns + na + (s)))
  const uint32_t tfull0 = bars + 8u * static_cast<uint32_t>(2 * ns + 2 * na);
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tfull0 + 32u;  // (+8: the second issuer's)
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.misc + 4);
  int* tile_base = reinterpret_cast<int*>(base + L.tiles);
  int* off = tile_base + (p.E + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t acc_cols = static_cast<uint32_t>(p.acc_cols);
  const uint32_t nbuf = static_cast<uint32_t>(p.acc_bufs);  // accumulator buffers (1 or 2)
  const uint32_t a_col0 = (DUAL ? 2u : 1u) * nbuf * acc_cols;            // TMEM column of converted slot 0
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = (rank == 0);
  constexpr uint32_t kCtas = PAIR ? 2u : 1u;
  static_assert(SK == 2 || SK == 4, "converted slots hold 2 or 4 k-blocks");
  static_assert(EW == 4 || EW == 8, "one or two epilogue warps per TMEM lane quarter");
  constexpr int kConv0 = 2 + EW;  // first converter warp
  // k-split: both groups convert every stage (group g its k-blocks 2g, 2g + 1)
  const bool ks = p.ksplit != 0;
  if (p.slot_kb != SK || p.dual != (DUAL ? 1 : 0) || p.epi_warps != EW || nbuf < 1u || nbuf > 2u ||
      (SK == kSuper && ns < na) ||
      (ks && (SK != kSuper || CG != 2)) ||
      (!ks && (na < (CG - 1) * (kSuper / SK) + 1 || ns % CG != 0)) ||
      a_col0 + 32u * static_cast<uint32_t>(SK * na) > kTmemCols) {
    if (threadIdx.x == 0) record_error(p.err, kErrTimeout, 0x500u);  // host plans never do this
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(RFULL(s), 1u);
      mbar_init(REMPTY(s), DUAL ? 2u : 1u);
    }
    for (int s = 0; s < na; ++s) {
      // the 4 warps of the stage's converter group, or of both groups with k-split (in each CTA)
      mbar_init(AFULL(s), (ks ? 4u * CG : 4u) * kCtas);
      mbar_init(AEMPTY(s), 1u);
    }
    mbar_init(tfull0, DUAL ? 2u : 1u);
    mbar_init(tfull0 + 8u, DUAL ? 2u : 1u);
    mbar_init(tempty0, static_cast<uint32_t>(EW) * kCtas);  // one arrival per epilogue warp (of each CTA)
    mbar_init(tempty0 + 8u, static_cast<uint32_t>(EW) * kCtas);
    mbar_init(drain_bar, 1u);
    if (DUAL) mbar_init(drain_bar + 8u, 1u);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b);
    tma_prefetch_desc(&maps.b64);
    tma_prefetch_desc(&maps.b16);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
      tmem_relinquish();
    }
  }
  pdl_wait();
  if (warp == 2) build_tile_table(p, lane, tile_base, off);
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const int units = tile_base[p.E] * p.P;
  const int first = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int stride = PAIR ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = p.w_stream ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t pol_t = l2_policy_evict_last();
      int st = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int u = first; u < units && ok; u += stride) {
        Unit t = decode_unit(u, tile_base, off, p);
        if (PAIR) {
          // this CTA: weight block 2*fb + rank, token rows [row0 + rank*n/2, + n/2)
          t.fb = 2 * t.fb + static_cast<int>(rank);
          const int n = (t.nvalid + 31) & ~31;
          t.n = n >> 1;
          t.row0 += static_cast<int>(rank) * t.n;
        }
        for (int kbs = t.kb0; kbs < t.kb1; kbs += kSuper) {
          const int nk = min(kSuper, t.kb1 - kbs);
          if (!mbar_wait(REMPTY(st), ph ^ 1u, abort_flag, p.err, 0x100u)) {
            ok = false;
            break;
          }
          const uint32_t stage = sR + st * L.r_stride;
          const bool full = (t.n == brows) || p.full_box;
          const uint32_t bbytes = full ? kSuper * btile : static_cast<uint32_t>(nk * t.n) * 128u;
          // int8: the stage's codes are two boxes of two k-blocks; a stage of at
          // most two k-blocks (the end of a K range) needs only the first
          const bool two_boxes = BITS == 8 && nk > 2;
          mbar_expect_tx(RFULL(st), (BITS == 8 && !two_boxes ? kCodeBox : kRaw) + bbytes);
          load_weight_tile<WKQ>(maps, p, t, stage, RFULL(st), kbs, pol_w);
          if (two_boxes) load_weight_tile<WKQ>(maps, p, t, stage + kCodeBox, RFULL(st), kbs + 2, pol_w);
          if (full) {
            tma_load_3d_hint(stage + kRaw, &maps.b, RFULL(st), 0, t.row0, kbs, pol_t);
          } else {
            // a tile below the full height: the fewest smaller boxes per k-block
            for (int j = 0; j < nk; ++j)
              load_rows_split<false>(maps, stage + kRaw + j * btile, RFULL(st), (kbs + j) * 64, t.row0, t.n,
                                     pol_t);
          }
          issued |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (ph << st);
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < ns; ++s)
          if ((issued >> s) & 1u) mbar_wait(RFULL(s), (issued_par >> s) & 1u, nullptr, p.err, 0x180u);
      }
    }
  } else if (warp == 1 || (DUAL && warp == kConv0 + 4 * CG)) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      // issuer j (DUAL): k-blocks [2j, 2j + 2) of every stage, partial accumulator j
      const int j = warp == 1 ? 0 : 1;
      const int jb0 = DUAL ? 2 * j : 0;
      int st = 0, as = 0;
      uint32_t ph = 0, aph = 0, acc = 0, accph = 0;
      bool ok = true, any = false;
      const uint64_t bd0 = sw128_kmajor_desc(0u);
      const uint32_t bd_lo0 = static_cast<uint32_t>(bd0), bd_hi = static_cast<uint32_t>(bd0 >> 32);
      const uint32_t btile16 = btile >> 4;
      const uint32_t a_tmem0 = tmem_base + a_col0;
      const uint32_t slot_cols = 32u * static_cast<uint32_t>(SK);
      for (int u = first; u < units && ok; u += stride) {
        const Unit t = decode_unit(u, tile_base, off, p);
        if (!mbar_wait(tempty0 + 8u * acc, accph ^ 1u, abort_flag, p.err, 0x200u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (DUAL ? 2u * acc + static_cast<uint32_t>(j) : acc) * acc_cols;
        bool unit_any = !DUAL;  // DUAL: whether this thread issued any MMA of the unit
        const uint32_t n_mma = PAIR ? static_cast<uint32_t>((t.nvalid + 31) & ~31) : static_cast<uint32_t>(t.n);
        const uint32_t idesc = make_idesc(PAIR ? 256u : 128u, n_mma, 1u);
        if (SK == kSuper) {
          // Whole-stage slots: one wait, the stage's MMAs, one commit.  The next
          // stage's ring positions, barrier addresses and descriptor words are
          // worked out between this stage's first and remaining MMAs, so the
          // thread goes from the commit straight to the next wait (the tensor
          // pipe idles while this single thread does bookkeeping).
          uint32_t afull = AFULL(as), rempty = REMPTY(st);
          uint32_t b_lo = bd_lo0 + ((sR + st * L.r_stride + kRaw) >> 4);
          uint32_t a_tm = a_tmem0 + slot_cols * static_cast<uint32_t>(as);
          for (int kbs = t.kb0; kbs < t.kb1; kbs += kSuper) {
            const int nk = min(kSuper, t.kb1 - kbs);
            const int jend = DUAL ? min(nk, jb0 + 2) : nk;
            const bool mine = !DUAL || jb0 < jend;
            if (!mbar_wait(afull, aph, abort_flag, p.err, 0x210u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (mine)
              mma_kblock_tmem_a<PAIR>(d, a_tm + 32u * jb0, b_lo + btile16 * jb0, bd_hi, idesc,
                                      kbs > t.kb0 ? 1u : 0u);
            const int st_n = (st + 1 == ns) ? 0 : st + 1;
            const uint32_t ph_n = (st + 1 == ns) ? (ph ^ 1u) : ph;
            const int as_n = (as + 1 == na) ? 0 : as + 1;
            const uint32_t aph_n = (as + 1 == na) ? (aph ^ 1u) : aph;
            const uint32_t afull_n = AFULL(as_n), rempty_n = REMPTY(st_n);
            const uint32_t b_lo_n = bd_lo0 + ((sR + st_n * L.r_stride + kRaw) >> 4);
            const uint32_t a_tm_n = a_tmem0 + slot_cols * static_cast<uint32_t>(as_n);
            for (int jj = jb0 + 1; jj < jend; ++jj)
              mma_kblock_tmem_a<PAIR>(d, a_tm + 32u * jj, b_lo + btile16 * jj, bd_hi, idesc, 1u);
            if (mine) {
              if (PAIR) mma_commit_pair(rempty, 0x3); else mma_commit(rempty);
            } else {
              // read nothing of this stage
              for (uint32_t r = 0; r < kCtas; ++r) mbar_arrive_cluster(map_to_rank(rempty, r));
            }
            any = any || mine;
            unit_any = unit_any || mine;
            st = st_n;
            ph = ph_n;
            as = as_n;
            aph = aph_n;
            afull = afull_n;
            rempty = rempty_n;
            b_lo = b_lo_n;
            a_tm = a_tm_n;
          }
        } else
        for (int kbs = t.kb0; kbs < t.kb1 && ok; kbs += kSuper) {
          const int nk = min(kSuper, t.kb1 - kbs);
          // low descriptor word of the stage's first token tile
          const uint32_t b_lo = bd_lo0 + ((sR + st * L.r_stride + kRaw) >> 4);
          for (int jp = 0; jp < nk; jp += SK) {
            // the converted slot's barrier also covers the stage's token rows:
            // its converter group waited for the whole stage before converting
            if (!mbar_wait(AFULL(as), aph, abort_flag, p.err, 0x210u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_tmem = a_tmem0 + slot_cols * static_cast<uint32_t>(as);
            const uint32_t b0 = b_lo + static_cast<uint32_t>(jp) * btile16;
            mma_kblock_tmem_a<PAIR>(d, a_tmem, b0, bd_hi, idesc, kbs + jp > t.kb0 ? 1u : 0u);
            const int jn = min(SK, nk - jp);
            for (int jj = 1; jj < jn; ++jj)
              mma_kblock_tmem_a<PAIR>(d, a_tmem + 32u * jj, b0 + btile16 * jj, bd_hi, idesc, 1u);
            // whole-stage slots: the stage's REMPTY commit below also frees the slot
            if (SK != kSuper) {
              if (PAIR) mma_commit_pair(AEMPTY(as), 0x3); else mma_commit(AEMPTY(as));
            }
            any = true;
            if (++as == na) {
              as = 0;
              aph ^= 1u;
            }
          }
          if (!ok) break;
          if (PAIR) mma_commit_pair(REMPTY(st), 0x3); else mma_commit(REMPTY(st));
          if (++st == ns) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (unit_any) {
          if (PAIR) mma_commit_pair(tfull0 + 8u * acc, 0x3); else mma_commit(tfull0 + 8u * acc);
        } else {
          for (uint32_t r = 0; r < kCtas; ++r) mbar_arrive_cluster(map_to_rank(tfull0 + 8u * acc, r));
        }
        if (++acc == nbuf) {
          acc = 0u;
          accph ^= 1u;
        }
      }
      if (!ok && any) {
        const uint32_t db = drain_bar + 8u * static_cast<uint32_t>(j);
        if (PAIR) mma_commit_pair(db, 0x1); else mma_commit(db);
        mbar_wait(db, 0u, nullptr, p.err, 0x280u);
      }
    }
  } else if (warp < kConv0) {
    run_epilogue<WKQ, DUAL>(p, tile_base, off, units, first, stride, PAIR ? static_cast<int>(rank) : -1,
                          tmem_base, tfull0, map_to_rank(tempty0, 0), abort_flag, base + L.stg, warp, lane,
                          EW / 4);
  } else {
    // ---------------------------------------- int4 / int8 -> bf16 converters
    // The CTA's stages are numbered i = 0, 1, ... in (unit, k) order; a stage of
    // nk k-blocks fills ceil(nk / slot_kb) TMEM slots, numbered the same way.  Group
    // g (4 warps) converts the stages with i % CG == g (with k-split: k-blocks
    // 2g, 2g + 1 of every stage) and jumps straight from
    // one to the next: stepping through the other groups' stages one by one
    // costs hundreds of cycles each while the other groups saturate the
    // integer pipe.  The thread owns weight row m of the tile, which is TMEM
    // lane m of the converted tile.
    const int grp = (warp - kConv0) >> 2;
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const __half* scales = static_cast<const __half*>(p.w4_scale);
    // null zero points: signed codes, read as unsigned codes (sign bit flipped)
    // with zero point 8 (int4) or 128 (int8)
    const uint8_t* zeros = p.w4_zero;
    const uint32_t flip = zeros ? 0x43004300u : 0x43084308u;  // int4 (see dequant8)
    const bool paired = BITS == 4 && p.w4_paired != 0;       // int4 codes in the paired order
    const uint32_t flip8 = zeros ? 0u : 0x80808080u;           // int8
    const float zdef = BITS == 8 ? 128.0f : 8.0f;
    const uint32_t tlane = static_cast<uint32_t>(q * 32) << 16;
    int ci = 0, cst = 0, cs = 0, ca = 0;  // stage / slot index and their ring positions
    uint32_t cph = 0, cap = 0;
    int pi = 0, pst = 0;                  // ring position of stage i - astages (whole-stage slots)
    uint32_t pph = 0;
    int ui = 0, us = 0;                   // first stage / slot index of the current unit
    bool ok = true;
    const uint32_t afull_cl0 = map_to_rank(AFULL(0), 0);  // leader's AFULL(0)
    const int spp = kSuper / SK;                            // slots per full stage
    for (int u = first; u < units && ok; u += stride) {
      Unit t = decode_unit(u, tile_base, off, p);
      if (PAIR) t.fb = 2 * t.fb + static_cast<int>(rank);
      const int nkb = t.kb1 - t.kb0;
      const int nst = (nkb + kSuper - 1) / kSuper;
      const int grow = p.is_up ? (((m >> 4) & 1) * p.I + t.fb * 64 + (m >> 5) * 16 + (m & 15))
                               : (t.fb * 128 + m);
      const size_t grow_off = (static_cast<size_t>(t.e) * p.R + grow) * p.G;
      const __half* srow = scales + grow_off;
      int l = ks ? 0 : grp - ui % CG;
      if (l < 0) l += CG;
      for (; l < nst && ok; l += (ks ? 1 : CG)) {
        ring_advance(cst, cph, ci, ui + l, ns);
        ring_advance(ca, cap, cs, us + spp * l, na);  // every earlier stage of the unit is full
        const int kbs = t.kb0 + kSuper * l;
        const int nk = min(kSuper, t.kb1 - kbs);
        __half sc[kSuper];
        float zf[kSuper];
#pragma unroll
        for (int j = 0; j < kSuper; ++j) {
          const int g = min(kbs + j, t.kb1 - 1) >> 1;  // 128-wide group of k-block j
          sc[j] = srow[g];
          zf[j] = zeros ? static_cast<float>(zeros[grow_off + g]) : zdef;
        }
        if (!mbar_wait(RFULL(cst), cph, abort_flag, p.err, 0x400u)) {
          ok = false;
          break;
        }
        if (SK == kSuper && ui + l >= na) {
          // whole-stage slots: slot (i mod astages) is free once stage i - astages
          // has been consumed, i.e. after that stage's REMPTY completion
          ring_advance(pst, pph, pi, ui + l - na, ns);
          if (!mbar_wait(REMPTY(pst), pph, abort_flag, p.err, 0x410u)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint8_t* rrow = base + L.r + cst * L.r_stride + m * 128;
        int a = ca;
        uint32_t ap = cap;
        const int j0 = ks ? 2 * grp : 0;            // this warp's k-blocks of the stage: [j0, j1)
        const int j1 = ks ? min(nk, 2 * grp + 2) : nk;
#pragma unroll
        for (int j = 0; j < kSuper; ++j) {
          if (j < j0) continue;
          if (j >= j1) break;
          const int js = j & (SK - 1);  // k-block within the slot
          if (SK != kSuper && js == 0) {
            if (!mbar_wait(AEMPTY(a), ap ^ 1u, abort_flag, p.err, 0x410u)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          uint32_t outv[32];
          if (BITS == 4) {
            const __nv_bfloat162 s2 = __float2bfloat162_rn(__half2float(sc[j]));
            const __nv_bfloat162 off = __float2bfloat162_rn(128.0f + zf[j]);
            // 32 bytes of codes = 128-byte-swizzled chunks 2j and 2j+1 of the row
            const uint4 r0 = *reinterpret_cast<const uint4*>(rrow + (((2 * j) ^ (m & 7)) << 4));
            const uint4 r1 = *reinterpret_cast<const uint4*>(rrow + (((2 * j + 1) ^ (m & 7)) << 4));
            const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            if (paired) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint4 o = dequant8_paired(w[i], flip, off, s2);
                outv[4 * i + 0] = o.x;
                outv[4 * i + 1] = o.y;
                outv[4 * i + 2] = o.z;
                outv[4 * i + 3] = o.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint4 o = dequant8(w[i], flip, off, s2);
                outv[4 * i + 0] = o.x;
                outv[4 * i + 1] = o.y;
                outv[4 * i + 2] = o.z;
                outv[4 * i + 3] = o.w;
              }
            }
          } else {
            // 64 bytes of codes = chunks 4 (j & 1) .. + 3 of box j / 2
            const uint8_t* rb = rrow + (j >> 1) * kCodeBox;
            const float sf = __half2float(sc[j]);
            const float zoff = 8388608.0f + zf[j];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 r = *reinterpret_cast<const uint4*>(rb + ((((j & 1) * 4 + c) ^ (m & 7)) << 4));
              const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint2 o = dequant4_i8(w[i] ^ flip8, zoff, sf);
                outv[8 * c + 2 * i] = o.x;
                outv[8 * c + 2 * i + 1] = o.y;
              }
            }
          }
          tmem_st32(tmem_base + tlane + a_col0 + 32u * static_cast<uint32_t>(SK * a + js), outv);
          if (!ks && (js == SK - 1 || j == nk - 1)) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(afull_cl0 + 8u * static_cast<uint32_t>(a));
            if (++a == na) {
              a = 0;
              ap ^= 1u;
            }
          }
        }
        if (ks && ok) {  // one arrival per warp and stage, k-blocks or not
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(afull_cl0 + 8u * static_cast<uint32_t>(a));
        }
      }
      if (nst > 0) {
        ui += nst;
        us += spp * (nst - 1) + (nkb - kSuper * (nst - 1) + SK - 1) / SK;
      }
    }
  }
#undef RFULL
#undef REMPTY
#undef AFULL
#undef AEMPTY

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // no signals into either CTA remain in flight
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <typename K>
cudaError_t set_smem_attr(K kernel, int* configured_device) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (*configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (err != cudaSuccess) return err;
    *configured_device = dev;
  }
  return cudaSuccess;
}

template <int WK>
cudaError_t launch_dense(const GemmMaps& maps, const GemmParams& p, int grid, size_t smem,
                         cudaStream_t s) {
  static int configured = -1;  // attribute set once per device (single-device processes)
  cudaError_t err = set_smem_attr(grouped_gemm_kernel<WK>, &configured);
  if (err != cudaSuccess) return err;
  return launch_pdl(grouped_gemm_kernel<WK>, dim3(grid), dim3(gemm_threads(WK, 0, 0, p.epi_warps)), smem, s,
                    maps, p);
}

template <int WK>
cudaError_t launch_pair(const GemmMaps& maps, const GemmParams& p, int grid, size_t smem,
                        cudaStream_t s) {
  static int configured = -1;
  cudaError_t err = set_smem_attr(grouped_gemm_pair_kernel<WK>, &configured);
  if (err != cudaSuccess) return err;
  return launch_pdl_cluster(grouped_gemm_pair_kernel<WK>, dim3(grid & ~1), dim3(gemm_threads(WK, 0, 0, p.epi_warps)),
                            smem, s, 2u, maps, p);
}

template <int BITS, int CG, bool PAIR, int SK, bool DUAL = false, int EW = 4>
cudaError_t launch_wna16(const GemmMaps& maps, const GemmParams& p, int grid, size_t smem,
                         cudaStream_t s) {
  static int configured = -1;
  cudaError_t err = set_smem_attr(grouped_gemm_wna16_kernel<BITS, CG, PAIR, SK, DUAL, EW>, &configured);
  if (err != cudaSuccess) return err;
  return launch_pdl_cluster(grouped_gemm_wna16_kernel<BITS, CG, PAIR, SK, DUAL, EW>,
                            dim3(PAIR ? (grid & ~1) : grid), dim3(gemm_threads(kW_INT4, CG, DUAL ? 1 : 0, EW)),
                            smem, s, PAIR ? 2u : 1u, maps, p);
}

// int4 / int8 CTA-pair kernels with two converter groups and whole-stage slots
// come with eight epilogue warps as well as four
template <int BITS>
cudaError_t launch_wna16_pair_cg2(const GemmMaps& maps, const GemmParams& p, int grid, size_t smem,
                                  cudaStream_t s) {
  if (p.epi_warps == 8) {
    if (p.dual) return launch_wna16<BITS, 2, true, 4, true, 8>(maps, p, grid, smem, s);
    return launch_wna16<BITS, 2, true, 4, false, 8>(maps, p, grid, smem, s);
  }
  if (p.dual) return launch_wna16<BITS, 2, true, 4, true>(maps, p, grid, smem, s);
  return launch_wna16<BITS, 2, true, 4>(maps, p, grid, smem, s);
}

}  // namespace

size_t gemm_smem_bytes(int wkind, int bn_max, int stages, int astages, int E, int epi_warps) {
  return smem_layout(wkind, bn_max, stages, astages, E, epi_warps).total;
}

int gemm_threads(int wkind, int conv_groups, int dual, int epi_warps) {
  return 64 + 32 * epi_warps + (converts(wkind) ? 128 * conv_groups + (dual ? 32 : 0) : 0);
}

bool gemm_epi8_supported(int wkind, int conv_groups, int pair, int slot_kb) {
  if (!converts(wkind)) return true;
  return pair && conv_groups == 2 && slot_kb == kSuper;
}

cudaError_t launch_grouped_gemm(int wkind, const GemmMaps& maps, const GemmParams& p, int grid,
                                size_t smem, cudaStream_t s) {
  if (p.epi_warps != 4 && !(p.epi_warps == 8 && gemm_epi8_supported(wkind, p.conv_groups, p.pair, p.slot_kb)))
    return cudaErrorInvalidValue;
  switch (wkind) {
    case kW_BF16:
      return p.pair ? launch_pair<kW_BF16>(maps, p, grid, smem, s) : launch_dense<kW_BF16>(maps, p, grid, smem, s);
    case kW_FP8:
      return p.pair ? launch_pair<kW_FP8>(maps, p, grid, smem, s) : launch_dense<kW_FP8>(maps, p, grid, smem, s);
    case kW_INT4:
      if (p.slot_kb == 4) {
        if (p.pair && p.conv_groups == 3) return launch_wna16<4, 3, true, 4>(maps, p, grid, smem, s);
        if (p.pair && p.conv_groups == 2) return launch_wna16_pair_cg2<4>(maps, p, grid, smem, s);
        if (!p.pair && p.conv_groups == 3 && p.dual) return launch_wna16<4, 3, false, 4, true>(maps, p, grid, smem, s);
        if (!p.pair && p.conv_groups == 2) {
          if (p.dual) return launch_wna16<4, 2, false, 4, true>(maps, p, grid, smem, s);
          return launch_wna16<4, 2, false, 4>(maps, p, grid, smem, s);
        }
      } else if (p.slot_kb == 2) {
        if (p.pair && p.conv_groups == 3) return launch_wna16<4, 3, true, 2>(maps, p, grid, smem, s);
        if (p.pair && p.conv_groups == 2) return launch_wna16<4, 2, true, 2>(maps, p, grid, smem, s);
        if (!p.pair && p.conv_groups == 2) return launch_wna16<4, 2, false, 2>(maps, p, grid, smem, s);
      }
      return cudaErrorInvalidValue;
    case kW_INT8:  // two converter groups only
      if (p.conv_groups != 2) return cudaErrorInvalidValue;
      if (p.slot_kb == 4) {
        if (p.pair) return launch_wna16_pair_cg2<8>(maps, p, grid, smem, s);
        if (p.dual) return launch_wna16<8, 2, false, 4, true>(maps, p, grid, smem, s);
        return launch_wna16<8, 2, false, 4>(maps, p, grid, smem, s);
      } else if (p.slot_kb == 2) {
        if (p.pair) return launch_wna16<8, 2, true, 2>(maps, p, grid, smem, s);
        return launch_wna16<8, 2, false, 2>(maps, p, grid, smem, s);
      }
      return cudaErrorInvalidValue;
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
