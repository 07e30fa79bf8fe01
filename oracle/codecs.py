"""Number-format codecs for the oracle, written from the format definitions.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
tests/, the smoke check and the benchmark's CPU-baseline leg use it.

Formats:
  * bfloat16: the top 16 bits of an IEEE-754 binary32 value.
  * fp8 e4m3 ("E4M3" as used for the fp8 W8A8 path on "[kernel] introduce
    fused_moe_triton_splitk to sglang" and the FBGEMM grouped-GEMM blog's
    "fp8 per-tensor quant"): 1 sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; no infinities; S.1111.111 is NaN; the largest finite
    magnitude is 1.75 * 2^8 = 448; subnormals are m * 2^-9.
  * int4 with a per-group scale ("gptq/awq" W4A16 on "[Kernel] add triton
    fused moe kernel for gptq/awq"): a signed two's-complement code in
    [-8, 7], two per byte with the low nibble holding the even index; value =
    code * scale, one fp16 scale per group of 128 consecutive K elements
    (symmetric).  The asymmetric form of the same page (AWQ checkpoints,
    `zero_point` in the quantisation config): unsigned codes q in [0, 15] and
    one integer zero point z per group, value = (q - z) * scale.
  * int8 with a per-group scale (the 8-bit, group-128 GPTQ Mixtral-8x7B
    checkpoint a user runs on "Optimized fused MoE Kernel, take 2"; the
    W{4,8}A16 `moe_wna16` path of "[Kernel] add triton fused moe kernel for
    gptq/awq"): one signed two's-complement code in [-128, 127] per byte,
    value = code * scale; asymmetric: unsigned q in [0, 255], zero point z in
    [0, 255], value = (q - z) * scale.  Same fp16 group scales.

All decoders return exact float64 values.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """Values taken exactly (float64 or float32) -> nearest bf16 bit patterns
    (uint16), ties to even.  bf16: 1 sign bit, 8 exponent bits with bias 127,
    7 stored mantissa bits; the quantum is 2^(e-7) for |x| in [2^e, 2^(e+1)),
    e >= -126 (below that the subnormal quantum 2^-133); results past the
    largest finite value (2 - 2^-7) * 2^127 round to infinity; NaN -> 0x7FC0.
    One rounding from the exact value (no detour through float32)."""
    with np.errstate(invalid="ignore"):
        v = np.asarray(x).astype(np.float64)
    nan = np.isnan(v)
    neg = np.signbit(v)
    inf = np.isinf(v)
    a = np.abs(np.where(nan | inf, 0.0, v))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    e = np.maximum(e, -126.0)
    q = np.exp2(e - 7.0)
    r = np.rint(a / q) * q               # RNE on the exact quotient (q is a power of two)
    over = (r >= 2.0 ** 128) | inf
    r32 = np.where(over, np.inf, r).astype(np.float32)   # exact: r has at most 8 significant bits
    bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = bits | np.where(neg, np.uint16(0x8000), np.uint16(0))
    return np.where(nan, np.uint16(0x7FC0), bits).astype(np.uint16)


def dynamic_scale(values: np.ndarray) -> float:
    """Per-tensor dynamic fp8 scale: float32(max |v|) / 448 in float32
    arithmetic (the largest magnitude maps to the e4m3 maximum); 1.0 when the
    tensor is empty or all zero (any scale then quantises it to zeros)."""
    v = np.asarray(values, dtype=np.float64)
    amax = float(np.max(np.abs(v))) if v.size else 0.0
    if amax == 0.0:
        return 1.0
    return float(np.float32(amax) / np.float32(E4M3_MAX))


def decode_fp16(bits_or_values: np.ndarray) -> np.ndarray:
    a = np.asarray(bits_or_values)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return a.astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3 codes -> exact float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    bexp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    sub = man * 2.0 ** -9
    nor = (1.0 + man / 8.0) * np.exp2((bexp - 7).astype(np.float64))
    v = np.where(bexp == 0, sub, nor)
    v = np.where((bexp == 15) & ((c & 7) == 7), np.nan, v)
    return sign * v


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """Round float values to e4m3 codes: round-to-nearest-even, saturating.

    Magnitudes at or beyond 448 (after rounding) become +-448; NaN stays NaN.
    The input is taken at its own precision (callers pass float32 values so
    that the rounding decision is the one a float32 pipeline makes).
    """
    v = np.asarray(x, dtype=np.float64)
    nan = np.isnan(v)
    neg = np.signbit(v)
    a = np.abs(np.where(nan, 0.0, v))
    # Exponent of the normal range: a in [2^e, 2^(e+1)), e >= -6.
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 may be off by one ulp at exact powers of two: repair.
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    e = np.maximum(e, -6.0)
    # Quantum is 2^(e-3) in both the normal (e >= -6) and subnormal ranges.
    q = np.exp2(e - 3.0)
    m = np.rint(a / q)               # numpy rint = round half to even
    r = m * q                         # rounded magnitude, exact
    r = np.minimum(r, E4M3_MAX)       # saturate
    # Re-derive fields from the rounded magnitude.
    small = r < 2.0 ** -6
    code_sub = np.rint(r / 2.0 ** -9)
    with np.errstate(divide="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    er = np.where(np.exp2(er) > r, er - 1, er)
    er = np.where(np.exp2(er + 1) <= r, er + 1, er)
    man = np.rint((r / np.exp2(er) - 1.0) * 8.0)
    code_nor = (er + 7) * 8 + man
    code = np.where(small, code_sub, code_nor).astype(np.int64)
    code = code | np.where(neg, 0x80, 0)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> int64 codes [..., K] in [-8, 7]; low nibble = even k."""
    p = np.asarray(packed).astype(np.int64)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def unpack_uint4(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> int64 codes [..., K] in [0, 15]; low nibble = even k
    (the unsigned codes of the zero-point format)."""
    p = np.asarray(packed).astype(np.int64)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = (p >> 4) & 0xF
    return out


def decode_int4_grouped_zp(packed: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                           group_size: int) -> np.ndarray:
    """Asymmetric int4 (AWQ / GPTQ style): unsigned codes q in [0, 15], one fp16
    scale s and one integer zero point z in [0, 15] per group of `group_size`
    along K; w = (q - z) * s."""
    q = unpack_uint4(packed).astype(np.float64)
    s = decode_fp16(scales)
    z = np.asarray(zeros).astype(np.float64)
    K = q.shape[-1]
    assert s.shape[-1] * group_size == K and z.shape == s.shape, (s.shape, z.shape, K, group_size)
    return (q - np.repeat(z, group_size, axis=-1)) * np.repeat(s, group_size, axis=-1)


def decode_int4_grouped(packed: np.ndarray, scales: np.ndarray, group_size: int) -> np.ndarray:
    """Packed int4 [..., K/2] with fp16 scales [..., K/G] -> float64 [..., K]."""
    q = unpack_int4(packed).astype(np.float64)
    s = decode_fp16(scales)
    K = q.shape[-1]
    assert s.shape[-1] * group_size == K, (s.shape, K, group_size)
    return q * np.repeat(s, group_size, axis=-1)


def _grouped(q: np.ndarray, scales: np.ndarray, zeros, group_size: int) -> np.ndarray:
    """(q - z) * s with s (and z) repeated over each group of `group_size` along K."""
    s = decode_fp16(scales)
    K = q.shape[-1]
    assert s.shape[-1] * group_size == K, (s.shape, K, group_size)
    w = q.astype(np.float64)
    if zeros is not None:
        z = np.asarray(zeros).astype(np.float64)
        assert z.shape == s.shape, (z.shape, s.shape)
        w = w - np.repeat(z, group_size, axis=-1)
    return w * np.repeat(s, group_size, axis=-1)


def int8_codes(codes: np.ndarray) -> np.ndarray:
    """Bytes read as signed two's-complement codes in [-128, 127] (int64)."""
    return np.asarray(codes).astype(np.uint8).view(np.int8).astype(np.int64)


def decode_int8_grouped(codes: np.ndarray, scales: np.ndarray, group_size: int) -> np.ndarray:
    """Symmetric int8: one signed code per byte [..., K], fp16 scales [..., K/G]."""
    return _grouped(int8_codes(codes), scales, None, group_size)


def decode_int8_grouped_zp(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                           group_size: int) -> np.ndarray:
    """Asymmetric int8: unsigned codes q in [0, 255], zero points z in [0, 255]
    per group; w = (q - z) * s."""
    return _grouped(np.asarray(codes).astype(np.uint8).astype(np.int64), scales, zeros, group_size)
