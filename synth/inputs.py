"""Seeded synthetic inputs for the fused MoE layer.

This module is shared by the tests, the benchmark and the smoke check.  It only
draws random numbers and encodes them into the storage formats the layer reads
(bf16, fp8 e4m3 with a per-expert scale, int4 with a per-group fp16 scale).  It
holds none of the layer's arithmetic: no gating, no permutation, no GEMM, no
SwiGLU, no reduction.  Both the oracle and the CUDA path consume what it makes.

Workload shapes follow the five model shapes the pages benchmark MoE kernels on
(Mixtral-8x7B on "Optimized fused MoE Kernel, take 2"; Qwen2-57B-A14B on
"fused_moe_triton_splitk" and the FBGEMM grouped-GEMM blog; DeepSeek-V3 on
"triton fused moe kernel for gptq/awq" and "Add deepseek_v3 fused gate";
Llama-4-Scout on the FBGEMM grouped-GEMM blog), plus a tiny shape for the
oracle.  No model weights or datasets are used: every tensor is drawn here.

Storage formats (the layer's input contract):
  * bf16 weights: torch.bfloat16, w13 [E, 2I, H], w2 [E, H, I].
  * fp8 weights: e4m3 codes as uint8 with the same shapes, plus one fp32 scale
    per expert and matrix (w = e4m3(code) * scale[e]).
  * int4 weights: two signed (two's-complement) 4-bit codes per byte along K,
    the low nibble holding the even K index: w13 [E, 2I, H/2], w2 [E, H, I/2]
    uint8; per-group fp16 scales w13_scale [E, 2I, H/G], w2_scale [E, H, I/G]
    with G = 128 (w = code * scale).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Static description of one MoE layer shape and its routing recipe."""
    name: str
    H: int
    I: int
    E: int
    top_k: int
    scoring: str              # "softmax" | "sigmoid"
    renormalize: bool
    n_group: int = 0          # 0 = ungrouped
    topk_group: int = 0
    routed_scaling_factor: float = 1.0
    wdtype: str = "bf16"      # "bf16" | "fp8" | "int4" | "int8"
    group_size: int = 128     # int4 / int8 only
    logit_sd: float = 1.0
    has_bias: bool = False
    routing: str = "iid"      # "iid" | "half_to_expert0"
    weight_sd: float = 0.02
    zero_point: bool = False  # int4 / int8: unsigned codes with per-group zero points
    act_scale: str = "static"  # fp8: "static" scales from the generator, or "dynamic" (computed per batch)
    int4_order: str = "packed"  # int4: weights are generated packed; "paired": the library gets a copy
                                # prepared by moe_repack_int4 (format MOE_W_INT4_G128_PAIRED)


SHAPES = {
    # Tiny shape the CPU oracle finishes in well under a second.
    "tiny": MoEShape("tiny", H=256, I=512, E=8, top_k=2, scoring="softmax", renormalize=True),
    # Mixtral-8x7B MoE layer.
    "mixtral": MoEShape("mixtral", H=4096, I=14336, E=8, top_k=2, scoring="softmax", renormalize=True),
    # Qwen2-57B-A14B routed experts, fp8 W8A8 per-tensor.
    "qwen2": MoEShape("qwen2", H=3584, I=2560, E=64, top_k=8, scoring="softmax", renormalize=False,
                      wdtype="fp8", logit_sd=2.0),
    # DeepSeek-V3 routed experts, int4 W4A16 group 128, grouped sigmoid gate.
    "dsv3": MoEShape("dsv3", H=7168, I=2048, E=256, top_k=8, scoring="sigmoid", renormalize=True,
                     n_group=8, topk_group=4, routed_scaling_factor=2.5, wdtype="int4", has_bias=True),
    # Llama-4-Scout-style: top-1 with a sigmoid weight, half the tokens forced to expert 0.
    "scout": MoEShape("scout", H=5120, I=8192, E=16, top_k=1, scoring="sigmoid", renormalize=False,
                      routing="half_to_expert0"),
}

# DeepSeek-V3 with asymmetric AWQ-style int4 (unsigned codes, per-group zero
# points), the format of the DeepSeek-V3-AWQ checkpoints the pages benchmark.
SHAPES["dsv3_awq"] = dataclasses.replace(SHAPES["dsv3"], name="dsv3_awq", zero_point=True)
# The same int4 weights prepared once by moe_repack_int4 (codes paired for the
# converters), symmetric and with zero points.
SHAPES["dsv3_paired"] = dataclasses.replace(SHAPES["dsv3"], name="dsv3_paired", int4_order="paired")
SHAPES["dsv3_awq_paired"] = dataclasses.replace(SHAPES["dsv3_awq"], name="dsv3_awq_paired", int4_order="paired")
# Mixtral-8x7B with 8-bit group-128 GPTQ-style weights (W8A16, symmetric).
SHAPES["mixtral_w8"] = dataclasses.replace(SHAPES["mixtral"], name="mixtral_w8", wdtype="int8")
# Qwen2-57B-A14B fp8 W8A8 with dynamic per-tensor activation scales.
SHAPES["qwen2_dyn"] = dataclasses.replace(SHAPES["qwen2"], name="qwen2_dyn", act_scale="dynamic")

# Tensor-parallel slices of the same layers as the pages run them (the expert
# intermediate size split over the TP ranks; one rank's share on one GPU):
# Mixtral-8x7B TP2, Qwen2-57B-A14B TP4, DeepSeek-V3 TP8, Llama-4-Scout TP8.
for _base, _tp in (("mixtral", 2), ("qwen2", 4), ("dsv3", 8), ("scout", 8), ("dsv3_paired", 8)):
    _s = SHAPES[_base]
    SHAPES[f"{_base}_tp{_tp}"] = dataclasses.replace(_s, name=f"{_base}_tp{_tp}", I=_s.I // _tp)
del _base, _tp, _s

T_SWEEP = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)


def shrink(shape: MoEShape, H: int, I: int, E: int | None = None, name: str | None = None) -> MoEShape:
    """Same routing/dtype recipe at smaller H, I (and optionally E)."""
    kw = dict(H=H, I=I, name=name or f"{shape.name}_small")
    if E is not None:
        kw["E"] = E
    return dataclasses.replace(shape, **kw)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weight_seed(seed: int) -> int:
    return 1_000_003 * int(seed) + 7


def token_seed(seed: int, T: int) -> int:
    return 1_000_003 * int(seed) + 104_729 * int(T) + 13


@dataclasses.dataclass
class Weights:
    wdtype: str
    w13: torch.Tensor
    w2: torch.Tensor
    w13_scale: torch.Tensor | None = None
    w2_scale: torch.Tensor | None = None
    w13_zero: torch.Tensor | None = None  # int4 / int8 with zero points: uint8 [E, 2I, H/G]
    w2_zero: torch.Tensor | None = None   # uint8 [E, H, I/G]


def _pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """codes int8 in [-8, 7], last dim even -> uint8, low nibble = even index."""
    u = (codes.to(torch.int16) & 0xF).to(torch.uint8)
    lo = u[..., 0::2]
    hi = u[..., 1::2]
    return lo | (hi << 4)


def _encode_expert_zp(w: torch.Tensor, group_size: int, bits: int = 4):
    """Asymmetric int4 / int8 of one fp32 matrix [rows, K]: per group of
    `group_size` along K, with qmax = 2^bits - 1, s = (max - min) / qmax (fp16),
    z = round(-min / s) in [0, qmax], q = round(w / s) + z clamped to
    [0, qmax]; returns (codes uint8, packed two per byte for int4, s, z)."""
    qmax = (1 << bits) - 1
    rows, K = w.shape
    g = w.reshape(rows, K // group_size, group_size)
    lo, hi = g.amin(dim=-1), g.amax(dim=-1)
    s16 = ((hi - lo) / qmax).clamp_min(2.0 ** -14).to(torch.float16)
    sf = s16.float()
    z = torch.round(-lo / sf).clamp(0, qmax)
    q = (torch.round(g / sf.unsqueeze(-1)) + z.unsqueeze(-1)).clamp(0, qmax).to(torch.uint8)
    q = q.reshape(rows, K)
    if bits == 4:
        q = q[..., 0::2] | (q[..., 1::2] << 4)
    return q, s16, z.to(torch.uint8)


def _encode_expert(w: torch.Tensor, wdtype: str, group_size: int):
    """Encode one fp32 expert matrix [rows, K] into the storage format."""
    if wdtype == "bf16":
        return w.to(torch.bfloat16), None
    if wdtype == "fp8":
        scale = w.abs().amax().clamp_min(1e-30) / 448.0
        q = (w / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        return q, scale.to(torch.float32).reshape(())
    if wdtype == "int4":
        rows, K = w.shape
        g = w.reshape(rows, K // group_size, group_size)
        s16 = (g.abs().amax(dim=-1) / 7.0).clamp_min(2.0 ** -14).to(torch.float16)
        q = torch.round(g / s16.float().unsqueeze(-1)).clamp(-8, 7).to(torch.int8)
        return _pack_int4(q.reshape(rows, K)), s16
    if wdtype == "int8":
        rows, K = w.shape
        g = w.reshape(rows, K // group_size, group_size)
        s16 = (g.abs().amax(dim=-1) / 127.0).clamp_min(2.0 ** -14).to(torch.float16)
        q = torch.round(g / s16.float().unsqueeze(-1)).clamp(-128, 127).to(torch.int8)
        return q.reshape(rows, K).view(torch.uint8), s16
    raise ValueError(wdtype)


def make_weights(shape: MoEShape, device="cpu", seed: int = 0) -> Weights:
    """Expert weights ~ N(0, weight_sd), encoded into the shape's storage format.

    Experts are drawn one at a time (w13_e then w2_e) so the fp32 working set
    stays at one expert even for the largest shapes.
    """
    E, H, I = shape.E, shape.H, shape.I
    gen = _gen(device, weight_seed(seed))
    wd = shape.wdtype
    if wd == "bf16":
        w13 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
        w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
        s13 = s2 = None
    elif wd == "fp8":
        w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
        w2 = torch.empty((E, H, I), dtype=torch.uint8, device=device)
        s13 = torch.empty((E,), dtype=torch.float32, device=device)
        s2 = torch.empty((E,), dtype=torch.float32, device=device)
    elif wd == "int4":
        G = shape.group_size
        assert H % G == 0 and I % G == 0
        w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
        w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
        s13 = torch.empty((E, 2 * I, H // G), dtype=torch.float16, device=device)
        s2 = torch.empty((E, H, I // G), dtype=torch.float16, device=device)
    elif wd == "int8":
        G = shape.group_size
        assert H % G == 0 and I % G == 0
        w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
        w2 = torch.empty((E, H, I), dtype=torch.uint8, device=device)
        s13 = torch.empty((E, 2 * I, H // G), dtype=torch.float16, device=device)
        s2 = torch.empty((E, H, I // G), dtype=torch.float16, device=device)
    else:
        raise ValueError(wd)
    zp = wd in ("int4", "int8") and shape.zero_point
    bits = 8 if wd == "int8" else 4
    z13 = torch.empty((E, 2 * I, H // shape.group_size), dtype=torch.uint8, device=device) if zp else None
    z2 = torch.empty((E, H, I // shape.group_size), dtype=torch.uint8, device=device) if zp else None
    for e in range(E):
        a = torch.randn((2 * I, H), generator=gen, device=device, dtype=torch.float32) * shape.weight_sd
        if zp:
            q, s, z = _encode_expert_zp(a, shape.group_size, bits)
            z13[e].copy_(z)
        else:
            q, s = _encode_expert(a, wd, shape.group_size)
        w13[e].copy_(q)
        if s is not None:
            s13[e].copy_(s)
        del a
        b = torch.randn((H, I), generator=gen, device=device, dtype=torch.float32) * shape.weight_sd
        if zp:
            q, s, z = _encode_expert_zp(b, shape.group_size, bits)
            z2[e].copy_(z)
        else:
            q, s = _encode_expert(b, wd, shape.group_size)
        w2[e].copy_(q)
        if s is not None:
            s2[e].copy_(s)
        del b
    return Weights(wd, w13, w2, s13, s2, z13, z2)


@dataclasses.dataclass
class Tokens:
    x: torch.Tensor               # [T, H] bf16
    logits: torch.Tensor          # [T, E] fp32
    bias: torch.Tensor | None     # [E] fp32
    a1_scale: torch.Tensor | None  # [1] fp32 (fp8 only)
    a2_scale: torch.Tensor | None  # [1] fp32 (fp8 only)
    forced: torch.Tensor | None = None  # tokens forced to expert 0 (scout recipe)


def static_act_scale(shape: MoEShape) -> float:
    """Static per-tensor fp8 scale for the SwiGLU activation.

    Chosen from the input distributions, not from any computed activation:
    h = W x has standard deviation sigma = weight_sd * sqrt(H) for x ~ N(0, 1),
    and |silu(g) * u| stays below (6 sigma)^2 except on a negligible fraction of
    rows, so that bound maps to the e4m3 maximum 448.  Larger values saturate
    (both the oracle and the kernel saturate the same way).
    """
    sigma = shape.weight_sd * math.sqrt(shape.H)
    return float((6.0 * sigma) ** 2 / 448.0)


def make_tokens(shape: MoEShape, T: int, device="cpu", seed: int = 0) -> Tokens:
    gen = _gen(device, token_seed(seed, T))
    x = torch.randn((T, shape.H), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn((T, shape.E), generator=gen, device=device, dtype=torch.float32) * shape.logit_sd
    forced = None
    if shape.routing == "half_to_expert0" and T > 0:
        # floor(T/2) tokens, chosen by a seeded permutation, get expert 0's logit
        # raised 1.0 above the row maximum; the rest keep iid N(0,1) logits.
        order = torch.randperm(T, generator=gen, device=device)
        forced = order[: T // 2]
        if forced.numel():
            row_max = logits[forced].amax(dim=1)
            logits[forced, 0] = row_max + 1.0
    bias = None
    if shape.has_bias:
        bias = (torch.rand((shape.E,), generator=gen, device=device, dtype=torch.float32) * 0.2 - 0.1)
    a1 = a2 = None
    if shape.wdtype == "fp8" and shape.act_scale == "static":
        amax = x.float().abs().amax() if T > 0 else torch.tensor(1.0, device=device)
        a1 = (amax.clamp_min(1e-12) / 448.0).reshape(1).to(torch.float32)
        a2 = torch.full((1,), static_act_scale(shape), dtype=torch.float32, device=device)
    return Tokens(x, logits, bias, a1, a2, forced)


def l2_flush_buffer(device, nbytes: int) -> torch.Tensor:
    return torch.empty((nbytes,), dtype=torch.uint8, device=device)
