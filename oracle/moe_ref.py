"""Plain fp64 CPU oracle for the fused MoE layer forward pass.

TEST INFRASTRUCTURE ONLY.  The library never imports, links or runs anything
in this package.  Only tests/, __graft_entry__.smoke() and the CPU-baseline leg
of bench.py use it.  It shares no code with the CUDA path.

What is computed, by stage (the pages describe the pipeline in prose only; no
page prints a formula, so each stage below states the plain reading it takes):

  1. Gate ("Add deepseek_v3 fused gate": the fused gate and the PyTorch
     reference gate it is checked against; TensorRT-LLM's fused MoE begins with
     the same gate).  Softmax top-k, optionally renormalised, or sigmoid scores
     with a per-expert correction bias and group-limited selection.
  2. Align/permute ("[Kernel] add triton fused moe kernel for gptq/awq", note 1
     on moe_align_block_size; "Add deepseek_v3 fused gate", TensorRT-LLM's
     expand_and_permute, which needs no padding).  A stable counting sort of the
     T*k token slots by expert.
  3. Per-expert gate_up GEMM, SiLU-and-mul, down GEMM (the grouped GEMMs of
     every page: Triton fused_moe, split-K, FBGEMM grouped GEMM, CUTLASS).
  4. Unpermute and top-k weighted reduction (TensorRT-LLM's
     unpermute_and_reduce on "Add deepseek_v3 fused gate").

Readings where the pages are silent:
  * Softmax selection keys are the raw fp32 logits (softmax is monotone).
  * Ids are ordered by key, descending; equal keys go to the lower index.
  * Sigmoid gate: s = sigmoid(l); key = s + bias (bias only steers selection);
    group score = sum of the two largest keys in the group; groups are
    contiguous blocks of E / n_group experts; the topk_group best groups are
    kept (ties to the lower group); weights are s of the chosen experts,
    renormalised if asked, then times routed_scaling_factor.  With no bias and
    no groups the keys are the raw logits (sigmoid is monotone).
  * w13 rows [0, I) are the gate projection (SiLU applied), rows [I, 2I) the up
    projection; silu(z) = z / (1 + exp(-z)).
  * fp8 W8A8: x and the SiLU-and-mul activation are quantised to e4m3 with
    static per-tensor scales a1, a2 (value / scale in float32, round to nearest
    even, saturate at 448); the oracle emulates both quantisation points.
  * Everything else is exact fp64 over the exactly decoded inputs.

Sigmoid keys are computed in fp64 here and in fp32 on the GPU, so a token
whose selection hinges on two keys closer than NEAR_TIE is flagged as
ambiguous; either choice is then accepted (the forward can be re-run with the
other side's ids for those tokens).
"""
from __future__ import annotations

import dataclasses
import time

import numpy as np

from .codecs import (decode_bf16, decode_e4m3, decode_int4_grouped, decode_int4_grouped_zp, decode_int8_grouped,
                     decode_int8_grouped_zp, dynamic_scale, encode_bf16, encode_e4m3)

NEAR_TIE = 4e-6


@dataclasses.dataclass(frozen=True)
class Problem:
    T: int
    H: int
    I: int
    E: int
    top_k: int
    scoring: str = "softmax"          # "softmax" | "sigmoid"
    renormalize: bool = True
    n_group: int = 0
    topk_group: int = 0
    routed_scaling_factor: float = 1.0
    wdtype: str = "bf16"              # "bf16" | "fp8" | "int4" | "int8"
    group_size: int = 128
    act_scale: str = "static"         # fp8: "static" (given a1, a2) | "dynamic" (per-tensor amax)

    @property
    def dynamic(self) -> bool:
        return self.wdtype == "fp8" and self.act_scale == "dynamic"

    @property
    def S(self) -> int:
        return self.T * self.top_k


# --------------------------------------------------------------------------- gate

def _topk_desc_lower_index(keys: np.ndarray, k: int) -> np.ndarray:
    """Per row: indices of the k largest keys, descending, ties -> lower index."""
    T, E = keys.shape
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -keys), axis=-1)
    return order[:, :k]


def logits_fp64(logits: np.ndarray) -> np.ndarray:
    """Router logits as float64, a NaN read as -infinity.

    The pages say nothing about NaN logits.  Reading: a NaN logit is an expert
    the router scores lowest, i.e. -inf: softmax probability 0 (and left out of
    the normalising sum), sigmoid score 0, selection key of a -inf logit (with
    a bias the key is then the bias alone).  Rows must keep at least one finite
    logit for the softmax to be defined.  When renormalisation meets selected
    scores that are all zero (every selected logit NaN: with groups, a row's
    finite experts may all sit in groups that lost), the weights are zero."""
    l = np.asarray(logits, dtype=np.float64)
    return np.where(np.isnan(l), -np.inf, l)


def softmax_fp64(logits: np.ndarray) -> np.ndarray:
    l = logits_fp64(logits)
    m = l.max(axis=1, keepdims=True)
    z = np.exp(l - m)
    return z / z.sum(axis=1, keepdims=True)


def sigmoid_fp64(logits: np.ndarray) -> np.ndarray:
    l = logits_fp64(logits)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def _keys(p: Problem, logits: np.ndarray, bias):
    l = logits_fp64(logits)
    if p.scoring == "softmax":
        return l, True
    if p.n_group == 0 and bias is None:
        return l, True
    c = sigmoid_fp64(l)
    if bias is not None:
        c = c + np.asarray(bias, dtype=np.float64)[None, :]
    return c, False


def group_scores(p: Problem, keys: np.ndarray) -> np.ndarray:
    """Sum of the two largest keys in each contiguous group of E/n_group experts."""
    T = keys.shape[0]
    gs = p.E // p.n_group
    c = keys.reshape(T, p.n_group, gs)
    top = -np.sort(-c, axis=-1)[..., : min(2, gs)]
    return top.sum(axis=-1)


def gate_select(p: Problem, logits: np.ndarray, bias=None):
    """Returns (ids int32 [T,k], ambiguous bool [T]).

    ids are ordered by key descending, ties to the lower expert index.
    """
    T = logits.shape[0]
    keys, exact = _keys(p, logits, bias)
    amb = np.zeros(T, dtype=bool)
    if p.n_group > 0:
        gsc = group_scores(p, keys)
        g_order = _topk_desc_lower_index(gsc, p.n_group)
        kept = g_order[:, : p.topk_group]
        mask = np.zeros((T, p.n_group), dtype=bool)
        np.put_along_axis(mask, kept, True, axis=1)
        emask = np.repeat(mask, p.E // p.n_group, axis=1)
        keys = np.where(emask, keys, -np.inf)
        if not exact and p.topk_group < p.n_group:
            srt = np.take_along_axis(gsc, g_order, axis=1)
            gap = srt[:, p.topk_group - 1] - srt[:, p.topk_group]
            amb |= gap < NEAR_TIE
    ids = _topk_desc_lower_index(keys, p.top_k)
    if not exact:
        m = min(p.top_k + 1, p.E)
        full = _topk_desc_lower_index(keys, m)
        srt = np.take_along_axis(keys, full, axis=1)
        fin = np.isfinite(srt)
        gaps = srt[:, :-1] - srt[:, 1:]
        both = fin[:, :-1] & fin[:, 1:]
        amb |= np.any((gaps < NEAR_TIE) & both, axis=1)
    return ids.astype(np.int32), amb


def gate_weights(p: Problem, logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Top-k weights (float64 [T,k]) for the given ids."""
    if p.scoring == "softmax":
        score = softmax_fp64(logits)
    else:
        score = sigmoid_fp64(logits)
    w = np.take_along_axis(score, ids.astype(np.int64), axis=1)
    if p.renormalize:
        # a token whose selected scores are all zero (possible only when every
        # selected logit is NaN) gets zero weights rather than 0 / 0
        tot = w.sum(axis=1, keepdims=True)
        w = np.divide(w, tot, out=np.zeros_like(w), where=tot > 0)
    return w * float(p.routed_scaling_factor)


def gate(p: Problem, logits: np.ndarray, bias=None):
    ids, amb = gate_select(p, logits, bias)
    return ids, gate_weights(p, logits, ids), amb


# ------------------------------------------------------------------ align/permute

def align(ids: np.ndarray, E: int):
    """Stable counting sort of the flat slots f = t*k + j by expert id.

    Returns counts[E], offsets[E+1] (exclusive prefix sum), perm[S] (row ->
    slot: the r-th slot, in ascending f, routed to e sits at row offsets[e]+r)
    and inv[S] (slot -> row).
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    S = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.empty(S, dtype=np.int64)
    for f in range(S):
        e = flat[f]
        perm[fill[e]] = f
        fill[e] += 1
    inv = np.empty(S, dtype=np.int64)
    inv[perm] = np.arange(S)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv.astype(np.int32))


def align_block_size(counts: np.ndarray, offsets: np.ndarray, perm: np.ndarray, block: int):
    """Padded view of the sorted slots (the moe_align_block_size layout).

    Each expert's segment is padded up to a multiple of `block`; padding holds
    the sentinel S.  Returns sorted_ids[total], block_expert[total/block],
    total (= sum of the padded segment lengths).
    """
    E = counts.size
    S = int(perm.size)
    padded = [((int(c) + block - 1) // block) * block for c in counts]
    total = int(sum(padded))
    sorted_ids = np.full(total, S, dtype=np.int32)
    block_expert = np.empty(total // block, dtype=np.int32)
    pos = 0
    for e in range(E):
        c = int(counts[e])
        sorted_ids[pos: pos + c] = perm[offsets[e]: offsets[e] + c]
        block_expert[pos // block: (pos + padded[e]) // block] = e
        pos += padded[e]
    return sorted_ids, block_expert, total


# --------------------------------------------------------------------- experts

class ExpertWeights:
    """Decodes one expert's weights to exact float64 on demand."""

    def __init__(self, p: Problem, w13, w2, w13_scale=None, w2_scale=None, w13_zero=None, w2_zero=None):
        self.p = p
        self.w13, self.w2 = w13, w2
        self.s13, self.s2 = w13_scale, w2_scale
        self.z13, self.z2 = w13_zero, w2_zero  # int4 / int8 zero points (None: signed codes)
        self.prep_seconds = 0.0

    def __call__(self, e: int):
        t0 = time.perf_counter()
        p = self.p
        if p.wdtype == "bf16":
            W13 = decode_bf16(self.w13[e])
            W2 = decode_bf16(self.w2[e])
        elif p.wdtype == "fp8":
            W13 = decode_e4m3(self.w13[e]) * float(np.float32(self.s13[e]))
            W2 = decode_e4m3(self.w2[e]) * float(np.float32(self.s2[e]))
        elif p.wdtype == "int4" and self.z13 is not None:
            W13 = decode_int4_grouped_zp(self.w13[e], self.s13[e], self.z13[e], p.group_size)
            W2 = decode_int4_grouped_zp(self.w2[e], self.s2[e], self.z2[e], p.group_size)
        elif p.wdtype == "int4":
            W13 = decode_int4_grouped(self.w13[e], self.s13[e], p.group_size)
            W2 = decode_int4_grouped(self.w2[e], self.s2[e], p.group_size)
        elif p.wdtype == "int8" and self.z13 is not None:
            W13 = decode_int8_grouped_zp(self.w13[e], self.s13[e], self.z13[e], p.group_size)
            W2 = decode_int8_grouped_zp(self.w2[e], self.s2[e], self.z2[e], p.group_size)
        elif p.wdtype == "int8":
            W13 = decode_int8_grouped(self.w13[e], self.s13[e], p.group_size)
            W2 = decode_int8_grouped(self.w2[e], self.s2[e], p.group_size)
        else:
            raise ValueError(p.wdtype)
        self.prep_seconds += time.perf_counter() - t0
        return W13, W2


def quantize_fp8(values: np.ndarray, scale) -> np.ndarray:
    """e4m3 codes of value/scale, the division done in float32."""
    v32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    q32 = v32 / np.float32(scale)
    return encode_e4m3(q32)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_act(p: Problem, X: np.ndarray, W13: np.ndarray) -> np.ndarray:
    """act = silu(X W1^T) * (X W3^T), with W1 = W13[:I], W3 = W13[I:] (fp64)."""
    h = X @ W13.T
    I = p.I
    return silu(h[:, :I]) * h[:, I:]


def quantize_act(p: Problem, act: np.ndarray, a2) -> np.ndarray:
    """The second quantisation point of the fp8 W8A8 path: act as the down
    GEMM reads it.  Static: e4m3(act / a2) * a2.  Dynamic: act is first stored
    in bf16 (the pages' fused-MoE code keeps the SwiGLU output in the model
    dtype and quantises it in a separate pass), then e4m3(bf16(act) / a2) * a2
    with a2 the dynamic scale of the whole bf16 tensor."""
    if p.wdtype != "fp8":
        return act
    a2f = float(np.float32(a2))
    if p.dynamic:
        act = decode_bf16(encode_bf16(act))
    return decode_e4m3(quantize_fp8(act, a2f)) * a2f


def gate_up_swiglu(p: Problem, X: np.ndarray, W13: np.ndarray, a2=None) -> np.ndarray:
    """SwiGLU activation of one expert's rows as the down GEMM reads it (fp8:
    quantised with a2, see quantize_act)."""
    return quantize_act(p, swiglu_act(p, X, W13), a2)


def down(act: np.ndarray, W2: np.ndarray) -> np.ndarray:
    return act @ W2.T


def input_rows(p: Problem, x_bits: np.ndarray, a1=None) -> np.ndarray:
    """Token rows as the GEMMs see them: exact bf16, or e4m3(x/a1)*a1 for fp8."""
    x = decode_bf16(x_bits)
    if p.wdtype == "fp8":
        a1f = float(np.float32(a1))
        return decode_e4m3(quantize_fp8(x, a1f)) * a1f
    return x


def reduce(p: Problem, y_perm: np.ndarray, inv: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t] = sum_j w[t,j] * y_perm[inv[t*k+j]], summed in j order."""
    T, k = p.T, p.top_k
    inv2 = np.asarray(inv, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j: j + 1] * y_perm[inv2[:, j]]
    return out


def forward(p: Problem, x_bits, logits, bias, experts: ExpertWeights, a1=None, a2=None,
            ids=None, stats: dict | None = None):
    """Whole layer.  Returns a dict with every intermediate.

    `ids` overrides the gate's selection (weights are recomputed for them), for
    tokens flagged as near-ties.  `stats` receives compute and weight-decode
    seconds separately.  Dynamic fp8 scales (p.dynamic) ignore a1 / a2 and use
    a1 = dynamic_scale(x) over all T tokens and a2 = dynamic_scale(bf16(act))
    over all S rows; both are returned.
    """
    t0 = time.perf_counter()
    prep0 = experts.prep_seconds
    sel, amb = gate_select(p, logits, bias)
    if ids is None:
        ids = sel
    w = gate_weights(p, logits, ids)
    counts, offsets, perm, inv = align(ids, p.E)
    if p.dynamic:
        a1 = dynamic_scale(decode_bf16(x_bits))
    X = input_rows(p, x_bits, a1)
    x_perm = X[np.asarray(perm, dtype=np.int64) // p.top_k]
    act = np.zeros((p.S, p.I), dtype=np.float64)
    y_perm = np.zeros((p.S, p.H), dtype=np.float64)
    W2s = {}
    for e in range(p.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        W13, W2s[e] = experts(e)
        act[lo:hi] = swiglu_act(p, x_perm[lo:hi], W13)
    if p.dynamic:
        a2 = dynamic_scale(decode_bf16(encode_bf16(act)))
    act = quantize_act(p, act, a2)
    for e, W2 in W2s.items():
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        y_perm[lo:hi] = down(act[lo:hi], W2)
    out = reduce(p, y_perm, inv, w)
    if stats is not None:
        total = time.perf_counter() - t0
        prep = experts.prep_seconds - prep0
        stats["seconds"] = total - prep
        stats["prep_seconds"] = prep
    return dict(ids=ids, w=w, ambiguous=amb, selected=sel, counts=counts, offsets=offsets,
                perm=perm, inv=inv, x_perm=x_perm, act=act, y_perm=y_perm, out=out, a1=a1, a2=a2)


def token_outputs(p: Problem, tokens, x_bits, logits, bias, experts: ExpertWeights,
                  a1=None, a2=None, ids=None):
    """Output rows for a subset of tokens only (per-token definition, no permute).

    out[t] = sum_j w[t,j] * MLP_{ids[t,j]}(x_t); used to check sampled rows of
    full-size runs.  `ids`, if given, is the full [T,k] id array to use.  With
    dynamic fp8 scales the caller passes a1 and a2 (they depend on the whole
    batch); a2 = None then skips the second quantisation (act kept exact).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    lg = np.asarray(logits)[tokens]
    if ids is None:
        sel, _ = gate_select(p, lg, bias)
    else:
        sel = np.asarray(ids)[tokens]
    w = gate_weights(p, lg, sel)
    X = input_rows(p, np.asarray(x_bits)[tokens], a1)
    out = np.zeros((tokens.size, p.H), dtype=np.float64)
    for e in np.unique(sel):
        W13, W2 = experts(int(e))
        rows, cols = np.nonzero(sel == e)
        act = swiglu_act(p, X[rows], W13)
        if not (p.dynamic and a2 is None):
            act = quantize_act(p, act, a2)
        y = down(act, W2)
        for r, c, yy in zip(rows, cols, y):
            out[r] += w[r, c] * yy
    return out
