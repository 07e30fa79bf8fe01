"""Helpers for the GPU parity tests: run every stage through the C ABI and
compare against the oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import mixture_experts_layer_gate_gb300 as moe
import oracle
from synth import make_tokens, make_weights
from oracle.torch_io import np_of, oracle_inputs

TOL = {"bf16": 1e-2, "fp8": 3e-2, "int4": 4e-2, "int8": 2e-2}


def lib_wdtype(shape):
    # int4 weights the library receives prepared by moe_repack_int4
    return "int4_paired" if shape.int4_order == "paired" else shape.wdtype


def lib_problem(shape, T):
    return moe.problem(T, shape.H, shape.I, shape.E, shape.top_k, scoring=shape.scoring,
                       renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                       routed_scaling_factor=shape.routed_scaling_factor, wdtype=lib_wdtype(shape),
                       group_size=shape.group_size, act_scale=shape.act_scale)


def lib_weights(w, tok, shape=None):
    # the oracle reads the generated (packed) codes; the library a repacked copy
    # where the shape asks for the paired format
    w13, w2 = w.w13, w.w2
    if shape is not None and shape.int4_order == "paired":
        w13, w2 = moe.repack_int4(w.w13), moe.repack_int4(w.w2)
    return moe.Weights(w13, w2, w.w13_scale, w.w2_scale, tok.a1_scale, tok.a2_scale,
                       w.w13_zero, w.w2_zero)


@dataclasses.dataclass
class StageOut:
    ids: torch.Tensor
    w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv: torch.Tensor
    x_perm: torch.Tensor
    act: torch.Tensor
    y_perm: torch.Tensor
    out: torch.Tensor
    out_forward: torch.Tensor
    scales: np.ndarray | None = None  # dynamic fp8: {a1, a2} of the staged run (float32)


def run_stages(shape, T, weights, tok, device) -> StageOut:
    p = lib_problem(shape, T)
    wts = lib_weights(weights, tok, shape)
    k, S, H, I, E = shape.top_k, T * shape.top_k, shape.H, shape.I, shape.E
    adt = torch.uint8 if shape.wdtype == "fp8" else torch.bfloat16
    ids = torch.full((T, k), -1, dtype=torch.int32, device=device)
    w = torch.zeros((T, k), dtype=torch.float32, device=device)
    counts = torch.full((E,), -1, dtype=torch.int32, device=device)
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device=device)
    perm = torch.full((S,), -1, dtype=torch.int32, device=device)
    inv = torch.full((S,), -1, dtype=torch.int32, device=device)
    x_perm = torch.zeros((S, H), dtype=adt, device=device)
    act = torch.zeros((S, I), dtype=adt, device=device)
    y_perm = torch.zeros((S, H), dtype=torch.bfloat16, device=device)
    out = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
    out_f = torch.zeros((T, H), dtype=torch.bfloat16, device=device)
    ws = moe.alloc_workspace(p, device, full=False)
    moe.gate_topk(p, tok.logits, tok.bias, ids, w)
    moe.align_permute(p, ids, tok.x, tok.a1_scale, counts, offsets, perm, inv, x_perm, ws)
    moe.grouped_gemm_swiglu(p, wts, x_perm, offsets, act, ws)
    moe.grouped_gemm_down(p, wts, act, offsets, y_perm, ws)
    moe.unpermute_reduce(p, y_perm, inv, w, out, ws)
    assert moe.get_device_error(ws) == 0
    wsf = moe.alloc_workspace(p, device, full=True)
    moe.forward(p, wts, tok.x, tok.logits, tok.bias, out_f, wsf)
    assert moe.get_device_error(wsf) == 0
    torch.cuda.synchronize()
    scales = None
    if shape.act_scale == "dynamic":
        scales = moe.dynamic_scales(ws).cpu().numpy()
        assert np.array_equal(scales, moe.dynamic_scales(wsf).cpu().numpy())
    return StageOut(ids, w, counts, offsets, perm, inv, x_perm, act, y_perm, out, out_f, scales)


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / scale)


def to_f64(t: torch.Tensor, wdtype: str, scale=None) -> np.ndarray:
    """bf16 tensor -> exact float64; e4m3 codes (uint8) -> decoded * scale."""
    if t.dtype == torch.uint8:
        v = oracle.decode_e4m3(t.cpu().numpy())
        return v * (1.0 if scale is None else float(np.float32(scale)))
    return t.float().cpu().numpy().astype(np.float64)


def check_gate(shape, T, tok, g: StageOut):
    """ids bit-exact except near-ties (where any valid choice is accepted);
    weights to 1e-5 relative for the GPU's ids.  Returns the ids to use."""
    p, inp = oracle_inputs(shape, _NoWeights(), tok)
    ids_o, amb = oracle.gate_select(p, inp["logits"], inp["bias"])
    ids_g = g.ids.cpu().numpy()
    assert ids_g.min() >= 0 and ids_g.max() < shape.E
    for row in ids_g:
        assert len(set(row.tolist())) == shape.top_k
    mism = np.any(ids_o != ids_g, axis=1)
    assert not np.any(mism & ~amb), f"ids differ on unflagged tokens {np.nonzero(mism & ~amb)[0][:10]}"
    w_o = oracle.gate_weights(p, inp["logits"], ids_g)
    w_g = g.w.cpu().numpy().astype(np.float64)
    assert np.allclose(w_g, w_o, rtol=1e-5, atol=1e-7), np.abs(w_g - w_o).max()
    return ids_g, int(mism.sum()), int(amb.sum())


def check_align(shape, ids_g, g: StageOut):
    counts, offsets, perm, inv = oracle.align(ids_g, shape.E)
    assert np.array_equal(g.counts.cpu().numpy(), counts)
    assert np.array_equal(g.offsets.cpu().numpy(), offsets)
    assert np.array_equal(g.perm.cpu().numpy(), perm)
    assert np.array_equal(g.inv.cpu().numpy(), inv)
    return counts, offsets, perm, inv


class _NoWeights:
    w13 = w2 = w13_scale = w2_scale = w13_zero = w2_zero = None


def plant_nan_logits(tok, frac, seed):
    """Sets a seeded fraction of the router logits to NaN, keeping one finite
    logit per row (column t mod E) so every softmax row stays defined; a few
    rows lose all but that one, so NaN experts get selected there."""
    T, E = tok.logits.shape
    g = torch.Generator(device="cpu")
    g.manual_seed(1234 + seed)
    mask = torch.rand((T, E), generator=g) < frac
    mask[: max(1, T // 16)] = True
    mask[torch.arange(T), torch.arange(T) % E] = False
    tok.logits[mask.to(tok.logits.device)] = float("nan")
    return int(mask.sum())


def full_check(shape, T, device, seed=0, check_stages=True, nan_logits=0.0):
    """Whole-layer parity on a size the oracle computes completely."""
    w = make_weights(shape, device, seed)
    tok = make_tokens(shape, T, device, seed)
    if nan_logits:
        plant_nan_logits(tok, nan_logits, seed)
    g = run_stages(shape, T, w, tok, device)
    assert torch.equal(g.out, g.out_forward), "moe_forward differs from the staged calls"
    ids_g, n_mism, n_amb = check_gate(shape, T, tok, g)
    counts, offsets, perm, inv = check_align(shape, ids_g, g)
    p, inp = oracle_inputs(shape, w, tok)
    res = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"], inp["a1"],
                         inp["a2"], ids=ids_g)
    tol = TOL[shape.wdtype]
    a1, a2 = inp["a1"], inp["a2"]
    a2_g = a2
    if shape.act_scale == "dynamic":
        # a1 = amax(x) / 448: exact on both sides; a2 from the bf16 SwiGLU output,
        # whose largest element may round to a neighbouring bf16 on the GPU
        a1, a2 = res["a1"], res["a2"]
        assert np.float32(g.scales[0]) == np.float32(a1), (g.scales[0], a1)
        a2_g = float(g.scales[1])
        assert abs(a2_g - a2) <= 2.0 ** -7 * a2, (a2_g, a2)
    if check_stages:
        # x_perm: exact copy (bf16) or exact e4m3 codes of x / a1
        xg = g.x_perm.cpu()
        if shape.wdtype == "fp8":
            codes = oracle.quantize_fp8(oracle.decode_bf16(inp["x_bits"]), a1)
            assert np.array_equal(xg.numpy(), codes[perm // shape.top_k])
        else:
            assert np.array_equal(to_f64(xg, "bf16"), oracle.decode_bf16(inp["x_bits"])[perm // shape.top_k])
        # act from the same x_perm
        act_g = to_f64(g.act, shape.wdtype, a2_g)
        if shape.wdtype == "fp8":
            # compare in e4m3 steps (each side's codes): neighbours allowed on a small
            # fraction.  Near zero the code is decided by the gate_up sums' own error
            # (the e4m3 tensor-core product accumulates thousands of terms in its
            # internal precision; the oracle is exact), not by the rounding: there a
            # difference of up to 2^-7 (four subnormal steps, in units of a2) is
            # accepted instead of one step.
            vals = np.sort(oracle.decode_e4m3(np.arange(256, dtype=np.uint8)))
            vals = vals[np.isfinite(vals)]
            sg = act_g / float(np.float32(a2_g))
            so = res["act"] / float(np.float32(a2))
            idx_g = np.searchsorted(vals, sg)
            idx_o = np.searchsorted(vals, so)
            diff = np.abs(idx_g - idx_o)
            near_zero = np.abs(sg - so) <= 2.0 ** -7
            assert diff[~near_zero].max(initial=0) <= 1, diff[~near_zero].max(initial=0)
            assert np.mean(diff > 0) < 0.02, np.mean(diff > 0)
        else:
            assert rel_err(act_g, res["act"]) <= tol, rel_err(act_g, res["act"])
        # y_perm against the oracle's own
        assert rel_err(to_f64(g.y_perm, "bf16"), res["y_perm"]) <= tol, \
            rel_err(to_f64(g.y_perm, "bf16"), res["y_perm"])
    err = rel_err(to_f64(g.out, "bf16"), res["out"])
    assert err <= tol, f"{shape.name} T={T}: out rel err {err}"
    return dict(err=err, mism=n_mism, amb=n_amb, counts=counts)


def sampled_check(shape, T, device, n_sample=4, seed=0):
    """Full-size parity: gate and align on every token, output on sampled tokens."""
    w = make_weights(shape, device, seed)
    tok = make_tokens(shape, T, device, seed)
    g = run_stages(shape, T, w, tok, device)
    assert torch.equal(g.out, g.out_forward)
    ids_g, n_mism, n_amb = check_gate(shape, T, tok, g)
    counts, offsets, perm, inv = check_align(shape, ids_g, g)
    p, inp = oracle_inputs(shape, w, tok)
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, size=n_sample)]))
    a1, a2 = inp["a1"], inp["a2"]
    if shape.act_scale == "dynamic":
        # a1 depends on x alone: exact.  a2 needs every row's activation, so only
        # a bound holds here: it covers the sampled tokens' bf16 activations;
        # the sampled outputs are compared with the activation unquantised.
        a1 = oracle.dynamic_scale(oracle.decode_bf16(inp["x_bits"]))
        assert np.float32(g.scales[0]) == np.float32(a1)
        X = oracle.input_rows(p, inp["x_bits"][rows], a1)
        sel = ids_g[rows]
        amax = 0.0
        for e in np.unique(sel):
            W13, _ = inp["experts"](int(e))
            r, _ = np.nonzero(sel == e)
            act = oracle.decode_bf16(oracle.encode_bf16(oracle.swiglu_act(p, X[r], W13)))
            amax = max(amax, float(np.abs(act).max()))
        assert float(g.scales[1]) * 448.0 >= amax * (1 - 2.0 ** -7), (g.scales[1], amax)
        a2 = None
    ref = oracle.token_outputs(p, rows, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"],
                               a1, a2, ids=ids_g)
    got = to_f64(g.out[torch.as_tensor(rows, device=device)], "bf16")
    err = rel_err(got, ref)
    assert err <= TOL[shape.wdtype], f"{shape.name} T={T}: sampled out rel err {err}"
    return dict(err=err, mism=n_mism, amb=n_amb, counts=counts)
