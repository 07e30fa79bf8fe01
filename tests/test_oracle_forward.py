"""Pins for the oracle's expert MLP, reduce and whole-layer forward.

Anchors: the hand-derived SwiGLU fixture, a dense brute-force MoE (every expert
on every token, masked by a dense gate matrix, no permutation), the E=1/top_k=1
reduction to a plain SwiGLU MLP, and symmetry properties.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import Problem, ExpertWeights
from synth import SHAPES, make_weights, make_tokens, shrink
from oracle.torch_io import oracle_inputs, problem_for, np_of, bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    return bf16_bits(torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def test_golden_swiglu_single_expert():
    with open(os.path.join(GOLDEN, "swiglu_hand.json")) as f:
        g = json.load(f)
    H, I = g["H"], g["I"]
    x = np.array(g["x"])
    p = Problem(T=x.shape[0], H=H, I=I, E=1, top_k=1, renormalize=True)
    w13 = _bf16(g["w13"])[None]
    w2 = _bf16(g["w2"])[None]
    res = oracle.forward(p, _bf16(x), np.zeros((x.shape[0], 1), np.float32), None,
                         ExpertWeights(p, w13, w2))
    exp = np.array([[eval(s, {"e": math.e}) for s in row] for row in g["expected_out_expr"]])
    assert np.allclose(res["out"], exp, atol=g["tolerance"], rtol=0)
    assert np.all(res["w"] == 1.0)


def _dense_bruteforce(p, x, ids, w, W13s, W2s):
    """Every expert on every token, then a dense [T,E] gate matrix (zeros off top-k)."""
    T, E, I = p.T, p.E, p.I
    G = np.zeros((T, E))
    for t in range(T):
        for j in range(p.top_k):
            G[t, ids[t, j]] += w[t, j]
    out = np.zeros((T, p.H))
    for e in range(E):
        W1, W3 = W13s[e][:I], W13s[e][I:]
        for t in range(T):
            g = W1 @ x[t]
            u = W3 @ x[t]
            a = g * scipy.special.expit(g) * u
            out[t] += G[t, e] * (W2s[e] @ a)
    return out


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen2_bf16", "dsv3", "scout"])
def test_forward_matches_dense_bruteforce(name):
    if name == "qwen2_bf16":
        base = SHAPES["qwen2"]
        shape = shrink(base, H=64, I=32, E=16)
        import dataclasses
        shape = dataclasses.replace(shape, wdtype="bf16")
    else:
        shape = shrink(SHAPES[name], H=128 if name != "tiny" else 256,
                       I=128 if name != "tiny" else 512,
                       E=min(SHAPES[name].E, 32 if name == "dsv3" else 16))
        if name == "dsv3":
            import dataclasses
            shape = dataclasses.replace(shape, n_group=8, topk_group=4)
    T = 24
    w = make_weights(shape, "cpu", seed=1)
    tok = make_tokens(shape, T, "cpu", seed=1)
    p, inp = oracle_inputs(shape, w, tok)
    res = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"])
    x = oracle.decode_bf16(inp["x_bits"])
    W = [inp["experts"](e) for e in range(p.E)]
    ref = _dense_bruteforce(p, x, res["ids"], res["w"], [a for a, _ in W], [b for _, b in W])
    scale = np.abs(ref).max()
    assert scale > 0
    assert np.abs(res["out"] - ref).max() <= 1e-12 * scale


def test_single_expert_reduces_to_plain_swiglu_mlp():
    shape = shrink(SHAPES["tiny"], H=64, I=96, E=1)
    import dataclasses
    shape = dataclasses.replace(shape, top_k=1)
    w = make_weights(shape, "cpu", seed=2)
    tok = make_tokens(shape, 10, "cpu", seed=2)
    p, inp = oracle_inputs(shape, w, tok)
    res = oracle.forward(p, inp["x_bits"], inp["logits"], None, inp["experts"])
    assert np.all(res["w"] == 1.0)
    X = torch.from_numpy(oracle.decode_bf16(inp["x_bits"]))
    W13 = w.w13[0].double()
    W2 = w.w2[0].double()
    ref = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(X, W13[:96])) *
        torch.nn.functional.linear(X, W13[96:]), W2).numpy()
    assert np.abs(res["out"] - ref).max() <= 1e-12 * np.abs(ref).max()


def test_zero_input_gives_zero_output():
    shape = SHAPES["tiny"]
    w = make_weights(shape, "cpu", seed=3)
    tok = make_tokens(shape, 8, "cpu", seed=3)
    p, inp = oracle_inputs(shape, w, tok)
    zeros = np.zeros_like(inp["x_bits"])
    res = oracle.forward(p, zeros, inp["logits"], None, inp["experts"])
    assert np.all(res["out"] == 0.0)


def test_token_permutation_equivariance():
    shape = SHAPES["tiny"]
    w = make_weights(shape, "cpu", seed=4)
    tok = make_tokens(shape, 40, "cpu", seed=4)
    p, inp = oracle_inputs(shape, w, tok)
    res = oracle.forward(p, inp["x_bits"], inp["logits"], None, inp["experts"])
    pi = np.random.default_rng(4).permutation(40)
    res2 = oracle.forward(p, inp["x_bits"][pi], inp["logits"][pi], None, inp["experts"])
    assert np.abs(res2["out"] - res["out"][pi]).max() <= 1e-13 * np.abs(res["out"]).max()


def test_expert_relabelling_invariance():
    shape = shrink(SHAPES["dsv3"], H=128, I=128, E=32)
    w = make_weights(shape, "cpu", seed=5)
    tok = make_tokens(shape, 16, "cpu", seed=5)
    p, inp = oracle_inputs(shape, w, tok)
    res = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"])
    # permute experts inside each group and permute the groups: group structure kept
    gs = 4
    rng = np.random.default_rng(5)
    gperm = rng.permutation(8)
    sigma = np.concatenate([g * gs + rng.permutation(gs) for g in gperm])   # new e' -> old sigma[e']
    w13 = np_of(w.w13)[sigma]
    w2 = np_of(w.w2)[sigma]
    s13 = np_of(w.w13_scale)[sigma]
    s2 = np_of(w.w2_scale)[sigma]
    ew = ExpertWeights(p, w13, w2, s13, s2)
    res2 = oracle.forward(p, inp["x_bits"], inp["logits"][:, sigma], inp["bias"][sigma], ew)
    assert np.array_equal(sigma[res2["ids"]], res["ids"])
    assert np.abs(res2["out"] - res["out"]).max() <= 1e-13 * np.abs(res["out"]).max()


def test_fp8_exact_inputs_quantise_to_themselves():
    # x values that are e4m3 codes times a1 are left unchanged by the x quantisation
    p = Problem(T=4, H=16, I=16, E=2, top_k=1, wdtype="fp8")
    a1 = 0.5
    codes = np.arange(0, 64, dtype=np.uint8).reshape(4, 16)
    vals = oracle.decode_e4m3(codes) * a1
    bits = bf16_bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))
    assert np.array_equal(oracle.decode_bf16(bits), vals)     # exact in bf16
    assert np.array_equal(oracle.input_rows(p, bits, a1), vals)


def test_fp8_act_quantisation_is_applied_and_bounded():
    shape = shrink(SHAPES["qwen2"], H=128, I=128, E=8)
    w = make_weights(shape, "cpu", seed=6)
    tok = make_tokens(shape, 32, "cpu", seed=6)
    p, inp = oracle_inputs(shape, w, tok)
    W13, _ = inp["experts"](0)
    X = oracle.input_rows(p, inp["x_bits"], inp["a1"])
    q = oracle.gate_up_swiglu(p, X, W13, inp["a2"])
    import dataclasses
    raw = oracle.gate_up_swiglu(dataclasses.replace(p, wdtype="bf16"), X, W13)
    # every quantised value is an e4m3 value times a2, within half an e4m3 step (1/16 rel)
    a2 = inp["a2"]
    assert np.all(np.isin(np.round(q / a2, 9), np.round(oracle.decode_e4m3(np.arange(256, dtype=np.uint8)), 9)))
    big = np.abs(raw) > 2 ** -6 * a2
    assert np.all(np.abs(q - raw)[big] <= np.abs(raw)[big] / 16 + 1e-12)
    assert not np.array_equal(q, raw)


def test_token_outputs_match_forward_rows():
    for name in ("tiny", "dsv3"):
        shape = SHAPES[name] if name == "tiny" else shrink(SHAPES[name], H=256, I=128, E=32)
        if name == "dsv3":
            import dataclasses
            shape = dataclasses.replace(shape, n_group=8, topk_group=4)
        w = make_weights(shape, "cpu", seed=7)
        tok = make_tokens(shape, 20, "cpu", seed=7)
        p, inp = oracle_inputs(shape, w, tok)
        res = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"])
        rows = np.array([0, 5, 19])
        out = oracle.token_outputs(p, rows, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"])
        assert np.abs(out - res["out"][rows]).max() <= 1e-13 * np.abs(res["out"]).max()


def test_forward_stats_split_prep_from_compute():
    shape = SHAPES["tiny"]
    w = make_weights(shape, "cpu", seed=8)
    tok = make_tokens(shape, 64, "cpu", seed=0)
    p, inp = oracle_inputs(shape, w, tok)
    st = {}
    oracle.forward(p, inp["x_bits"], inp["logits"], None, inp["experts"], stats=st)
    assert st["seconds"] > 0 and st["prep_seconds"] > 0
