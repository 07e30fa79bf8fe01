"""Pins for the oracle's bf16 rounding and the dynamic per-tensor fp8 scales.

Anchors: torch's float32 -> bfloat16 cast (round to nearest even), closed-form
roundings that a detour through float32 would get wrong, the scale's closed
form, and a dense brute-force layer that quantises with one global amax over
every (token, selected expert) pair.
"""
import dataclasses

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import Problem
from synth import SHAPES, make_weights, make_tokens, shrink
from oracle.torch_io import oracle_inputs


def test_encode_bf16_matches_torch_cast_on_float32_values():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # every bf16 pattern, its float32 neighbours and the exact midpoints to the next pattern
    b16 = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    extra = np.concatenate([b16, b16 + 1, b16 - 1, b16 + 0x8000, b16 + 0x7FFF, b16 + 0x8001])
    f = np.concatenate([bits, extra]).view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.encode_bf16(f)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(oracle.decode_bf16(got[nan])))


def test_encode_bf16_rounds_once_from_the_exact_value():
    # b = 1 + 2^-6 (even mantissa 0b0000010); the midpoint to the next bf16 is a tie
    # that goes to b, but anything above it, however close, rounds up
    b, q = 1.0 + 2.0 ** -6, 2.0 ** -7
    mid = b + q / 2
    assert oracle.decode_bf16(oracle.encode_bf16(np.array([mid])))[0] == b
    assert oracle.decode_bf16(oracle.encode_bf16(np.array([mid + 2.0 ** -40])))[0] == b + q
    assert oracle.decode_bf16(oracle.encode_bf16(np.array([-(mid + 2.0 ** -40)])))[0] == -(b + q)
    # (float32 would first round mid + 2^-40 to mid, then tie to b)
    assert np.float32(mid + 2.0 ** -40) == np.float32(mid)


def test_encode_bf16_overflow_and_small_values():
    top = (2.0 - 2.0 ** -7) * 2.0 ** 127          # largest finite bf16
    mid = (2.0 - 2.0 ** -8) * 2.0 ** 127          # halfway to 2^128: ties to even = infinity
    got = oracle.decode_bf16(oracle.encode_bf16(np.array([top, mid, mid * (1 - 2.0 ** -30), 2.0 ** -133, 0.0])))
    assert got[0] == top and np.isinf(got[1]) and got[2] == top
    assert got[3] == 2.0 ** -133 and got[4] == 0.0


def test_dynamic_scale_closed_forms():
    assert oracle.dynamic_scale(np.array([0.0, -3.5, 2.0])) == 3.5 / 448.0
    assert oracle.dynamic_scale(np.zeros(7)) == 1.0
    assert oracle.dynamic_scale(np.zeros(0)) == 1.0
    # float32 division: 1/448 is not exact in binary; the scale is the float32 quotient
    assert oracle.dynamic_scale(np.array([1.0])) == float(np.float32(1.0) / np.float32(448.0))


def _dynamic_shape():
    return dataclasses.replace(shrink(SHAPES["qwen2"], H=128, I=64, E=8), top_k=3, act_scale="dynamic")


def _dense_dynamic_bruteforce(p, x, ids, w, W13s, W2s):
    """One row per (token, slot), no permutation: x quantised with a1 = amax(x)/448,
    every selected pair's SwiGLU output rounded to bf16, one amax over all pairs."""
    T, k, I = p.T, p.top_k, p.I
    a1 = np.float32(np.abs(x).max()) / np.float32(448.0)
    xq = np.array([[float(oracle.decode_e4m3(oracle.encode_e4m3(np.float32(v) / a1))) * float(a1)
                    for v in row] for row in x])
    acts = {}
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            g = W13s[e][:I] @ xq[t]
            u = W13s[e][I:] @ xq[t]
            acts[t, j] = oracle.decode_bf16(oracle.encode_bf16(g * scipy.special.expit(g) * u))
    a2 = np.float32(max(np.abs(a).max() for a in acts.values())) / np.float32(448.0)
    out = np.zeros((T, p.H))
    for (t, j), a in acts.items():
        aq = oracle.decode_e4m3(oracle.encode_e4m3(a.astype(np.float32) / a2)) * float(a2)
        out[t] += w[t, j] * (W2s[ids[t, j]] @ aq)
    return out, float(a1), float(a2)


def test_dynamic_forward_matches_dense_bruteforce():
    shape = _dynamic_shape()
    w = make_weights(shape, "cpu", seed=5)
    tok = make_tokens(shape, 12, "cpu", seed=5)
    p, inp = oracle_inputs(shape, w, tok)
    assert p.dynamic
    res = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"])
    x = oracle.decode_bf16(inp["x_bits"])
    W = [inp["experts"](e) for e in range(p.E)]
    ref, a1, a2 = _dense_dynamic_bruteforce(p, x, res["ids"], res["w"], [a for a, _ in W], [b for _, b in W])
    assert res["a1"] == a1 and res["a2"] == a2
    assert np.abs(res["out"] - ref).max() <= 1e-12 * np.abs(ref).max()
    # the static inputs are ignored
    res2 = oracle.forward(p, inp["x_bits"], inp["logits"], inp["bias"], inp["experts"], a1=123.0, a2=0.5)
    assert np.array_equal(res2["out"], res["out"])


def test_dynamic_scales_follow_a_power_of_two_rescaling_of_x():
    shape = _dynamic_shape()
    w = make_weights(shape, "cpu", seed=6)
    tok = make_tokens(shape, 9, "cpu", seed=6)
    p, inp = oracle_inputs(shape, w, tok)
    x = oracle.decode_bf16(inp["x_bits"])
    x4 = oracle.encode_bf16(4.0 * x)               # exact: a power of two
    r1 = oracle.forward(p, inp["x_bits"], inp["logits"], None, inp["experts"])
    r4 = oracle.forward(p, x4, inp["logits"], None, inp["experts"])
    assert r4["a1"] == 4.0 * r1["a1"]
    assert np.array_equal(r4["x_perm"], 4.0 * r1["x_perm"])   # same e4m3 codes
    # the largest |x| lands on the e4m3 maximum
    codes = oracle.quantize_fp8(x, r1["a1"])
    big = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(oracle.decode_e4m3(codes[big])) == 448.0


def test_static_problem_keeps_given_scales():
    p = Problem(T=2, H=16, I=16, E=1, top_k=1, wdtype="fp8")
    assert not p.dynamic and not dataclasses.replace(p, wdtype="bf16", act_scale="dynamic").dynamic
