"""Pins for the oracle's gate and align/permute stages.

Each check rests on something other than the oracle's own formula: hand-derived
closed forms (tests/golden), brute-force enumeration of every candidate subset,
library routines (scipy softmax / expit, numpy stable argsort) and invariants.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import Problem
from synth import SHAPES, make_tokens

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _expr(s):
    return float(eval(s, {"ln": math.log, "e": math.e}))


def _prob(E, k, **kw):
    return Problem(T=1, H=128, I=128, E=E, top_k=k, **kw)


# ----------------------------------------------------------------- closed forms

def test_golden_softmax_gate():
    g = _load("gate_softmax_closed_form.json")
    l = np.array([[_expr(s) for s in g["logits_expr"]]], dtype=np.float32)
    for renorm, key in ((True, "expected_w_renormalized"), (False, "expected_w_raw")):
        ids, w, amb = oracle.gate(_prob(4, g["top_k"], renormalize=renorm), l)
        assert ids[0].tolist() == g["expected_ids"]
        assert np.allclose(w[0], [_expr(s) for s in g[key]], atol=g["tolerance"], rtol=0)
        assert not amb.any()


def test_golden_sigmoid_grouped_gate():
    g = _load("gate_sigmoid_grouped_hand.json")
    l = np.array([[_expr(s) for s in g["logits_expr"]]], dtype=np.float32)
    bias = np.array(g["bias"], dtype=np.float32)
    p = _prob(g["E"], g["top_k"], scoring="sigmoid", renormalize=True, n_group=g["n_group"],
              topk_group=g["topk_group"], routed_scaling_factor=g["routed_scaling_factor"])
    ids, w, _ = oracle.gate(p, l, bias)
    assert ids[0].tolist() == g["expected_ids"]
    assert np.allclose(w[0], g["expected_w"], atol=g["tolerance"], rtol=0)


def test_all_equal_logits():
    l = np.zeros((3, 8), dtype=np.float32)
    ids, w, _ = oracle.gate(_prob(8, 3, renormalize=True), l)
    assert (ids == np.array([0, 1, 2])).all()
    assert np.allclose(w, 1.0 / 3.0, rtol=0, atol=1e-15)
    ids, w, _ = oracle.gate(_prob(8, 3, renormalize=False), l)
    assert np.allclose(w, 1.0 / 8.0, rtol=0, atol=1e-15)


def test_one_hot_logit_goes_first():
    rng = np.random.default_rng(1)
    for e in range(8):
        l = rng.standard_normal((1, 8)).astype(np.float32)
        l[0, e] = 50.0
        ids, w, _ = oracle.gate(_prob(8, 2, renormalize=False), l)
        assert ids[0, 0] == e
        assert w[0, 0] > 0.999


def test_softmax_and_sigmoid_match_scipy():
    rng = np.random.default_rng(2)
    l = (rng.standard_normal((64, 64)) * 3).astype(np.float32)
    assert np.allclose(oracle.softmax_fp64(l), scipy.special.softmax(l.astype(np.float64), axis=1),
                       rtol=1e-13, atol=0)
    assert np.allclose(oracle.sigmoid_fp64(l), scipy.special.expit(l.astype(np.float64)),
                       rtol=1e-13, atol=0)


# ----------------------------------------------------------------- brute force

def _best_subset(keys, k):
    """Brute force: the k-subset with the largest key sum (unique for distinct keys)."""
    best, best_s = None, -np.inf
    for c in itertools.combinations(range(keys.size), k):
        s = keys[list(c)].sum()
        if s > best_s:
            best, best_s = c, s
    return set(best)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_softmax_topk_brute_force(k):
    rng = np.random.default_rng(10 + k)
    l = rng.standard_normal((200, 8)).astype(np.float32)
    ids, w, _ = oracle.gate(_prob(8, k, renormalize=True), l)
    p = scipy.special.softmax(l.astype(np.float64), axis=1)
    for t in range(l.shape[0]):
        assert set(ids[t].tolist()) == _best_subset(l[t].astype(np.float64), k)
        # descending order of logits inside the selection
        assert np.all(np.diff(l[t, ids[t]]) <= 0)
        assert np.allclose(w[t], p[t, ids[t]] / p[t, ids[t]].sum(), rtol=1e-14)


def test_grouped_sigmoid_brute_force():
    E, n_group, topk_group, k = 16, 4, 2, 3
    gs = E // n_group
    rng = np.random.default_rng(20)
    l = rng.standard_normal((150, E)).astype(np.float32)
    bias = (rng.uniform(-0.1, 0.1, E)).astype(np.float32)
    p = _prob(E, k, scoring="sigmoid", renormalize=True, n_group=n_group, topk_group=topk_group,
              routed_scaling_factor=2.5)
    ids, w, amb = oracle.gate(p, l, bias)
    s = scipy.special.expit(l.astype(np.float64))
    c = s + bias.astype(np.float64)
    for t in range(l.shape[0]):
        # group score by brute force: best pair inside the group
        gsc = [max(c[t, g * gs + a] + c[t, g * gs + b] for a in range(gs) for b in range(gs) if a != b)
               for g in range(n_group)]
        best_groups, best = None, -np.inf
        for gc in itertools.combinations(range(n_group), topk_group):
            v = sum(gsc[g] for g in gc)
            if v > best:
                best, best_groups = v, gc
        cand = [e for g in best_groups for e in range(g * gs, (g + 1) * gs)]
        best_set, bv = None, -np.inf
        for sub in itertools.combinations(cand, k):
            v = sum(c[t, e] for e in sub)
            if v > bv:
                bv, best_set = v, set(sub)
        assert set(ids[t].tolist()) == best_set, t
        assert np.all(np.diff(c[t, ids[t]]) <= 0)
        sel = s[t, ids[t]]
        assert np.allclose(w[t], sel / sel.sum() * 2.5, rtol=1e-14)
    assert amb.sum() <= 2


def test_gate_invariants_all_shapes():
    for name, shape in SHAPES.items():
        tok = make_tokens(shape, 257, device="cpu", seed=0)
        p = Problem(T=257, H=shape.H, I=shape.I, E=shape.E, top_k=shape.top_k, scoring=shape.scoring,
                    renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                    routed_scaling_factor=shape.routed_scaling_factor, wdtype=shape.wdtype)
        bias = None if tok.bias is None else tok.bias.numpy()
        ids, w, amb = oracle.gate(p, tok.logits.numpy(), bias)
        assert ids.shape == (257, shape.top_k)
        assert ids.min() >= 0 and ids.max() < shape.E
        for row in ids:
            assert len(set(row.tolist())) == shape.top_k
        if shape.renormalize:
            assert np.allclose(w.sum(1), shape.routed_scaling_factor, rtol=1e-13)
        else:
            assert np.all(w.sum(1) <= shape.routed_scaling_factor * (1 + 1e-13))
        if shape.n_group:
            grp = ids // (shape.E // shape.n_group)
            assert max(len(set(r.tolist())) for r in grp) <= shape.topk_group
        assert amb.sum() <= 3


def test_scout_recipe_routes_forced_tokens_to_expert0():
    shape = SHAPES["scout"]
    tok = make_tokens(shape, 1000, device="cpu", seed=0)
    p = Problem(T=1000, H=shape.H, I=shape.I, E=16, top_k=1, scoring="sigmoid", renormalize=False)
    ids, w, amb = oracle.gate(p, tok.logits.numpy())
    forced = tok.forced.numpy()
    assert forced.size == 500
    assert np.all(ids[forced, 0] == 0)
    share0 = np.mean(ids[:, 0] == 0)
    assert 0.45 < share0 < 0.62
    l = tok.logits.numpy().astype(np.float64)
    assert np.allclose(w[:, 0], scipy.special.expit(l[np.arange(1000), ids[:, 0]]), rtol=1e-14)
    assert not amb.any()


def test_near_tie_is_flagged():
    p = _prob(8, 2, scoring="sigmoid", renormalize=True, n_group=4, topk_group=2)
    l = np.zeros((1, 8), dtype=np.float32)
    bias = np.array([0.3, 0.0, 0.2, 0.0, 0.1, 0.0, 0.0, 0.0], dtype=np.float32)
    l2 = l.copy()
    l2[0, 4] = np.float32(1e-6)   # sigmoid gap ~2.5e-7 against nothing at the boundary
    _, amb = oracle.gate_select(p, l, bias)
    assert not amb.any()
    bias_tie = np.array([0.3, 0.0, 0.2, 0.0, 0.2, 0.0, 0.0, 0.0], dtype=np.float32)
    _, amb = oracle.gate_select(p, l, bias_tie)   # groups 1 and 2 tie exactly
    assert amb.all()


# ---------------------------------------------------------------- align/permute

def test_golden_align():
    g = _load("align_hand.json")
    ids = np.array(g["ids"], dtype=np.int32)
    counts, offsets, perm, inv = oracle.align(ids, g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm"]
    assert inv.tolist() == g["inv"]
    sorted_ids, block_expert, total = oracle.align_block_size(counts, offsets, perm, g["block"])
    assert sorted_ids.tolist() == g["sorted_ids"]
    assert block_expert.tolist() == g["block_expert"]
    assert total == g["total_padded"]


@pytest.mark.parametrize("E,k,T", [(8, 2, 1), (8, 2, 333), (64, 8, 129), (256, 8, 200), (16, 1, 77)])
def test_align_matches_stable_argsort(E, k, T):
    rng = np.random.default_rng(E * 1000 + T)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = oracle.align(ids, E)
    flat = ids.reshape(-1)
    ref = np.argsort(flat, kind="stable")
    assert np.array_equal(perm, ref)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert counts.sum() == T * k
    assert np.array_equal(inv[perm], np.arange(T * k))
    assert np.array_equal(perm[inv], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]: offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(flat[seg] == e)


def test_align_empty():
    counts, offsets, perm, inv = oracle.align(np.zeros((0, 2), dtype=np.int32), 4)
    assert counts.tolist() == [0, 0, 0, 0] and offsets.tolist() == [0] * 5
    assert perm.size == 0 and inv.size == 0


# ------------------------------------------------------------------ NaN logits
# Reading: a NaN logit is read as -inf (the pages are silent on NaN).  The pins
# below never feed a NaN to a library routine: they drop the NaN experts and
# solve the remaining problem by brute force or scipy.

@pytest.mark.parametrize("k,renorm", [(1, True), (2, True), (3, False)])
def test_nan_softmax_logits_equal_dropping_those_experts(k, renorm):
    rng = np.random.default_rng(40 + k)
    E = 8
    l = rng.standard_normal((120, E)).astype(np.float32)
    nan = rng.random((120, E)) < 0.25
    nan[:, 5] = False  # every row keeps a finite logit
    nan[:10, :] = True  # rows with fewer finite experts than k: NaN experts are then selected
    nan[:10, 5] = False
    l[nan] = np.nan
    ids, w, _ = oracle.gate(_prob(E, k, renormalize=renorm), l)
    for t in range(l.shape[0]):
        fin = np.nonzero(~nan[t])[0]
        pf = scipy.special.softmax(l[t, fin].astype(np.float64))
        if fin.size >= k:
            # the best k-subset of the finite experts, in descending logit order
            best, bs = None, -np.inf
            for c in itertools.combinations(fin.tolist(), k):
                s = float(np.sum(l[t, list(c)].astype(np.float64)))
                if s > bs:
                    best, bs = c, s
            assert set(ids[t].tolist()) == set(best), t
            sel = pf[np.searchsorted(fin, ids[t])]
            want = sel / sel.sum() if renorm else sel
            assert np.allclose(w[t], want, rtol=1e-14), t
        else:
            # all finite experts first (descending), then the NaN experts by index, weight 0
            order = fin[np.argsort(-l[t, fin].astype(np.float64), kind="stable")]
            rest = [e for e in range(E) if nan[t, e]][: k - fin.size]
            assert ids[t].tolist() == order.tolist() + rest, t
            assert np.all(w[t, fin.size:] == 0.0)
            want = pf[np.argsort(-l[t, fin].astype(np.float64), kind="stable")]
            assert np.allclose(w[t, :fin.size], want / want.sum() if renorm else want, rtol=1e-14)


def test_nan_sigmoid_grouped_key_is_the_bias():
    # E = 8, 2 groups of 4 keep 1, k = 2.  Expert 6's logit is NaN: its score is 0
    # and its key is bias[6] = 0.95.  Group 1 = {4..7} has keys
    # sigmoid(0) + 0 = 0.5, sigmoid(-1) = 0.2689, 0.95, sigmoid(-2) = 0.1192 -> score
    # 0.95 + 0.5 = 1.45; group 0 = {0..3}: sigmoid(1) = 0.7311, sigmoid(0.5) = 0.6225,
    # sigmoid(0) = 0.5, sigmoid(-0.5) = 0.3775 -> 1.3536.  Group 1 wins; its best
    # two keys are expert 6 (0.95) then expert 4 (0.5); weights 0 and sigmoid(0),
    # renormalised: 0 and 1, times 2.5.
    l = np.array([[1.0, 0.5, 0.0, -0.5, 0.0, -1.0, np.nan, -2.0]], dtype=np.float32)
    bias = np.array([0, 0, 0, 0, 0, 0, 0.95, 0], dtype=np.float32)
    p = _prob(8, 2, scoring="sigmoid", renormalize=True, n_group=2, topk_group=1, routed_scaling_factor=2.5)
    ids, w, _ = oracle.gate(p, l, bias)
    assert ids[0].tolist() == [6, 4]
    assert w[0].tolist() == [0.0, 2.5]


def test_nan_sigmoid_raw_keys_rank_last():
    # no bias, no groups (the Llama-4-Scout gate): a NaN expert is chosen only
    # after every finite one; the weight is sigmoid of the chosen logit
    rng = np.random.default_rng(50)
    l = rng.standard_normal((80, 16)).astype(np.float32)
    nan = rng.random((80, 16)) < 0.3
    nan[:, 0] = False
    l[nan] = np.nan
    p = _prob(16, 1, scoring="sigmoid", renormalize=False)
    ids, w, _ = oracle.gate(p, l)
    for t in range(80):
        fin = np.nonzero(~nan[t])[0]
        best = fin[np.argmax(l[t, fin])]
        assert ids[t, 0] == best
        assert w[t, 0] == pytest.approx(scipy.special.expit(float(l[t, best])), rel=1e-15)


def test_nan_only_selection_gets_zero_weights():
    # E = 8, 2 groups of 4 keep 1, k = 2, bias 0.3 on group 1 only.  Expert 0 is
    # the only finite logit (0.0, score 0.5, key 0.5): group 0 scores 0.5 + 0
    # (the NaN experts' keys are their zero bias), group 1 scores 0.3 + 0.3 = 0.6
    # and wins, so experts 4 and 5 (both NaN, score 0) are selected; renormalising
    # two zero scores gives zero weights, not 0 / 0.
    l = np.array([[0.0] + [np.nan] * 7], dtype=np.float32)
    bias = np.array([0, 0, 0, 0, 0.3, 0.3, 0.3, 0.3], dtype=np.float32)
    p = _prob(8, 2, scoring="sigmoid", renormalize=True, n_group=2, topk_group=1, routed_scaling_factor=2.5)
    ids, w, _ = oracle.gate(p, l, bias)
    assert ids[0].tolist() == [4, 5]
    assert w[0].tolist() == [0.0, 0.0]
