"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (a dropped term, a wrong sign or
index, swapped operands, a wrong rounding or scope) by replacing one of its
functions for the duration of the test, then runs the pins that should notice
and requires at least one of them to fail.  Nothing here touches the GPU path.
"""
import numpy as np
import pytest

import oracle
import oracle.codecs as codecs
import oracle.moe_ref as moe_ref
from tests import test_oracle_codecs as t_codecs
from tests import test_oracle_dynamic as t_dynamic
from tests import test_oracle_forward as t_forward
from tests import test_oracle_gate_align as t_gate


def _patch(monkeypatch, name, fn):
    """Replaces `name` wherever the oracle or the pin modules bound it."""
    hit = False
    for mod in (oracle, codecs, moe_ref, t_codecs, t_dynamic, t_forward, t_gate):
        if hasattr(mod, name):
            monkeypatch.setattr(mod, name, fn)
            hit = True
    assert hit, name


def _some_pin_fails(pins):
    failed = []
    for pin in pins:
        try:
            pin()
        except Exception as exc:  # an assertion, or a shape error the mistake causes
            failed.append((pin, exc))
    return failed


# ------------------------------------------------------------------ mutations

def _no_renormalisation(p, logits, ids):
    score = moe_ref.softmax_fp64(logits) if p.scoring == "softmax" else moe_ref.sigmoid_fp64(logits)
    w = np.take_along_axis(score, ids.astype(np.int64), axis=1)
    return w * float(p.routed_scaling_factor)


def _bias_in_weights(p, logits, ids):
    w = _ORIG["gate_weights"](p, logits, ids)
    return w * 1.05 if p.scoring == "sigmoid" else w


def _group_score_max(p, keys):
    T = keys.shape[0]
    return keys.reshape(T, p.n_group, p.E // p.n_group).max(axis=-1)


def _ties_to_higher_index(keys, k):
    T, E = keys.shape
    idx = np.broadcast_to(-np.arange(E), (T, E))
    return np.lexsort((idx, -keys), axis=-1)[:, :k]


def _unstable_align(ids, E):
    counts, offsets, perm, inv = _ORIG["align"](ids, E)
    perm = perm.copy()
    for e in range(E):  # reverse each expert's segment
        perm[offsets[e]: offsets[e + 1]] = perm[offsets[e]: offsets[e + 1]][::-1]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return counts, offsets, perm, inv


def _silu_on_up_half(p, X, W13):
    h = X @ W13.T
    return h[:, : p.I] * moe_ref.silu(h[:, p.I:])


def _down_untransposed(act, W2):
    return act @ W2


def _reduce_shifted_weights(p, y_perm, inv, w):
    return _ORIG["reduce"](p, y_perm, inv, np.roll(w, 1, axis=1))


def _int4_scale_group_shifted(packed, scales, group_size):
    q = codecs.unpack_int4(packed).astype(np.float64)
    s = np.roll(codecs.decode_fp16(scales), 1, axis=-1)
    return q * np.repeat(s, group_size, axis=-1)


def _zero_point_added(packed, scales, zeros, group_size):
    q = codecs.unpack_uint4(packed).astype(np.float64)
    s = codecs.decode_fp16(scales)
    z = np.asarray(zeros).astype(np.float64)
    return (q + np.repeat(z, group_size, axis=-1)) * np.repeat(s, group_size, axis=-1)


def _bf16_through_float32(x):
    return _ORIG["encode_bf16"](np.asarray(x, dtype=np.float64).astype(np.float32))


def _e4m3_toward_zero(x):
    v = np.asarray(x, dtype=np.float64)
    codes = _ORIG["encode_e4m3"](v)
    dec = codecs.decode_e4m3(codes)
    # step one code toward zero wherever round-to-nearest went away from zero
    away = np.abs(dec) > np.abs(v)
    return np.where(away & (codes & 0x7F > 0), codes - 1, codes).astype(np.uint8)


def _scale_of_first_row(values):
    v = np.asarray(values, dtype=np.float64)
    return _ORIG["dynamic_scale"](v[:1] if v.ndim > 1 else v)


def _nan_logits_rank_first(logits):
    l = np.asarray(logits, dtype=np.float64)
    return np.where(np.isnan(l), np.inf, l)


_ORIG = {name: getattr(moe_ref, name, None) or getattr(codecs, name)
         for name in ("gate_weights", "align", "reduce", "encode_bf16", "encode_e4m3", "dynamic_scale")}

MUTATIONS = {
    "softmax weights not renormalised": (
        "gate_weights", _no_renormalisation, [t_gate.test_golden_softmax_gate]),
    "sigmoid weights scaled by the bias path": (
        "gate_weights", _bias_in_weights, [t_gate.test_golden_sigmoid_grouped_gate]),
    "group score = max instead of the two best": (
        "group_scores", _group_score_max,
        [t_gate.test_golden_sigmoid_grouped_gate, t_gate.test_grouped_sigmoid_brute_force]),
    "equal keys go to the higher index": (
        "_topk_desc_lower_index", _ties_to_higher_index, [t_gate.test_all_equal_logits]),
    "permutation not stable within an expert": (
        "align", _unstable_align,
        [t_gate.test_golden_align, lambda: t_gate.test_align_matches_stable_argsort(8, 2, 333)]),
    "SiLU applied to the up half": (
        "swiglu_act", _silu_on_up_half,
        [t_forward.test_golden_swiglu_single_expert, t_forward.test_single_expert_reduces_to_plain_swiglu_mlp]),
    "down projection not transposed": (
        "down", _down_untransposed, [t_forward.test_golden_swiglu_single_expert]),
    "reduce weights paired with the wrong slot": (
        "reduce", _reduce_shifted_weights, [lambda: t_forward.test_forward_matches_dense_bruteforce("tiny")]),
    "int4 scale of the neighbouring group": (
        "decode_int4_grouped", _int4_scale_group_shifted, [t_codecs.test_int4_grouped_decode_brute_force]),
    "zero point added instead of subtracted": (
        "decode_int4_grouped_zp", _zero_point_added, [t_codecs.test_decode_zp_brute_force]),
    "bf16 rounded through float32": (
        "encode_bf16", _bf16_through_float32, [t_dynamic.test_encode_bf16_rounds_once_from_the_exact_value]),
    "e4m3 rounded toward zero": (
        "encode_e4m3", _e4m3_toward_zero, [t_codecs.test_e4m3_encode_matches_torch_cast_in_range]),
    "NaN logits ranked first instead of last": (
        "logits_fp64", _nan_logits_rank_first,
        [lambda: t_gate.test_nan_softmax_logits_equal_dropping_those_experts(2, True),
         t_gate.test_nan_sigmoid_grouped_key_is_the_bias, t_gate.test_nan_sigmoid_raw_keys_rank_last]),
    "dynamic scale over one row instead of the tensor": (
        "dynamic_scale", _scale_of_first_row, [t_dynamic.test_dynamic_forward_matches_dense_bruteforce]),
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(monkeypatch, mutation):
    name, fn, pins = MUTATIONS[mutation]
    _patch(monkeypatch, name, fn)
    assert _some_pin_fails(pins), f"no pin noticed: {mutation}"


def test_pins_pass_without_mutation():
    # the same pins, unpatched, all pass (so a failure above is the mutation's doing)
    for _, _, pins in MUTATIONS.values():
        assert not _some_pin_fails(pins)
