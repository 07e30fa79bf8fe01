"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
entry point include/moe.h declares, and rejects bad arguments before touching
the device."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_gate_gb300 as moe
from mixture_experts_layer_gate_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moe.LIB_PATH):
        from mixture_experts_layer_gate_gb300 import build
        build.build()
    return moe.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("moe_gate_topk", "moe_align_permute", "moe_grouped_gemm_swiglu", "moe_grouped_gemm_down",
              "moe_unpermute_reduce", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(binding.EXPORTED) | set(names)


def test_struct_layout_matches_header():
    assert ctypes.sizeof(binding.Problem) == 52
    assert ctypes.sizeof(binding.WeightsStruct) == 64
    assert ctypes.sizeof(binding.Plan) == 92     # 23 four-byte fields
    assert ctypes.sizeof(binding.Tuning) == 52   # 13 four-byte fields


def test_status_strings(lib):
    assert moe.status_string(0) == "ok"
    assert "workspace" in moe.status_string(3)
    assert moe.status_string(99) == "unknown status"


@pytest.mark.parametrize("bad", [
    dict(H=100), dict(I=96), dict(top_k=9), dict(E=2048), dict(T=-1),
    dict(scoring="softmax", n_group=2, topk_group=1),
    dict(scoring="sigmoid", n_group=3, topk_group=1),
    dict(scoring="sigmoid", n_group=4, topk_group=5),
    dict(scoring="sigmoid", n_group=4, topk_group=1, top_k=3, E=8),
    dict(wdtype="int4", group_size=64),
])
def test_invalid_problems_rejected(lib, bad):
    kw = dict(T=4, H=256, I=512, E=8, top_k=2)
    kw.update(bad)
    p = moe.problem(**kw)
    assert moe.workspace_size(p) == 0
    assert moe.scratch_size(p) == 0
    st = lib.moe_gate_topk(ctypes.byref(p), None, None, None, None, None)
    assert st in (1, 2)


def test_null_and_misaligned_arguments_rejected(lib):
    p = moe.problem(4, 256, 512, 8, 2)
    assert lib.moe_gate_topk(ctypes.byref(p), None, None, None, None, None) == 1
    assert lib.moe_gate_topk(None, None, None, None, None, None) == 1
    # workspace too small / missing
    assert lib.moe_align_permute(ctypes.byref(p), None, None, None, None, None, None, None, None,
                                 None, 0, None) == 3
    assert lib.moe_unpermute_reduce(ctypes.byref(p), 16, 16, 16, 16, 256, 8, None) == 3
    w = binding.WeightsStruct(None, None, None, None, None, None)
    assert lib.moe_forward(ctypes.byref(p), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    w = binding.WeightsStruct(4096, 4097, None, None, None, None)   # misaligned w2
    assert lib.moe_forward(ctypes.byref(p), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    pf = moe.problem(4, 256, 512, 8, 2, wdtype="fp8")
    w = binding.WeightsStruct(4096, 8192, None, None, None, None)   # fp8 needs scales
    assert lib.moe_forward(ctypes.byref(pf), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    # zero points: only for int4, and both or neither
    w = binding.WeightsStruct(4096, 8192, None, None, None, None, 4096, 4096)
    assert lib.moe_forward(ctypes.byref(p), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    p4 = moe.problem(4, 256, 512, 8, 2, wdtype="int4")
    w = binding.WeightsStruct(4096, 8192, 4096, 4096, None, None, 4096, None)
    assert lib.moe_forward(ctypes.byref(p4), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    w = binding.WeightsStruct(4096, 8192, 4096, 4096, None, None, None, 4096)
    assert lib.moe_grouped_gemm_down(ctypes.byref(p4), ctypes.byref(w), 16, 16, 16, 256, 1 << 30, None) == 1
    # dynamic fp8 scales: computed, so neither activation scale may be given
    pd = moe.problem(4, 256, 512, 8, 2, wdtype="fp8", act_scale="dynamic")
    w = binding.WeightsStruct(4096, 8192, 4096, 4096, 4096, None)
    assert lib.moe_forward(ctypes.byref(pd), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1
    assert lib.moe_align_permute(ctypes.byref(pd), 16, 16, 16, 16, 16, 16, 16, 16, 256, 1 << 30, None) == 1
    w = binding.WeightsStruct(4096, 8192, 4096, 4096, None, None)     # static fp8 needs both
    assert lib.moe_forward(ctypes.byref(pf), ctypes.byref(w), 16, 16, None, 16, 256, 1 << 30, None) == 1


def test_dynamic_scale_problems(lib):
    # only fp8 takes dynamic scales; they add a bf16 [S, I] scratch buffer
    assert moe.scratch_size(moe.problem(4, 256, 512, 8, 2, act_scale="dynamic")) == 0
    assert moe.scratch_size(moe.problem(4, 256, 512, 8, 2, wdtype="int4", act_scale="dynamic")) == 0
    bad = moe.problem(4, 256, 512, 8, 2, wdtype="fp8")
    bad.act_scale = 2
    assert moe.scratch_size(bad) == 0
    for T in (1, 100, 4096):
        st = moe.scratch_size(moe.problem(T, 256, 512, 8, 2, wdtype="fp8"))
        dy = moe.scratch_size(moe.problem(T, 256, 512, 8, 2, wdtype="fp8", act_scale="dynamic"))
        assert dy - st >= T * 2 * 512 * 2
    # the scales' address is plain arithmetic on ws (no device access)
    assert lib.moe_dynamic_scales(None) is None
    assert lib.moe_dynamic_scales(ctypes.c_void_p(1 << 20)) == (1 << 20) + 80
    assert lib.moe_dynamic_scales(ctypes.c_void_p((1 << 20) + 8)) is None


def test_workspace_sizes_are_monotone_and_cover_intermediates(lib):
    prev = 0
    for T in (1, 2, 8, 64, 512, 4096):
        p = moe.problem(T, 4096, 14336, 8, 2)
        ws = moe.workspace_size(p)
        S = 2 * T
        # at least x_perm + act + y_perm + ids/w/perm/inv
        assert ws >= S * (4096 * 2 + 14336 * 2 + 4096 * 2) + 4 * S * 4
        assert moe.scratch_size(p) <= ws
        prev = ws
    pe = moe.problem(0, 4096, 14336, 8, 2)
    assert moe.workspace_size(pe) > 0


def test_padded_capacity(lib):
    p = moe.problem(4, 256, 512, 4, 2)
    assert moe.padded_capacity(p, 2) == 8 + 4
    assert moe.padded_capacity(p, 1) == 8
    assert moe.padded_capacity(p, 0) == 0


def _all_problems():
    from synth import SHAPES, T_SWEEP
    for s in SHAPES.values():
        for T in (0,) + tuple(T_SWEEP) + (3, 37, 1000, 8192):
            yield s, moe.problem(T, s.H, s.I, s.E, s.top_k, scoring=s.scoring, renormalize=s.renormalize,
                                 n_group=s.n_group, topk_group=s.topk_group,
                                 routed_scaling_factor=s.routed_scaling_factor, wdtype=s.wdtype,
                                 act_scale=s.act_scale)


def _check_plan(shape, pl):
    for side in ("up", "down"):
        bn = getattr(pl, f"bn_max_{side}")
        assert 16 <= bn <= 256 and bn % 16 == 0
        assert 1 <= getattr(pl, f"splits_{side}") <= 16
        st, ast = getattr(pl, f"stages_{side}"), getattr(pl, f"astages_{side}")
        assert st >= 2
        assert getattr(pl, f"smem_{side}") <= 232448
        issuers = getattr(pl, f"issuers_{side}")
        assert issuers in (1, 2)
        ew = getattr(pl, f"epi_warps_{side}")
        assert ew in (4, 8)
        if ew == 8 and shape.wdtype in ("int4", "int8"):
            # eight epilogue warps exist only for CTA pairs, two converter groups and
            # whole-stage slots
            assert getattr(pl, f"pair_{side}") == 1 and getattr(pl, f"conv_groups_{side}") == 2
            assert getattr(pl, f"slot_kb_{side}") == 4
        if shape.wdtype in ("int4", "int8"):
            # TMEM holds the accumulators (two buffers, or with two issuing threads
            # two partials per buffer and one buffer above 64 columns) and the
            # converted-weight slot ring
            sk = getattr(pl, f"slot_kb_{side}")
            assert sk in (2, 4) and (bn <= 128 or getattr(pl, f"pair_{side}") == 1)
            acc = (bn + 31) // 32 * 32
            bufs = getattr(pl, f"acc_bufs_{side}")
            if acc > 128:
                # one issuer; one buffer beside two slots, or (short-K units, <= 192
                # columns) two buffers beside one slot that both groups fill
                assert issuers == 1
                assert bufs == 1 or (bufs == 2 and ast == 1 and acc <= 192 and sk == 4)
            else:
                # two buffers, or one with two issuers above 64 columns
                assert bufs == (2 if issuers == 1 or acc <= 64 else 1)
            assert 1 <= ast <= 7 and issuers * bufs * acc + 32 * sk * ast <= 512
            # a ring of g converter groups alternating stages needs (g - 1) * 4 / sk + 1
            # slots and a stage count that is a multiple of g (one slot: k-split)
            assert ast >= 4 // sk + 1 or ast == 1
            if sk == 4:
                # whole-stage slots reuse the stage ring's barriers; an odd depth only
                # with both groups converting every stage (k-split, for a shallow ring)
                assert st >= ast and (st % 2 == 0 or st == 3 or ast == 1)
            else:
                assert st % 2 == 0 or st % 3 == 0
            cg = getattr(pl, f"conv_groups_{side}")
            assert cg in (2, 3) and (ast >= (cg - 1) * (4 // sk) + 1 or (ast == 1 and cg == 2))
            if issuers == 2:  # whole-stage slots
                assert sk == 4
            if cg == 3 and issuers == 2:  # int4 tiles of <= 32 tokens on one CTA
                assert shape.wdtype == "int4" and acc <= 32 and getattr(pl, f"pair_{side}") == 0
                assert st % 3 == 0
        else:
            assert ast == 0 and getattr(pl, f"slot_kb_{side}") == 0 and issuers == 1
    return pl


@pytest.mark.parametrize("sms", [148, 152, 160])
def test_plans_respect_hardware_and_pipeline_invariants(lib, sms):
    for shape, p in _all_problems():
        pl = _check_plan(shape, moe.get_plan(p, num_sms=sms))
        for side in ("up", "down"):
            # int4 / int8 tiles of <= 32 tokens run one CTA per 128 weight rows,
            # otherwise CTA pairs exactly when the weight blocks pair up; two
            # MMA-issuing threads for int4, and for int8 tiles of <= 32 tokens
            bn = getattr(pl, f"bn_max_{side}")
            fb = shape.I // 64 if side == "up" else shape.H // 128
            small = shape.wdtype in ("int4", "int8") and bn <= 32
            kb = (shape.H if side == "up" else shape.I) // 64 // getattr(pl, f"splits_{side}")
            # ... except units of <= 8 k-blocks once the batch has >= 64 rows
            short_units = kb <= 8 and p.T * shape.top_k >= 64
            # two issuers share TMEM with two buffers of partials: tiles of <= 128 tokens;
            # above 64 tokens (one buffer of partials) only for units of >= 16 k-blocks
            two = (shape.wdtype == "int4" and bn <= 128 and (bn <= 64 or kb >= 16)) or \
                  (shape.wdtype == "int8" and small)
            assert getattr(pl, f"pair_{side}") == (1 if fb % 2 == 0 and (not small or short_units) else 0)
            assert getattr(pl, f"issuers_{side}") == (2 if two else 1)
            # eight epilogue warps on bf16 / fp8 CTA pairs, four elsewhere
            conv = shape.wdtype in ("int4", "int8")
            assert getattr(pl, f"epi_warps_{side}") == (8 if getattr(pl, f"pair_{side}") and not conv else 4)


@pytest.mark.parametrize("pair", [0, 1])
def test_plans_with_two_mma_issuers(lib, pair):
    # forced, on one CTA or CTA pairs: every int4 / int8 GEMM takes two issuing
    # threads (bf16 / fp8 keep one); the invariants above still hold
    seen = 0
    with moe.tuning(dual=1, pair=pair):
        for shape, p in _all_problems():
            pl = _check_plan(shape, moe.get_plan(p, num_sms=152))
            for side in ("up", "down"):
                # tiles above 128 tokens leave TMEM room for one issuer's accumulator only
                two = shape.wdtype in ("int4", "int8") and getattr(pl, f"bn_max_{side}") <= 128
                assert getattr(pl, f"issuers_{side}") == (2 if two else 1)
                seen += two and getattr(pl, f"pair_{side}") == int(pair)
    assert seen > 0


def test_tuning_overrides_are_explicit_and_validated(lib, monkeypatch):
    p = moe.problem(37, 1024, 256, 64, 8, scoring="sigmoid", n_group=8, topk_group=4, wdtype="int4")
    base = moe.get_plan(p, num_sms=152)
    # the environment is never read
    for k in ("MOE_PAIR", "MOE_DUAL", "MOE_BN_MAX", "MOE_STAGES", "MOE_SPLITS", "MOE_SLOT_KB"):
        monkeypatch.setenv(k, "1" if k in ("MOE_PAIR", "MOE_DUAL") else "2")
    again = moe.get_plan(p, num_sms=152)
    assert bytes(again) == bytes(base)
    with moe.tuning(pair=1 - base.pair_up, stages=2):
        forced = moe.get_plan(p, num_sms=152)
        assert forced.pair_up == 1 - base.pair_up and forced.stages_up == 2
    assert bytes(moe.get_plan(p, num_sms=152)) == bytes(base)  # restored on exit
    for bad in (dict(bn_max=24), dict(bn_max=512), dict(slot_kb=3), dict(pair=2), dict(splits=17),
                dict(stages=1), dict(conv_groups=4), dict(epi_warps=6)):
        with pytest.raises(moe.MoEError):
            moe.set_tuning(**bad)
        assert bytes(moe.get_plan(p, num_sms=152)) == bytes(base)  # a rejected call changes nothing
    with pytest.raises(ValueError):
        moe.set_tuning(no_such_knob=1)


def test_epilogue_warp_override(lib):
    from synth import SHAPES
    # eight epilogue warps where a kernel has them (int4 / int8 CTA pairs with two
    # converter groups and whole-stage slots); a one-CTA int4 plan keeps four
    big = moe.problem(4096, 7168, 256, 256, 8, scoring="sigmoid", n_group=8, topk_group=4, wdtype="int4")
    with moe.tuning(epi_warps=8):
        pl = _check_plan(SHAPES["dsv3_tp8"], moe.get_plan(big, num_sms=152))
        assert pl.pair_down == 1 and pl.epi_warps_down == 8
        small = moe.problem(4, 7168, 256, 256, 8, scoring="sigmoid", n_group=8, topk_group=4, wdtype="int4")
        ps = moe.get_plan(small, num_sms=152)
        assert ps.pair_up == 0 and ps.epi_warps_up == 4
    bf = moe.problem(4096, 4096, 14336, 8, 2, wdtype="bf16")
    with moe.tuning(epi_warps=4):
        assert moe.get_plan(bf, num_sms=152).epi_warps_up == 4
    pl = moe.get_plan(bf, num_sms=152)
    assert pl.epi_warps_up == 8 and pl.stages_up >= 6  # the second staging half leaves the ring depth


def test_repack_int4_rejects_bad_arguments(lib):
    # refused before any device work: sizes that are not whole 4-byte words,
    # misaligned or null pointers; an empty tensor is a no-op
    vp = ctypes.c_void_p
    assert lib.moe_repack_int4(vp(256), vp(512), 6, None) == 1  # MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(vp(258), vp(512), 8, None) == 1  # MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(vp(256), vp(514), 8, None) == 1  # MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(None, vp(512), 8, None) == 1  # MOE_ERR_INVALID_ARG
    assert lib.moe_repack_int4(vp(256), vp(512), 0, None) == binding.MOE_OK


def test_paired_int4_plans_match_packed_int4(lib):
    # the paired code order changes only the converters' instructions
    for T in (1, 37, 512, 4096):
        a = moe.problem(T, 7168, 2048, 256, 8, scoring="sigmoid", n_group=8, topk_group=4, wdtype="int4")
        b = moe.problem(T, 7168, 2048, 256, 8, scoring="sigmoid", n_group=8, topk_group=4, wdtype="int4_paired")
        assert bytes(moe.get_plan(a, num_sms=152)) == bytes(moe.get_plan(b, num_sms=152))
    assert moe.scratch_size(b) == moe.scratch_size(a) > 0
