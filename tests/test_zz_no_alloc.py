"""The workspace-free align/permute entry point (for callers that may not
allocate device memory, e.g. an operator plugin given no scratch buffer, or a
serving loop that forbids cudaMalloc after start-up) must give exactly the
results of the regular entry point that takes a workspace.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It also passes on its own in a fresh process.
"""
import dataclasses

import pytest
import torch

import mixture_experts_layer_gate_gb300 as moe
from synth import SHAPES, make_tokens, shrink

pytestmark = pytest.mark.gpu


def _problem(shape, T):
    return moe.problem(T, shape.H, shape.I, shape.E, shape.top_k, scoring=shape.scoring,
                       renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                       routed_scaling_factor=shape.routed_scaling_factor, wdtype=shape.wdtype)


def _outputs(shape, T, dev):
    S = T * shape.top_k
    adt = torch.uint8 if shape.wdtype == "fp8" else torch.bfloat16
    return dict(counts=torch.full((shape.E,), -1, dtype=torch.int32, device=dev),
                offsets=torch.full((shape.E + 1,), -1, dtype=torch.int32, device=dev),
                perm=torch.full((S,), -1, dtype=torch.int32, device=dev),
                inv=torch.full((S,), -1, dtype=torch.int32, device=dev),
                x_perm=torch.zeros((S, shape.H), dtype=adt, device=dev))


@pytest.mark.parametrize("name", ["dsv3", "qwen2"])
def test_noalloc_align_permute_matches_workspace_entry_point(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    moe.load()
    base = SHAPES[name]
    shape = shrink(base, H=1024, I=256, E=64)
    if name == "dsv3":
        shape = dataclasses.replace(shape, n_group=8, topk_group=4)
    # two calls in a row with different batches: stale contents of the shared
    # scratch array from the first call must not leak into the second
    for T, seed in ((300, 0), (1000, 1)):
        tok = make_tokens(shape, T, dev, seed)
        p = _problem(shape, T)
        ids = torch.empty((T, shape.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, shape.top_k), dtype=torch.float32, device=dev)
        moe.gate_topk(p, tok.logits, tok.bias, ids, w)
        ref = _outputs(shape, T, dev)
        ws = moe.alloc_workspace(p, dev, full=False)
        moe.align_permute(p, ids, tok.x, tok.a1_scale, ref["counts"], ref["offsets"], ref["perm"], ref["inv"],
                          ref["x_perm"], ws)
        got = _outputs(shape, T, dev)
        moe.align_permute_noalloc(p, ids, tok.x, tok.a1_scale, got["counts"], got["offsets"], got["perm"],
                                  got["inv"], got["x_perm"])
        torch.cuda.synchronize()
        assert moe.get_device_error(ws) == 0
        for key in ref:
            assert torch.equal(got[key], ref[key]), (name, T, key)


def test_noalloc_empty_batch_and_exactly_full_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    moe.load()
    # T = 0: nothing to sort; counts and offsets come back all zero
    shape = shrink(SHAPES["tiny"], H=128, I=128)
    p = _problem(shape, 0)
    got = _outputs(shape, 0, dev)
    none = torch.empty(0, dtype=torch.int32, device=dev)
    moe.align_permute_noalloc(p, none, none, None, got["counts"], got["offsets"], none, none, none)
    torch.cuda.synchronize()
    assert torch.count_nonzero(got["counts"]).item() == 0
    assert torch.count_nonzero(got["offsets"]).item() == 0
    # the largest accepted problem: ceil(T*k / 1024) * E == 65536 histogram
    # entries exactly fills the 256 KiB array (E = 1024, T*k = 65536)
    shape = dataclasses.replace(SHAPES["tiny"], name="fill", H=128, I=128, E=1024, top_k=2)
    T = 32768
    tok = make_tokens(shape, T, dev, 2)
    p = _problem(shape, T)
    ids = torch.empty((T, 2), dtype=torch.int32, device=dev)
    w = torch.empty((T, 2), dtype=torch.float32, device=dev)
    moe.gate_topk(p, tok.logits, tok.bias, ids, w)
    ref = _outputs(shape, T, dev)
    ws = moe.alloc_workspace(p, dev, full=False)
    moe.align_permute(p, ids, tok.x, None, ref["counts"], ref["offsets"], ref["perm"], ref["inv"],
                      ref["x_perm"], ws)
    got = _outputs(shape, T, dev)
    moe.align_permute_noalloc(p, ids, tok.x, None, got["counts"], got["offsets"], got["perm"], got["inv"],
                              got["x_perm"])
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0
    for key in ref:
        assert torch.equal(got[key], ref[key]), ("fill", key)


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()
    # ceil(T*k/1024) * E must stay <= 65536: E = 1024 with T*k = 65 538 slots needs 65 CTAs
    p = moe.problem(32769, 256, 256, 1024, 2)
    assert moe.scratch_size(p) > 0       # a valid problem, only too large for the fixed array
    x = torch.empty(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(moe.MoEError) as ei:
        moe.align_permute_noalloc(p, x, x, None, x, x, x, x, x)
    assert ei.value.status == 2
    # a problem beyond the library's own limits gets the status moe_align_permute gives
    big = moe.problem(70000, 256, 256, 8, 2)
    with pytest.raises(moe.MoEError) as ei:
        moe.align_permute_noalloc(big, x, x, None, x, x, x, x, x)
    assert ei.value.status == 2
    bad = moe.problem(8, 100, 256, 8, 2)  # H % 128 != 0
    with pytest.raises(moe.MoEError) as ei:
        moe.align_permute_noalloc(bad, x, x, None, x, x, x, x, x)
    assert ei.value.status == 1
