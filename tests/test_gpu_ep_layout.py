"""Expert-parallel layout (single rank): the grouped GEMM entry points run over
a rank's local experts with rows an external dispatcher grouped by expert and
counts it supplied (offsets = exclusive scan of the counts, empty experts
included), no gate or permutation of ours involved.  The problem then has
T = rows received, top_k = 1 and E = local experts.  Compared per expert with
the oracle's SwiGLU MLP."""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_layer_gate_gb300 as moe
import oracle
from synth import SHAPES, make_weights, shrink
from tests.gpu_cases import TOL
from oracle.torch_io import LazyExperts, bf16_bits, np_of, problem_for

pytestmark = pytest.mark.gpu

COUNTS = [0, 37, 1, 0, 300, 5]  # rows per local expert: empty, ragged, single, > one 256-row tile


def _local_shape(name):
    base = {"bf16": shrink(SHAPES["mixtral"], H=512, I=1024),
            "fp8": shrink(SHAPES["qwen2"], H=384, I=256),
            "int4": shrink(SHAPES["dsv3"], H=1024, I=256),
            "int8": shrink(SHAPES["mixtral_w8"], H=512, I=256)}[name]
    # no gate runs here: an ungrouped softmax problem with one row per "token"
    return dataclasses.replace(base, E=len(COUNTS), top_k=1, n_group=0, topk_group=0,
                               scoring="softmax", routed_scaling_factor=1.0, has_bias=False)


@pytest.mark.parametrize("wdtype", ["bf16", "fp8", "int4", "int8"])
def test_grouped_gemms_over_dispatched_rows(wdtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    moe.load()
    shape = _local_shape(wdtype)
    R = sum(COUNTS)
    g = torch.Generator(device="cpu").manual_seed(7)
    x = torch.randn(R, shape.H, generator=g).to(torch.bfloat16)
    a1 = a2 = None
    if wdtype == "fp8":
        # dispatched rows arrive already quantised: finite e4m3 codes of either sign
        codes = torch.randint(0, 0x7F, (R, shape.H), generator=g, dtype=torch.int32)
        codes = codes | (torch.randint(0, 2, (R, shape.H), generator=g, dtype=torch.int32) << 7)
        x_perm = codes.to(torch.uint8).to(dev)
        a1 = torch.tensor([0.05], device=dev)
        a2 = torch.tensor([0.01], device=dev)
    else:
        x_perm = x.to(dev)
    w = make_weights(shape, dev, seed=3)
    wts = moe.Weights(w.w13, w.w2, w.w13_scale, w.w2_scale, a1, a2, w.w13_zero, w.w2_zero)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(COUNTS)]), dtype=torch.int32, device=dev)
    p = moe.problem(R, shape.H, shape.I, shape.E, 1, scoring="softmax", renormalize=False,
                    wdtype=shape.wdtype)
    ws = moe.alloc_workspace(p, dev)
    adt = torch.uint8 if wdtype == "fp8" else torch.bfloat16
    act = torch.empty((R, shape.I), dtype=adt, device=dev)
    y = torch.empty((R, shape.H), dtype=torch.bfloat16, device=dev)
    moe.grouped_gemm_swiglu(p, wts, x_perm, offsets, act, ws)
    moe.grouped_gemm_down(p, wts, act, offsets, y, ws)
    torch.cuda.synchronize()
    assert moe.get_device_error(ws) == 0

    op = problem_for(shape, R)
    experts = LazyExperts(op, w)
    if wdtype == "fp8":
        X = oracle.decode_e4m3(np_of(x_perm)) * float(a1.cpu()[0])
    else:
        X = oracle.decode_bf16(bf16_bits(x))
    y_gpu = oracle.decode_bf16(bf16_bits(y))
    o = np.concatenate([[0], np.cumsum(COUNTS)])
    for e, c in enumerate(COUNTS):
        if c == 0:
            continue
        W13, W2 = experts(e)
        a_ref = oracle.gate_up_swiglu(op, X[o[e]:o[e + 1]], W13, None if a2 is None else float(a2.cpu()[0]))
        y_ref = oracle.down(a_ref, W2)
        err = np.abs(y_gpu[o[e]:o[e + 1]] - y_ref).max() / np.abs(y_ref).max()
        assert err <= TOL[wdtype], (wdtype, e, err)
