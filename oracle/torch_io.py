"""Moves synthetic torch inputs into the numpy arrays the oracle reads.

TEST INFRASTRUCTURE ONLY, like the rest of this package: argument marshalling
for tests/, __graft_entry__.smoke() and the CPU-baseline leg of bench.py.  It is
not imported by the package's __init__, so the oracle itself needs no torch.
"""
import numpy as np
import torch

from .moe_ref import Problem, ExpertWeights


def problem_for(shape, T) -> Problem:
    return Problem(T=T, H=shape.H, I=shape.I, E=shape.E, top_k=shape.top_k, scoring=shape.scoring,
                   renormalize=shape.renormalize, n_group=shape.n_group, topk_group=shape.topk_group,
                   routed_scaling_factor=shape.routed_scaling_factor, wdtype=shape.wdtype,
                   group_size=shape.group_size, act_scale=shape.act_scale)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_of(t):
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype == torch.float16:
        return t.numpy()
    return t.numpy()


class LazyExperts(ExpertWeights):
    """ExpertWeights that copies one expert at a time off the device."""

    def __init__(self, p, weights):
        super().__init__(p, None, None)
        self._w = weights

    def __call__(self, e):
        w = self._w
        self.w13 = {e: np_of(w.w13[e])}
        self.w2 = {e: np_of(w.w2[e])}
        if w.w13_scale is not None:
            self.s13 = {e: np_of(w.w13_scale[e])}
            self.s2 = {e: np_of(w.w2_scale[e])}
        if getattr(w, "w13_zero", None) is not None:
            self.z13 = {e: np_of(w.w13_zero[e])}
            self.z2 = {e: np_of(w.w2_zero[e])}
        return super().__call__(e)


def oracle_inputs(shape, weights, tokens):
    T = tokens.x.shape[0]
    p = problem_for(shape, T)
    experts = LazyExperts(p, weights)
    a1 = None if tokens.a1_scale is None else float(tokens.a1_scale.cpu()[0])
    a2 = None if tokens.a2_scale is None else float(tokens.a2_scale.cpu()[0])
    return p, dict(x_bits=bf16_bits(tokens.x), logits=np_of(tokens.logits), bias=np_of(tokens.bias),
                   experts=experts, a1=a1, a2=a2)
