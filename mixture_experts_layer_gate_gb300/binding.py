"""ctypes binding of the C ABI in include/moe.h.

Argument marshalling only: every function passes tensor device pointers, sizes
and the current CUDA stream to the library, which does all the work in its own
kernels.  PyTorch is used for device memory and streams.  If the shared library
has not been built, loading it raises (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_BAD_INDEX", 6: "MOE_ERR_TIMEOUT"}
WDTYPES = {"bf16": 0, "fp8": 1, "int4": 2, "int8": 3, "int4_paired": 4}
ACT_SCALES = {"static": 0, "dynamic": 1}
SCORING = {"softmax": 0, "sigmoid": 1}

EXPORTED = ("moe_scratch_size", "moe_workspace_size", "moe_padded_capacity", "moe_gate_topk",
            "moe_align_permute", "moe_align_block_size", "moe_grouped_gemm_swiglu",
            "moe_grouped_gemm_down", "moe_unpermute_reduce", "moe_forward", "moe_get_device_error",
            "moe_status_string", "moe_get_plan", "moe_get_plan_for_sms", "moe_align_permute_noalloc",
            "moe_dynamic_scales", "moe_launch_count", "moe_set_tuning", "moe_repack_int4")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("wdtype", ctypes.c_int32), ("group_size", ctypes.c_int32), ("act_scale", ctypes.c_int32)]

    @property
    def S(self) -> int:
        return self.T * self.top_k


class WeightsStruct(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("a1_scale", ctypes.c_void_p),
                ("a2_scale", ctypes.c_void_p), ("w13_zero", ctypes.c_void_p), ("w2_zero", ctypes.c_void_p)]


class Plan(ctypes.Structure):
    _fields_ = [("bn_max_up", ctypes.c_int32), ("splits_up", ctypes.c_int32),
                ("stages_up", ctypes.c_int32), ("astages_up", ctypes.c_int32), ("smem_up", ctypes.c_int32),
                ("bn_max_down", ctypes.c_int32), ("splits_down", ctypes.c_int32),
                ("stages_down", ctypes.c_int32), ("astages_down", ctypes.c_int32),
                ("smem_down", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("slot_kb_up", ctypes.c_int32), ("slot_kb_down", ctypes.c_int32),
                ("pair_up", ctypes.c_int32), ("pair_down", ctypes.c_int32),
                ("issuers_up", ctypes.c_int32), ("issuers_down", ctypes.c_int32),
                ("conv_groups_up", ctypes.c_int32), ("conv_groups_down", ctypes.c_int32),
                ("epi_warps_up", ctypes.c_int32), ("epi_warps_down", ctypes.c_int32),
                ("acc_bufs_up", ctypes.c_int32), ("acc_bufs_down", ctypes.c_int32)]


class Tuning(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("bn_max", "stages", "splits", "pair", "conv_groups", "slot_kb",
                                             "ksplit", "dual", "full_box", "w_stream", "unit_order",
                                             "epi_warps", "acc_bufs")]


TUNING_KNOBS = tuple(n for n, _ in Tuning._fields_)

_lib = None


def load(path: str = LIB_PATH):
    """Loads the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -m mixture_experts_layer_gate_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(Problem)
    vp, sz, i32, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int
    sig = {
        "moe_scratch_size": (sz, [P]),
        "moe_workspace_size": (sz, [P]),
        "moe_padded_capacity": (sz, [P, i32]),
        "moe_gate_topk": (st, [P, vp, vp, vp, vp, vp]),
        "moe_align_permute": (st, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_align_block_size": (st, [P, vp, vp, i32, vp, vp, vp, vp]),
        "moe_align_permute_noalloc": (st, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_grouped_gemm_swiglu": (st, [P, ctypes.POINTER(WeightsStruct), vp, vp, vp, vp, sz, vp]),
        "moe_grouped_gemm_down": (st, [P, ctypes.POINTER(WeightsStruct), vp, vp, vp, vp, sz, vp]),
        "moe_unpermute_reduce": (st, [P, vp, vp, vp, vp, vp, sz, vp]),
        "moe_forward": (st, [P, ctypes.POINTER(WeightsStruct), vp, vp, vp, vp, vp, sz, vp]),
        "moe_get_device_error": (st, [vp, vp]),
        "moe_status_string": (ctypes.c_char_p, [st]),
        "moe_get_plan": (st, [P, ctypes.POINTER(Plan)]),
        "moe_get_plan_for_sms": (st, [P, i32, ctypes.POINTER(Plan)]),
        "moe_dynamic_scales": (vp, [vp]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_set_tuning": (st, [ctypes.POINTER(Tuning)]),
        "moe_repack_int4": (st, [vp, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().moe_status_string(int(status)).decode()
    except Exception:  # library missing: still report the code
        return STATUS_NAMES.get(status, str(status))


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def problem(T, H, I, E, top_k, scoring="softmax", renormalize=True, n_group=0, topk_group=0,
            routed_scaling_factor=1.0, wdtype="bf16", group_size=128, act_scale="static") -> Problem:
    return Problem(int(T), int(H), int(I), int(E), int(top_k), SCORING[scoring], int(bool(renormalize)),
                   int(n_group), int(topk_group), float(routed_scaling_factor), WDTYPES[wdtype],
                   int(group_size), ACT_SCALES[act_scale])


class Weights:
    """Expert weights as the library reads them; keeps the tensors alive."""

    def __init__(self, w13, w2, w13_scale=None, w2_scale=None, a1_scale=None, a2_scale=None,
                 w13_zero=None, w2_zero=None):
        self.tensors = (w13, w2, w13_scale, w2_scale, a1_scale, a2_scale, w13_zero, w2_zero)
        self.struct = WeightsStruct(*[None if t is None else t.data_ptr() for t in self.tensors])


def scratch_size(p: Problem) -> int:
    return int(load().moe_scratch_size(ctypes.byref(p)))


def workspace_size(p: Problem) -> int:
    return int(load().moe_workspace_size(ctypes.byref(p)))


def padded_capacity(p: Problem, block: int) -> int:
    return int(load().moe_padded_capacity(ctypes.byref(p), int(block)))


def alloc_workspace(p: Problem, device, full: bool = True):
    """Zeroed workspace (the error header must start at zero)."""
    import torch
    n = workspace_size(p) if full else scratch_size(p)
    if n == 0:
        raise MoEError(1, "workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def gate_topk(p: Problem, logits, bias, topk_ids, topk_w, stream=None):
    _check(load().moe_gate_topk(ctypes.byref(p), _ptr(logits), _ptr(bias), _ptr(topk_ids), _ptr(topk_w),
                                _stream(stream)), "moe_gate_topk")


def align_permute(p: Problem, topk_ids, x, a1_scale, counts, offsets, perm, inv, x_perm, ws, stream=None):
    _check(load().moe_align_permute(ctypes.byref(p), _ptr(topk_ids), _ptr(x), _ptr(a1_scale), _ptr(counts),
                                    _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm), _ptr(ws),
                                    ws.numel(), _stream(stream)), "moe_align_permute")


def align_permute_noalloc(p: Problem, topk_ids, x, a1_scale, counts, offsets, perm, inv, x_perm, stream=None):
    """moe_align_permute for callers that cannot allocate: no workspace argument;
    the library's fixed device-side array holds the scratch (see include/moe.h)."""
    _check(load().moe_align_permute_noalloc(ctypes.byref(p), _ptr(topk_ids), _ptr(x), _ptr(a1_scale),
                                            _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm),
                                            _stream(stream)), "moe_align_permute_noalloc")


def align_block_size(p: Problem, offsets, perm, block, sorted_ids, block_expert, total_padded, stream=None):
    _check(load().moe_align_block_size(ctypes.byref(p), _ptr(offsets), _ptr(perm), int(block),
                                       _ptr(sorted_ids), _ptr(block_expert), _ptr(total_padded),
                                       _stream(stream)), "moe_align_block_size")


def grouped_gemm_swiglu(p: Problem, w: Weights, x_perm, offsets, act, ws, stream=None):
    _check(load().moe_grouped_gemm_swiglu(ctypes.byref(p), ctypes.byref(w.struct), _ptr(x_perm),
                                          _ptr(offsets), _ptr(act), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_gemm_swiglu")


def grouped_gemm_down(p: Problem, w: Weights, act, offsets, y_perm, ws, stream=None):
    _check(load().moe_grouped_gemm_down(ctypes.byref(p), ctypes.byref(w.struct), _ptr(act), _ptr(offsets),
                                        _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_gemm_down")


def unpermute_reduce(p: Problem, y_perm, inv, topk_w, out, ws, stream=None):
    _check(load().moe_unpermute_reduce(ctypes.byref(p), _ptr(y_perm), _ptr(inv), _ptr(topk_w), _ptr(out),
                                       _ptr(ws), ws.numel(), _stream(stream)), "moe_unpermute_reduce")


def forward(p: Problem, w: Weights, x, logits, bias, out, ws, stream=None):
    _check(load().moe_forward(ctypes.byref(p), ctypes.byref(w.struct), _ptr(x), _ptr(logits), _ptr(bias),
                              _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_forward")


def get_device_error(ws, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the sticky device error code."""
    return int(load().moe_get_device_error(_ptr(ws), _stream(stream)))


def launch_count() -> int:
    """Kernel launches the library has issued in this process (graph captures once)."""
    return int(load().moe_launch_count())


def repack_int4(codes, out=None, stream=None):
    """int4 codes (uint8 tensor, packed order) -> a tensor of the same shape in the
    paired order of MOE_W_INT4_G128_PAIRED (moe_repack_int4); `out` may be
    `codes` itself (in place) but must not partly overlap it.  Returns the output
    tensor."""
    import torch
    if out is None:
        out = torch.empty_like(codes)
    if out.numel() != codes.numel() or codes.dtype != torch.uint8 or out.dtype != torch.uint8:
        raise ValueError("repack_int4: uint8 tensors of equal size")
    if not (codes.is_contiguous() and out.is_contiguous()):
        raise ValueError("repack_int4: contiguous tensors")
    _check(load().moe_repack_int4(_ptr(codes), _ptr(out), codes.numel(), _stream(stream)), "moe_repack_int4")
    return out


def dynamic_scales(ws):
    """The workspace's dynamic fp8 scales {a1, a2} as a float32 view [2] of ws."""
    import torch
    ptr = load().moe_dynamic_scales(_ptr(ws))
    if not ptr:
        raise MoEError(1, "moe_dynamic_scales")
    off = ptr - ws.data_ptr()
    return ws[off: off + 8].view(torch.float32)


def get_plan(p: Problem, num_sms: int | None = None) -> Plan:
    """Launch plan on the current device, or for `num_sms` SMs (no GPU needed)."""
    plan = Plan()
    if num_sms is None:
        _check(load().moe_get_plan(ctypes.byref(p), ctypes.byref(plan)), "moe_get_plan")
    else:
        _check(load().moe_get_plan_for_sms(ctypes.byref(p), int(num_sms), ctypes.byref(plan)),
               "moe_get_plan_for_sms")
    return plan


def set_tuning(**knobs):
    """Planner overrides (moe_set_tuning): keyword per knob, e.g. pair=0, dual=1;
    no keywords restores the planner's choices.  For tests and benchmarks."""
    unknown = set(knobs) - set(TUNING_KNOBS)
    if unknown:
        raise ValueError(f"unknown tuning knobs {sorted(unknown)}")
    if not knobs:
        _check(load().moe_set_tuning(None), "moe_set_tuning")
        return
    t = Tuning(*[int(knobs.get(n, -1)) for n in TUNING_KNOBS])
    _check(load().moe_set_tuning(ctypes.byref(t)), "moe_set_tuning")


class tuning:
    """Context manager: planner overrides inside the block, defaults after it."""

    def __init__(self, **knobs):
        self.knobs = knobs

    def __enter__(self):
        set_tuning(**self.knobs)
        return self

    def __exit__(self, *exc):
        set_tuning()


class MoELayer:
    """Convenience wrapper: one problem shape (up to a token budget), its weights
    and a workspace; `__call__` runs moe_forward on the current stream."""

    def __init__(self, H, I, E, top_k, weights: Weights, max_tokens: int, device, **gate):
        self.shape = dict(H=H, I=I, E=E, top_k=top_k, **gate)
        self.weights = weights
        self.ws = alloc_workspace(problem(max_tokens, H, I, E, top_k, **gate), device)

    def problem(self, T: int) -> Problem:
        return problem(T, **self.shape)

    def __call__(self, x, logits, bias=None, out=None, stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.shape["H"]), dtype=torch.bfloat16, device=x.device)
        p = self.problem(T)
        if workspace_size(p) > self.ws.numel():
            self.ws = alloc_workspace(p, x.device)
        forward(p, self.weights, x, logits, bias, out, self.ws, stream)
        return out
