"""Fused Mixture-of-Experts layer forward pass for GB300 (sm_103a).

The compute lives in libmoe_gb300.so (hand-written CUDA, C ABI in
include/moe.h); this package is its thin Python binding.
"""
from .binding import (MoEError, Problem, Plan, Weights, MoELayer, load, problem, scratch_size,
                      workspace_size, padded_capacity, alloc_workspace, gate_topk, align_permute,
                      align_permute_noalloc,
                      align_block_size, grouped_gemm_swiglu, grouped_gemm_down, unpermute_reduce,
                      forward, get_device_error, get_plan, dynamic_scales, launch_count, status_string, EXPORTED,
                      LIB_PATH, set_tuning, tuning, TUNING_KNOBS, repack_int4)
