"""fp64 CPU oracle for the fused MoE layer.

TEST INFRASTRUCTURE ONLY: used by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py; never by the library.  Shares no code with the
CUDA path.
"""
from .codecs import (decode_bf16, decode_e4m3, encode_e4m3, unpack_int4, decode_int4_grouped,
                     unpack_uint4, decode_int4_grouped_zp, int8_codes, decode_int8_grouped,
                     decode_int8_grouped_zp, decode_fp16, encode_bf16, dynamic_scale, E4M3_MAX)
from .moe_ref import (Problem, NEAR_TIE, gate, gate_select, gate_weights, group_scores, softmax_fp64,
                      sigmoid_fp64, align, align_block_size, ExpertWeights, quantize_fp8, silu,
                      gate_up_swiglu, swiglu_act, quantize_act, down, input_rows, reduce, forward,
                      token_outputs)
