"""Seeded synthetic input generators shared by the oracle tests and the CUDA path."""
from .inputs import (MoEShape, SHAPES, T_SWEEP, Weights, Tokens, make_weights, make_tokens,
                     shrink, static_act_scale, weight_seed, token_seed)
