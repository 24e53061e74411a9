"""CPU oracle of early-exit decoding -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library does not use it.
"""
from .model import *  # noqa: F401,F403
from .model import (  # noqa: F401
    Oracle, Weights, ModelConfig, StepResult, build_oracle, calibrate_gammas, forward_full,
    quantize_int4_group, pack_int4, unpack_int4, dequant_int4, bf16_to_f32, bf16_to_f64,
    f32_to_bf16_bits, rmsnorm, rope, attention_decode, swiglu, silu, head_logits, max_softmax,
    argmax_lowest, top2_margin, layer_decode, linear, state_transition_similarity, layer_full,
)
