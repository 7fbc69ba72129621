"""Seeded synthetic inputs for the DFlash drafting round.

This package is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It draws numbers and holds shapes; it contains none of the
method's arithmetic (no norm, projection, attention, argmax or acceptance).
"""
from .gen import (  # noqa: F401
    splitmix64_bits,
    stream_key,
    uniform,
    normal,
    f64_to_bf16_bits,
    bf16_bits_to_f32,
)
from .configs import DraftConfig, CONFIGS, TEST_CONFIGS, get_config  # noqa: F401
from .inputs import (  # noqa: F401
    make_weights,
    make_target_weights,
    prompt_tokens,
    feature_rows,
    match_stream,
    context_lengths,
    match_probs,
    WEIGHT_NAMES,
)
