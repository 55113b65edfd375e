"""CPU oracle for the Qwen3-style dense decoder over Q8_0 weights.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path. See qw3_oracle.py.
"""
from .qw3_oracle import *  # noqa: F401,F403
from .qw3_oracle import (  # noqa: F401
    QK8_0, Q8_0_BYTES, OracleError, NonFiniteValue, InvalidShape,
    InvalidSequenceLength, KvCacheOverflow, q8_0_quantize_parts, q8_0_quantize,
    q8_0_unpack, q8_0_dequantize, matrix_from_blocks, rms_norm, rope_inv_freq,
    rope_neox, kv_head_map, attention, silu, swiglu, add_f32, argmax_lowest,
    QLinear, KvCache, OracleModel,
)
