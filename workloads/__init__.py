"""Seeded synthetic inputs for the canvas pass (shared by the CUDA path's tests/bench and the oracle).

This package holds random-number plumbing and the workload recipes only: it contains none of
the sampler's arithmetic (no logits, softmax, top-k, hash or stop rule).
"""
from .gen import (  # noqa: F401
    CONFIGS,
    WorkloadConfig,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_pass_inputs,
    make_loop_inputs,
    normal_f32,
    quantize_rows_e4m3_bits,
    quantize_rows_nvfp4_bits,
    uniform_ints,
)
