"""Double-precision CPU oracle for the uniform-state canvas pass (TEST INFRASTRUCTURE ONLY).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may import this
package. The product library (``uniform_state_denoising_vocab_b300``) never imports, links or
runs anything here, and this package imports nothing from the product.
"""
from .oracle import (  # noqa: F401
    OR_BF16,
    OR_E4M3,
    OR_F32,
    OR_NVFP4,
    bf16_round,
    build,
    draw,
    e4m3_round,
    e4m3_value,
    e2m1_round,
    e2m1_value,
    quant_rows_nvfp4,
    head_stats,
    keys,
    loop,
    num_threads,
    quant_rows_e4m3,
    select,
    sm64,
    step,
    synth_denoise,
    temperature,
    blocks,
)
