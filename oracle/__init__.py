"""CPU oracle (test infrastructure; see ``mx_oracle`` for what it defines).

Only ``tests/``, the package entry point's ``smoke()`` and the bench's CPU
baseline may import this package.
"""
from .mx_oracle import *  # noqa: F401,F403
from .mx_oracle import (  # noqa: F401
    bf16_bits_to_f64, bf16_round, block_scale_exponent, column_sums, dequantize, dgelu_tanh, e4m3_decode, e4m3_encode,
    f64_to_bf16_bits, gelu_tanh, gemm_error_bound, grouped_layout, mx_gemm, mx_gemm_dgelu, mx_grouped_gemm,
    mx_grouped_wgrad, quantize_colwise_grouped,
    mx_scale_exponent, quantize_block, quantize_colwise, quantize_rowwise,
    block_gemm_fp32, block_scale_fp32, dequantize_fp32, quantize_block_fp32,
)
