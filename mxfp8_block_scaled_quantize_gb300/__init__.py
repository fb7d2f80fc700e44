"""temx: MXFP8 block-scaled quantisation and MXFP8 GEMM for GB300 (sm_103a).

The compute lives in libtemx.so (hand-written CUDA for sm_103a, C ABI in
include/temx.h); ``binding`` is its ctypes binding and ``workloads`` the
seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    EPI_ACCUMULATE_F32, EPI_BIAS, EPI_BIAS_GELU_AUX, EPI_DGELU, EPI_GELU_AUX, EPI_NONE, TemxError, block_quantize,
    block_quantize_fp32, gemm, gemm_fp32_scales, grouped_gemm, te_mx_block_quantize_fp32,
    te_mx_block_scale_pitch_fp32, te_mx_gemm_fp32_scales,
    grouped_gemm_wgrad, layernorm_quantize, quantize, quantize_colwise_grouped, te_mx_block_quantize,
    te_mx_grouped_gemm_wgrad, te_mx_layernorm_quantize, te_mx_quantize_colwise_grouped,
    te_mx_device_status, te_mx_gemm, te_mx_gemm_workspace_size, te_mx_grouped_gemm, te_mx_quantize,
    te_mx_scale_pitch, te_mx_version,
)
