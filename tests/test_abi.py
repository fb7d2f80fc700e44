"""The C-ABI library loads and exports every symbol include/temx.h declares
(no GPU needed), and the host-side helpers behave as documented."""
import os
import re

import pytest

from mxfp8_block_scaled_quantize_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "temx.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(te_mx_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from mxfp8_block_scaled_quantize_gb300 import _build
        _build.build()
    return binding.lib()


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("te_mx_quantize", "te_mx_gemm", "te_mx_grouped_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_scale_pitch(lib):
    assert binding.te_mx_scale_pitch(32) == 16
    assert binding.te_mx_scale_pitch(1024) == 32
    assert binding.te_mx_scale_pitch(7168) == 224
    assert binding.te_mx_scale_pitch(8192 + 32) == 272
    assert binding.te_mx_gemm_workspace_size(4096, 4096, 4096, 0) == 0


def test_version(lib):
    assert "sm_103a" in binding.te_mx_version()


def test_host_validation_rejects_bad_arguments_before_any_launch(lib):
    # these fail argument checks on the host, so they need no GPU
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_quantize(16, 32, 32, 32, 16, 0, 16, 0, 0, 0, 0)      # q_row without s_row
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):
        binding.te_mx_quantize(16, 32, 48, 48, 16, 16, 16, 0, 0, 0, 0)     # cols % 32
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):
        binding.te_mx_quantize(16, 48, 32, 32, 0, 0, 0, 16, 16, 16, 0)     # colwise rows % 32
    with pytest.raises(binding.TemxError, match="MISALIGNED"):
        binding.te_mx_quantize(8, 32, 32, 32, 16, 16, 16, 0, 0, 0, 0)      # x not 16-aligned
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):
        binding.te_mx_gemm(16, 16, 16, 16, 16, 16, 128, 128, 96, 0, 0, 16, 0, 0, 0, 0)   # K % 128
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_gemm(16, 16, 16, 16, 16, 16, 128, 128, 128, 0, 1, 16, 0, 0, 0, 0)  # bias missing
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_gemm(16, 16, 16, 16, 16, 16, 128, 128, 128, 0, 2, 16, 0, 0, 0, 0)  # aux missing
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_grouped_gemm(0, 16, 128, 16, 16, 16, 16, 16, 16, 128, 128, 0, 0, 16, 0, 0, 0, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_block_quantize(16, 128, 128, 128, 2, 16, 16, 16, 0, 0, 0, 0)   # block_2d not 0/1
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):
        binding.te_mx_block_quantize(16, 128, 48, 48, 0, 16, 16, 16, 0, 0, 0, 0)     # cols % 32
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # gamma missing
        binding.te_mx_layernorm_quantize(16, 32, 64, 64, 0, 16, 1e-5, 16, 16, 16, 0, 0, 0, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # eps <= 0
        binding.te_mx_layernorm_quantize(16, 32, 64, 64, 16, 16, 0.0, 16, 16, 16, 0, 0, 0, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # hidden % 32
        binding.te_mx_layernorm_quantize(16, 32, 48, 48, 16, 16, 1e-5, 16, 16, 16, 0, 0, 0, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # mu / rsigma missing
        binding.te_mx_layernorm_quantize(16, 32, 64, 64, 16, 16, 1e-5, 16, 16, 16, 0, 0, 0, 0, 0, 0)
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # hidden too large
        binding.te_mx_layernorm_quantize(16, 32, 32800, 32800, 16, 16, 1e-5, 16, 16, 2064, 0, 0, 0, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # accumulate with a bias
        binding.te_mx_gemm(16, 16, 16, 16, 16, 16, 128, 128, 128, 16, 5, 16, 0, 0, 0, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # accumulate is not for the grouped GEMM
        binding.te_mx_grouped_gemm(2, 16, 128, 16, 16, 16, 16, 16, 16, 128, 128, 0, 5, 16, 0, 0, 0, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # wgrad accumulate flag not 0/1
        binding.te_mx_grouped_gemm_wgrad(2, 16, 128, 16, 16, 16, 16, 128, 128, 128, 16, 2, 16, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_block_quantize_fp32(16, 128, 128, 128, 2, 16, 16, 4, 0, 0, 0, 0)  # block_2d not 0/1
    with pytest.raises(binding.TemxError, match="MISALIGNED"):
        binding.te_mx_block_quantize_fp32(16, 128, 512, 512, 0, 16, 16, 2, 0, 0, 0, 0)  # ld_s_row % 4
    with pytest.raises(binding.TemxError, match="MISALIGNED"):
        binding.te_mx_block_quantize_fp32(16, 128, 640, 640, 0, 16, 16, 4, 0, 0, 0, 0)  # ld_s_row < 5 blocks
    with pytest.raises(binding.TemxError, match="MISALIGNED"):
        binding.te_mx_block_quantize_fp32(16, 128, 128, 128, 0, 0, 0, 0, 16, 8, 4, 0)   # s_col not 16-aligned
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):
        binding.te_mx_block_quantize_fp32(16, 128, 48, 48, 0, 16, 16, 4, 0, 0, 0, 0)    # cols % 32
    assert binding.te_mx_block_scale_pitch_fp32(7168) == 56 and binding.te_mx_block_scale_pitch_fp32(130) == 4
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # b_blocks_2d not 0/1
        binding.te_mx_gemm_fp32_scales(16, 16, 4, 16, 16, 4, 2, 128, 128, 256, 0, 0, 16, 0, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):      # no accumulating epilogue
        binding.te_mx_gemm_fp32_scales(16, 16, 4, 16, 16, 4, 1, 128, 128, 256, 0, 5, 16, 0, 0)
    with pytest.raises(binding.TemxError, match="MISALIGNED"):       # scale pitch % 4
        binding.te_mx_gemm_fp32_scales(16, 16, 2, 16, 16, 4, 1, 128, 128, 256, 0, 0, 16, 0, 0)
    with pytest.raises(binding.TemxError, match="MISALIGNED"):       # scale pitch < K/128
        binding.te_mx_gemm_fp32_scales(16, 16, 4, 16, 16, 4, 1, 128, 128, 1024, 0, 0, 16, 0, 0)
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # K % 128
        binding.te_mx_gemm_fp32_scales(16, 16, 4, 16, 16, 4, 1, 128, 128, 96, 0, 0, 16, 0, 0)
    binding.te_mx_gemm_fp32_scales(16, 16, 4, 16, 16, 4, 1, 0, 128, 256, 0, 0, 16, 0, 0)   # M == 0: no-op
    # zero-sized problems are no-ops
    binding.te_mx_layernorm_quantize(16, 0, 64, 64, 16, 16, 1e-5, 16, 16, 16, 0, 0, 0, 0, 0, 0)
    binding.te_mx_block_quantize(0, 0, 128, 128, 1, 0, 0, 0, 0, 0, 0, 0)
    binding.te_mx_quantize(0, 0, 64, 64, 0, 0, 0, 0, 0, 0, 0)
    binding.te_mx_gemm(16, 16, 16, 16, 16, 16, 0, 128, 128, 0, 0, 16, 0, 0, 0, 0)


def test_host_validation_of_the_backward_and_grouped_entry_points(lib):
    # te_mx_quantize_dbias: checks before any launch
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):         # dbias missing
        binding.te_mx_quantize_dbias(16, 32, 64, 64, 16, 16, 16, 0, 0, 0, 0, 16, 1 << 20, 0)
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # cols % 32
        binding.te_mx_quantize_dbias(16, 32, 48, 48, 16, 16, 16, 0, 0, 0, 16, 16, 1 << 20, 0)
    # (the dbias alignment and workspace checks follow the device check, so they need a GPU)
    assert binding.te_mx_quantize_dbias_workspace_size(32, 64) > 0
    # te_mx_quantize_colwise_grouped
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):         # no groups
        binding.te_mx_quantize_colwise_grouped(16, 128, 64, 64, 0, 16, 16, 256, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):         # more than 1024 groups
        binding.te_mx_quantize_colwise_grouped(16, 128, 64, 64, 1025, 16, 16, 256, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # cols % 32
        binding.te_mx_quantize_colwise_grouped(16, 128, 48, 48, 2, 16, 16, 256, 16, 16, 0)
    with pytest.raises(binding.TemxError, match="MISALIGNED"):          # ld_q % 16
        binding.te_mx_quantize_colwise_grouped(16, 128, 64, 64, 2, 16, 16, 200, 16, 16, 0)
    # te_mx_grouped_gemm_wgrad
    with pytest.raises(binding.TemxError, match="UNSUPPORTED_SHAPE"):   # N % 16
        binding.te_mx_grouped_gemm_wgrad(2, 16, 128, 16, 16, 16, 16, 128, 120, 256, 16, 0, 16, 0)
    with pytest.raises(binding.TemxError, match="MISALIGNED"):          # ld_s < 16
        binding.te_mx_grouped_gemm_wgrad(2, 16, 128, 16, 16, 16, 16, 128, 128, 256, 0, 0, 16, 0)
    # the failing call left its message
    assert binding.lib().te_mx_last_error()


@pytest.mark.parametrize("groups", [1, 3, 128])
def test_grouped_widths_cover_every_partition(lib, groups):
    # the host widths suffice for any split of total_m tokens into `groups` experts
    import numpy as np
    rng = np.random.default_rng(groups)
    for total in (0, 1, 127, 128, 129, 4096, 131072):
        cw = binding.te_mx_grouped_code_width(total, groups)
        sw = binding.te_mx_grouped_scale_width(total, groups)
        assert cw % 16 == 0 and sw % 16 == 0 and sw >= 16
        for _ in range(20):
            cuts = np.sort(rng.integers(0, total + 1, groups - 1))
            m = np.diff(np.concatenate([[0], cuts, [total]]))
            kp = (m + 127) // 128 * 128
            assert kp.sum() <= cw
            assert ((kp // 32 + 15) // 16 * 16).sum() <= sw
