"""GPU parity of te_mx_block_quantize (Float8BlockScaling, E8M0-cast scales)
against the oracle: bit-exact codes and scales, canary-guarded outputs.

Covers 1x128 / 128x1 and 128x128 blocks in each orientation subset, shapes
spanning several tiles with ragged right and bottom edges, every bf16 bit
pattern (NaN/inf blocks included), wide exponent ranges, pitched input, the
full-size FFN tensors (sampled rows and columns, 1D for X and dY, 2D for W),
and the block-scaled GEMM (1Dx1D and 1Dx2D) through te_mx_gemm on the GPU
quantiser's own output, within the GEMM bound.
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu


def randn_bf16(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


def check(x_cpu, block_2d, rowwise=True, colwise=True):
    got = U.gpu_quantize(x_cpu.cuda(), rowwise, colwise, block_2d=block_2d)
    q_row, s_row, q_col, s_col = O.quantize_block(U.bf16_bits(x_cpu), block_2d)
    if rowwise:
        U.assert_bytes_equal(got["s_row"], s_row, "row-wise scales")
        U.assert_bytes_equal(got["q_row"], q_row, "row-wise codes")
    if colwise:
        U.assert_bytes_equal(got["s_col"], s_col, "column-wise scales")
        U.assert_bytes_equal(got["q_col"], q_col, "column-wise codes")


SHAPES = [(128, 128), (32, 32), (96, 160), (256, 384), (544, 2080), (1024, 1056), (2048, 320)]


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_both_orientations(rows, cols, block_2d):
    check(randn_bf16(rows, cols, rows * 5 + cols + block_2d, std=2.0), block_2d)


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_one_orientation(rowwise, colwise, block_2d):
    check(randn_bf16(416, 672, 11 + 2 * block_2d + rowwise), block_2d, rowwise, colwise)


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 96), (200, 416)])
def test_rowwise_ragged_rows(rows, cols, block_2d):
    check(randn_bf16(rows, cols, rows + cols), block_2d, rowwise=True, colwise=False)


@pytest.mark.parametrize("block_2d", [False, True])
def test_every_bf16_pattern(block_2d):
    perm = np.random.default_rng(1).permutation(1 << 16).astype(np.uint16)
    for shape in ((512, 128), (128, 512), (2048, 32)):
        check(U.from_bits(np.ascontiguousarray(perm.reshape(shape))), block_2d)
    # finite patterns only, so that blocks are not swamped by NaN/inf
    finite = perm[(perm & 0x7F80) != 0x7F80][: 256 * 224]
    check(U.from_bits(np.ascontiguousarray(finite.reshape(256, 224))), block_2d)


@pytest.mark.parametrize("block_2d", [False, True])
def test_wide_exponent_range_and_outliers(block_2d):
    g = torch.Generator().manual_seed(6)
    x = torch.randn(512, 768, generator=g) * torch.pow(2.0, torch.randint(-130, 120, (512, 1), generator=g).float())
    x[:, ::97] *= 64.0
    x[7, :] = 0.0
    x[130:140, 300:400] = -0.0
    check(x.to(torch.bfloat16), block_2d)


def test_pitched_input_and_scale_pitch():
    base = randn_bf16(256, 512, 78)
    x = base.cuda()[:, :320]                     # ld_x = 512 > cols = 320
    out = {"q_row": torch.empty(256, 320, dtype=torch.uint8, device="cuda"),
           "s_row": torch.full((256, 32), 0xA5, dtype=torch.uint8, device="cuda"),
           "q_col": torch.empty(320, 256, dtype=torch.uint8, device="cuda"),
           "s_col": torch.full((320, 48), 0xA5, dtype=torch.uint8, device="cuda")}
    binding.block_quantize(x, block_2d=False, rowwise=True, colwise=True, out=out)
    binding.te_mx_device_status()
    q_row, s_row, q_col, s_col = O.quantize_block(U.bf16_bits(base[:, :320]), False)
    U.assert_bytes_equal(out["q_row"].cpu().numpy(), q_row, "row codes")
    U.assert_bytes_equal(out["q_col"].cpu().numpy(), q_col, "column codes")
    sr, sc = out["s_row"].cpu().numpy(), out["s_col"].cpu().numpy()
    U.assert_bytes_equal(sr[:, :10], s_row, "row scales")
    U.assert_bytes_equal(sc[:, :8], s_col, "column scales")
    assert np.all(sr[:, 10:] == 0xA5) and np.all(sc[:, 8:] == 0xA5)


def test_empty_is_noop():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    binding.block_quantize(x, block_2d=True, rowwise=True, colwise=True)
    binding.te_mx_device_status()


def _sampled_full_size(x_cpu, block_2d, seed, n_blocks=3):
    """Whole 128-row / 128-column bands sampled (a 1D or 2D block needs its
    full band), last band included."""
    x = x_cpu.cuda()
    out = binding.block_quantize(x, block_2d=block_2d, rowwise=True, colwise=True)
    binding.te_mx_device_status()
    rows, cols = x_cpu.shape
    rng = np.random.default_rng(seed)
    rb = sorted(set(rng.choice(rows // 128, n_blocks, replace=False).tolist()) | {rows // 128 - 1})
    cb = sorted(set(rng.choice(cols // 128, n_blocks, replace=False).tolist()) | {cols // 128 - 1})
    for r in rb:                                  # row band: rows r*128.., all columns
        q_row, s_row, _, _ = O.quantize_block(U.bf16_bits(x_cpu[r * 128:(r + 1) * 128]), block_2d)
        U.assert_bytes_equal(out["q_row"][r * 128:(r + 1) * 128].cpu().numpy(), q_row, f"row codes, band {r}")
        U.assert_bytes_equal(out["s_row"][r * 128:(r + 1) * 128, : cols // 32].cpu().numpy(), s_row,
                             f"row scales, band {r}")
    for c in cb:                                  # column band: all rows, columns c*128..
        _, _, q_col, s_col = O.quantize_block(U.bf16_bits(x_cpu[:, c * 128:(c + 1) * 128]), block_2d)
        U.assert_bytes_equal(out["q_col"][c * 128:(c + 1) * 128].cpu().numpy(), q_col, f"column codes, band {c}")
        U.assert_bytes_equal(out["s_col"][c * 128:(c + 1) * 128, : rows // 32].cpu().numpy(), s_col,
                             f"column scales, band {c}")


def test_full_size_ffn_tensors():
    d = workloads.make_ffn()
    _sampled_full_size(d["X"], False, 20)       # activations: 1x128 / 128x1
    _sampled_full_size(d["dY"], False, 21)      # gradients: 1x128 / 128x1
    _sampled_full_size(d["W"], True, 22)        # weights: 128x128


def _gemm_check(M, N, K, w_2d, seed):
    from tests.test_gemm_gpu import assert_within_bound, to_f64
    x = randn_bf16(M, K, seed, std=1.0)
    w = randn_bf16(N, K, seed + 1, std=0.02)
    qx = binding.block_quantize(x.cuda(), block_2d=False)
    qw = binding.block_quantize(w.cuda(), block_2d=w_2d)
    d, _ = binding.gemm(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"])
    binding.te_mx_device_status()
    ox = O.quantize_block(U.bf16_bits(x), False)
    ow = O.quantize_block(U.bf16_bits(w), w_2d)
    U.assert_bytes_equal(qx["q_row"].cpu().numpy(), ox[0], "X codes")
    U.assert_bytes_equal(qw["q_row"].cpu().numpy(), ow[0], "W codes")
    ref = O.mx_gemm(ox[0], ox[1], ow[0], ow[1])
    assert_within_bound(to_f64(d), ref["d"], ref["sigma"], "block-scaled D")


@pytest.mark.parametrize("w_2d", [False, True])
def test_block_scaled_gemm(w_2d):
    _gemm_check(384, 512, 1024, w_2d, 30 + w_2d)
