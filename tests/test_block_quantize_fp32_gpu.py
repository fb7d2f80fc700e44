"""GPU parity of te_mx_block_quantize_fp32 (Float8BlockScaling keeping FP32
scales) against the oracle: bit-exact codes and fp32 scale bit patterns.

Covers 1x128 / 128x1 and 128x128 blocks in each orientation subset, shapes
spanning several tiles with ragged right and bottom edges, every bf16 bit
pattern (NaN/inf blocks included), wide exponent ranges down to subnormal
amax (the capped multiplier), zero blocks, pitched input with canaries past
the scale pitch, and the full-size FFN tensors (sampled bands).
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu

CANARY = 0xA5A5A5A5
CANARY_I32 = CANARY - (1 << 32)             # the same bit pattern as int32


def randn_bf16(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


def f32_bits(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def run(x, block_2d, rowwise=True, colwise=True, extra_pitch=0):
    rows, cols = x.shape
    out = {}
    if rowwise:
        pr = binding.te_mx_block_scale_pitch_fp32(cols) + extra_pitch
        out["q_row"] = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
        out["s_row"] = torch.full((rows, pr), CANARY_I32, dtype=torch.int32, device="cuda").view(torch.float32)
    if colwise:
        pc = binding.te_mx_block_scale_pitch_fp32(rows) + extra_pitch
        out["q_col"] = torch.empty(cols, rows, dtype=torch.uint8, device="cuda")
        out["s_col"] = torch.full((cols, pc), CANARY_I32, dtype=torch.int32, device="cuda").view(torch.float32)
    binding.block_quantize_fp32(x, block_2d=block_2d, rowwise=rowwise, colwise=colwise, out=out)
    binding.te_mx_device_status()
    return {k: v.cpu().numpy() for k, v in out.items()}


def check(x_cpu, block_2d, rowwise=True, colwise=True, x_gpu=None, extra_pitch=0):
    got = run(x_cpu.cuda() if x_gpu is None else x_gpu, block_2d, rowwise, colwise, extra_pitch)
    q_row, s_row, q_col, s_col = O.quantize_block_fp32(U.bf16_bits(x_cpu), block_2d)
    for key, q, s in (("row", q_row, s_row), ("col", q_col, s_col)):
        if ("q_" + key) not in got:
            continue
        gs = f32_bits(got["s_" + key])
        n = s.shape[1]
        U.assert_bytes_equal(got["q_" + key], q, key + " codes")
        assert np.array_equal(gs[:, :n], f32_bits(s)), key + " scales"
        assert np.all(gs[:, n:] == CANARY), key + " scales written past the blocks"


SHAPES = [(128, 128), (32, 32), (96, 160), (256, 384), (544, 2080), (1024, 1056), (2048, 320)]


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_both_orientations(rows, cols, block_2d):
    check(randn_bf16(rows, cols, rows * 7 + cols + block_2d, std=2.0), block_2d)


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_one_orientation(rowwise, colwise, block_2d):
    check(randn_bf16(416, 672, 13 + 2 * block_2d + rowwise), block_2d, rowwise, colwise)


@pytest.mark.parametrize("block_2d", [False, True])
@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 96), (200, 416)])
def test_rowwise_ragged_rows(rows, cols, block_2d):
    check(randn_bf16(rows, cols, rows + cols + 1), block_2d, rowwise=True, colwise=False)


@pytest.mark.parametrize("block_2d", [False, True])
def test_every_bf16_pattern(block_2d):
    perm = np.random.default_rng(2).permutation(1 << 16).astype(np.uint16)
    for shape in ((512, 128), (128, 512), (2048, 32)):
        check(U.from_bits(np.ascontiguousarray(perm.reshape(shape))), block_2d)
    finite = perm[(perm & 0x7F80) != 0x7F80][: 256 * 224]
    check(U.from_bits(np.ascontiguousarray(finite.reshape(256, 224))), block_2d)


@pytest.mark.parametrize("block_2d", [False, True])
def test_wide_exponents_subnormal_and_zero_blocks(block_2d):
    g = torch.Generator().manual_seed(8)
    x = torch.randn(512, 768, generator=g) * torch.pow(2.0, torch.randint(-135, 120, (512, 1), generator=g).float())
    x[:, ::97] *= 64.0
    x[7, :] = 0.0
    x[130:140, 300:400] = -0.0
    x[256:384, 512:640] = 0.0                     # a whole zero 128x128 block
    check(x.to(torch.bfloat16), block_2d)


def test_pitched_input_and_scale_pitch():
    base = randn_bf16(256, 512, 79)
    check(base[:, :320], False, x_gpu=base.cuda()[:, :320], extra_pitch=4)


def test_empty_is_noop():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    binding.block_quantize_fp32(x, block_2d=True, rowwise=True, colwise=True)
    binding.te_mx_device_status()


def _sampled_full_size(x_cpu, block_2d, seed, n_blocks=3):
    x = x_cpu.cuda()
    out = binding.block_quantize_fp32(x, block_2d=block_2d, rowwise=True, colwise=True)
    binding.te_mx_device_status()
    rows, cols = x_cpu.shape
    rng = np.random.default_rng(seed)
    rb = sorted(set(rng.choice(rows // 128, n_blocks, replace=False).tolist()) | {rows // 128 - 1})
    cb = sorted(set(rng.choice(cols // 128, n_blocks, replace=False).tolist()) | {cols // 128 - 1})
    for r in rb:
        q_row, s_row, _, _ = O.quantize_block_fp32(U.bf16_bits(x_cpu[r * 128:(r + 1) * 128]), block_2d)
        U.assert_bytes_equal(out["q_row"][r * 128:(r + 1) * 128].cpu().numpy(), q_row, f"row codes, band {r}")
        got = f32_bits(out["s_row"][r * 128:(r + 1) * 128, : cols // 128].cpu().numpy())
        assert np.array_equal(got, f32_bits(s_row)), f"row scales, band {r}"
    for c in cb:
        _, _, q_col, s_col = O.quantize_block_fp32(U.bf16_bits(x_cpu[:, c * 128:(c + 1) * 128]), block_2d)
        U.assert_bytes_equal(out["q_col"][c * 128:(c + 1) * 128].cpu().numpy(), q_col, f"column codes, band {c}")
        got = f32_bits(out["s_col"][c * 128:(c + 1) * 128, : rows // 128].cpu().numpy())
        assert np.array_equal(got, f32_bits(s_col)), f"column scales, band {c}"


def test_full_size_ffn_tensors():
    d = workloads.make_ffn()
    _sampled_full_size(d["X"], False, 40)
    _sampled_full_size(d["W"], True, 41)
