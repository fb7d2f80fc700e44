"""GPU parity of te_mx_quantize against the oracle: bit-exact codes and scales.

Covers small and ragged shapes spanning several units and a ragged tail,
every bf16 bit pattern, the hand-worked golden blocks, wide exponent ranges,
and the full-size workload tensors (sampled rows and columns), with canary
guards around every output.
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U
from tests.test_oracle_quantize import parse_golden, to_bf16_bits

pytestmark = pytest.mark.gpu


def check_against_oracle(x_cpu: torch.Tensor, rowwise=True, colwise=True):
    x = x_cpu.cuda()
    got = U.gpu_quantize(x, rowwise, colwise)
    bits = U.bf16_bits(x_cpu)
    if rowwise:
        q, s = O.quantize_rowwise(bits)
        U.assert_bytes_equal(got["s_row"], s, "row-wise scales")
        U.assert_bytes_equal(got["q_row"], q, "row-wise codes")
    if colwise:
        q, s = O.quantize_colwise(bits)
        U.assert_bytes_equal(got["s_col"], s, "column-wise scales")
        U.assert_bytes_equal(got["q_col"], q, "column-wise codes")


def randn_bf16(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(32, 32), (32, 64), (64, 96), (96, 160), (256, 256),
                                       (1024, 1056), (544, 2048), (2048, 320)])
def test_both_orientations_small(rows, cols):
    check_against_oracle(randn_bf16(rows, cols, rows * 7 + cols))


@pytest.mark.parametrize("rows,cols", [(1, 32), (5, 64), (37, 96), (100, 224), (1000, 1024)])
def test_rowwise_ragged_rows(rows, cols):
    check_against_oracle(randn_bf16(rows, cols, rows + cols), rowwise=True, colwise=False)


@pytest.mark.parametrize("rows,cols", [(64, 96), (512, 1088)])
def test_colwise_only(rows, cols):
    check_against_oracle(randn_bf16(rows, cols, 3 * rows + cols), rowwise=False, colwise=True)


def test_every_bf16_pattern():
    # all 65536 patterns (incl. subnormals, +-0, inf, NaN) in a [2048 x 32] matrix,
    # shuffled so that blocks mix magnitudes in both orientations
    perm = np.random.default_rng(0).permutation(1 << 16).astype(np.uint16)
    bits = perm.reshape(2048, 32)
    check_against_oracle(U.from_bits(bits))
    check_against_oracle(U.from_bits(np.ascontiguousarray(bits.reshape(64, 1024))))


def test_golden_blocks_on_gpu():
    blocks = parse_golden()
    rows = np.stack([to_bf16_bits(b["vals"]) for b in blocks])        # [nblk, 32]
    pad = (-len(blocks)) % 32
    mat = np.concatenate([rows, np.zeros((pad, 32), np.uint16)])
    x = U.from_bits(mat).cuda()
    got = U.gpu_quantize(x, rowwise=True, colwise=False)
    for i, b in enumerate(blocks):
        assert int(got["s_row"][i, 0]) == b["scale"], b["name"]
        assert got["q_row"][i].tolist() == b["q"], b["name"]
    got = U.gpu_quantize(x.t().contiguous(), rowwise=False, colwise=True)
    for i, b in enumerate(blocks):
        assert int(got["s_col"][i, 0]) == b["scale"], b["name"]
        assert got["q_col"][i].tolist() == b["q"], b["name"]


def test_wide_exponent_range_and_outliers():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(512, 1024, generator=g) * torch.pow(2.0, torch.randint(-130, 120, (512, 1), generator=g).float())
    x[:, ::97] *= 64.0
    x[7, :] = 0.0
    x[9, 100:140] = -0.0
    check_against_oracle(x.to(torch.bfloat16))


def test_pitched_input_and_scale_pitch():
    base = randn_bf16(128, 256, 77)
    x = base.cuda()[:, :192]                     # ld_x = 256 > cols = 192
    assert x.stride(0) == 256
    out = {"q_row": torch.empty(128, 192, dtype=torch.uint8, device="cuda"),
           "s_row": torch.full((128, 32), 0xA5, dtype=torch.uint8, device="cuda")}   # pitch 32 > 16
    binding.quantize(x, rowwise=True, colwise=False, out=out)
    q, s = O.quantize_rowwise(U.bf16_bits(base[:, :192]))
    U.assert_bytes_equal(out["q_row"].cpu().numpy(), q, "codes")
    sc = out["s_row"].cpu().numpy()
    U.assert_bytes_equal(sc[:, :6], s, "scales")
    assert np.all(sc[:, 6:] == 0xA5)


def test_empty_is_noop():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    binding.quantize(x, rowwise=True, colwise=True)
    binding.te_mx_device_status()


def _sampled_full_size(x_cpu: torch.Tensor, seed: int, n_rows=48, n_cols=64):
    x = x_cpu.cuda()
    out = binding.quantize(x, rowwise=True, colwise=True)
    binding.te_mx_device_status()
    rows, cols = x_cpu.shape
    rng = np.random.default_rng(seed)
    r_idx = np.sort(rng.choice(rows, n_rows, replace=False))
    c_idx = np.sort(rng.choice(cols, n_cols, replace=False))
    r_idx[-1], c_idx[-1] = rows - 1, cols - 1          # include the last row / column
    bits_r = U.bf16_bits(x_cpu[torch.from_numpy(r_idx)])
    q, s = O.quantize_rowwise(bits_r)
    ri = torch.from_numpy(r_idx).cuda()
    U.assert_bytes_equal(out["q_row"][ri].cpu().numpy(), q, "row-wise codes (sampled rows)")
    U.assert_bytes_equal(out["s_row"][ri][:, : cols // 32].cpu().numpy(), s, "row-wise scales (sampled rows)")
    bits_c = U.bf16_bits(x_cpu[:, torch.from_numpy(c_idx)])
    q, s = O.quantize_colwise(bits_c)
    ci = torch.from_numpy(c_idx).cuda()
    U.assert_bytes_equal(out["q_col"][ci].cpu().numpy(), q, "column-wise codes (sampled columns)")
    U.assert_bytes_equal(out["s_col"][ci][:, : rows // 32].cpu().numpy(), s, "column-wise scales (sampled columns)")


def test_full_size_fc1_tensors():
    d = workloads.make_fc1()
    _sampled_full_size(d["X"], 1)
    _sampled_full_size(d["dY"], 2)


def test_full_size_ffn_tensors():
    d = workloads.make_ffn()
    for i, key in enumerate(("X", "W", "dY")):
        _sampled_full_size(d[key], 10 + i)
