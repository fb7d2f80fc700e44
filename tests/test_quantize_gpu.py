"""GPU parity of te_mx_quantize against the oracle: bit-exact codes and scales.

Covers small and ragged shapes spanning several units and a ragged tail,
every bf16 bit pattern, the hand-worked golden blocks, wide exponent ranges,
with canary guards around every output; every code and scale byte of every
tensor the five workloads quantise (the oracle runs slab by slab in a spawn
process pool); and an input larger than 2^31 bytes.
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


def _every_byte(x_cpu, rowwise, colwise, what):
    x = x_cpu.cuda()
    out = binding.quantize(x, rowwise=rowwise, colwise=colwise)
    binding.te_mx_device_status()
    U.check_every_byte(out, x_cpu, rowwise, colwise, what)


def test_full_size_tiny_every_byte():
    d = workloads.make_tiny()
    _every_byte(d["A"], True, True, "tiny A")
    _every_byte(d["B"], True, True, "tiny B")


def test_full_size_qkv_every_byte():
    d = workloads.make_qkv()
    _every_byte(d["X"], True, True, "qkv X")
    _every_byte(d["W"], True, True, "qkv W")


def test_full_size_fc1_every_byte():
    d = workloads.make_fc1()
    for key in ("X", "W", "dY"):
        _every_byte(d[key], True, True, "fc1 " + key)


def test_full_size_ffn_every_byte():
    d = workloads.make_ffn()
    _every_byte(d["X"], True, True, "ffn X")
    _every_byte(d["W"], True, True, "ffn W")         # row-wise: fprop; column-wise: dgrad
    _every_byte(d["dY"], True, True, "ffn dY")


def test_full_size_moe_every_byte():
    # the grouped GEMM's operands: X [131072 x 4096] and the stacked expert
    # weights [128*1536 x 4096] (1.6 GB of bf16), row-wise
    d = U.moe_workload()
    _every_byte(d["X"], True, False, "moe X")
    _every_byte(d["W"].view(128 * 1536, 4096), True, False, "moe W")


def _big_rows(base, rows):
    """Rows of the 2 GiB test matrix: row r = base[r % 4096] * 2^((r // 4096) % 16 - 8)
    (a power-of-two scaling, exact in bf16)."""
    rows = torch.as_tensor(rows)
    k = ((rows // 4096) % 16 - 8).to(torch.float32)
    return (base[rows % 4096].float() * torch.pow(2.0, k)[:, None]).to(torch.bfloat16)


def test_input_and_outputs_past_2_31_bytes():
    # [262208 x 4096] bf16 = 2^31 + 512 KiB of input: the last 64 rows (and
    # their column blocks) are read past byte 2^31; 64-bit offsets everywhere
    C = 4096
    R = (1 << 31) // (2 * C) + 64
    base = workloads.normal_bf16((4096, C), 1.0, 90)
    bd = base.cuda()
    x = torch.empty(R, C, dtype=torch.bfloat16, device="cuda")
    for b0 in range(0, R, 4096):
        n = min(4096, R - b0)
        x[b0:b0 + n] = _big_rows(bd, torch.arange(b0, b0 + n, device="cuda"))
    out = binding.quantize(x, rowwise=True, colwise=True)
    binding.te_mx_device_status()
    rows = U.band_rows(R, 4096, 3, extra=list(range(R - 64, R)) + [R - 65, (1 << 31) // (2 * C) - 1])
    U.check_rows_rowwise(out["q_row"], out["s_row"], _big_rows(base, rows), rows, "row-wise, rows", only_rows=True)
    # whole columns (each spans every row, so their last blocks are read past 2^31)
    cols = np.array([0, 1, 777, 2048, C - 1])
    xc = _big_rows(base[:, torch.from_numpy(cols)], torch.arange(R))
    U.check_cols_colwise(out["q_col"], out["s_col"], xc, np.arange(len(cols)), "column-wise, columns",
                         dev_index=cols)
