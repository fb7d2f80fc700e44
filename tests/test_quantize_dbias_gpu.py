"""GPU parity of te_mx_quantize_dbias: the same bit-exact codes as
te_mx_quantize plus dbias = bf16(column sums) within 2^-7 |exact| +
1e-5 sum|x|, deterministic across calls."""
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


def check_dbias(got_bits, x_cpu):
    s, a = O.column_sums(U.bf16_bits(x_cpu))
    ref = O.bf16_round(s)
    got = O.bf16_bits_to_f64(got_bits)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-5 * a
    bad = ~(np.abs(got - ref) <= bound)
    assert not bad.any(), f"{bad.sum()} columns outside the bound; first {np.argmax(bad)}"


@pytest.mark.parametrize("rows,cols,rowwise,colwise", [
    (64, 64, True, True), (96, 160, True, True), (1024, 1056, True, True),
    (37, 96, True, False), (100, 224, True, False), (512, 1088, False, True), (333, 64, False, False),
])
def test_dbias_with_each_orientation(rows, cols, rowwise, colwise):
    x_cpu = randn_bf16(rows, cols, rows + cols, std=3.0)
    x = x_cpu.cuda()
    o = binding.quantize(x, rowwise, colwise, dbias=True)
    binding.te_mx_device_status()
    check_dbias(U.bf16_bits(o["dbias"]), x_cpu)
    bits = U.bf16_bits(x_cpu)
    if rowwise:
        q, s = O.quantize_rowwise(bits)
        U.assert_bytes_equal(o["q_row"].cpu().numpy(), q, "row codes")
        U.assert_bytes_equal(o["s_row"].cpu().numpy()[:, : cols // 32], s, "row scales")
    if colwise:
        q, s = O.quantize_colwise(bits)
        U.assert_bytes_equal(o["q_col"].cpu().numpy(), q, "col codes")
        U.assert_bytes_equal(o["s_col"].cpu().numpy()[:, : rows // 32], s, "col scales")


def test_dbias_is_deterministic_and_ignores_workspace_contents():
    x = randn_bf16(2048, 4096, 9).cuda()
    ws = torch.full((binding.te_mx_quantize_dbias_workspace_size(2048, 4096),), 0x7F, dtype=torch.uint8, device="cuda")
    a = binding.quantize(x, True, True, dbias=True, workspace=ws)["dbias"].clone()
    ws.fill_(0xFF)
    b = binding.quantize(x, True, True, dbias=True, workspace=ws)["dbias"]
    binding.te_mx_device_status()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_dbias_workspace_too_small_is_rejected():
    x = randn_bf16(128, 256, 1).cuda()
    need = binding.te_mx_quantize_dbias_workspace_size(128, 256)
    assert need == 2 * 256 * 4
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.TemxError, match="WORKSPACE_TOO_SMALL"):
        binding.quantize(x, True, True, dbias=True, workspace=ws)


def test_full_size_fc1_dy_dbias():
    d = workloads.make_fc1()
    dy = d["dY"]
    o = binding.quantize(dy.cuda(), True, True, dbias=True)
    binding.te_mx_device_status()
    check_dbias(U.bf16_bits(o["dbias"]), dy)
