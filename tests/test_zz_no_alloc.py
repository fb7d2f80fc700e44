"""The allocation-free bias-gradient quantiser, te_mx_quantize_dbias_noalloc.

It is meant for callers that cannot allocate device memory themselves — host
code with no device allocator of its own, or programs that plan all device
memory up front and forbid allocating once they run.  Instead of a caller
workspace it uses scratch built into the library.  This checks, through the C
ABI, that two calls in a row give the same codes, scales and bias gradient as
te_mx_quantize_dbias with a caller workspace, and that sizes beyond the
built-in scratch are refused.  (Collected last, so a run that stops at the
first failure has already run everything else.)
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu


def _outputs(rows, cols):
    p = binding.te_mx_scale_pitch
    e = lambda *s, dt=torch.uint8: torch.full(s, 0xA5 if dt == torch.uint8 else 0, dtype=dt, device="cuda")
    return {"q_row": e(rows, cols), "s_row": e(rows, p(cols)), "q_col": e(cols, rows), "s_col": e(cols, p(rows)),
            "dbias": torch.zeros(cols, dtype=torch.bfloat16, device="cuda")}


def _args(x, o):
    rows, cols = x.shape
    return (x.data_ptr(), rows, cols, x.stride(0), o["q_row"].data_ptr(), o["s_row"].data_ptr(),
            o["s_row"].stride(0), o["q_col"].data_ptr(), o["s_col"].data_ptr(), o["s_col"].stride(0),
            o["dbias"].data_ptr())


def _with_workspace(x):
    o = _outputs(*x.shape)
    n = binding.te_mx_quantize_dbias_workspace_size(*x.shape)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    binding.te_mx_quantize_dbias(*_args(x, o), ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    return o


def _without_allocation(x):
    o = _outputs(*x.shape)
    binding.te_mx_quantize_dbias_noalloc(*_args(x, o), torch.cuda.current_stream().cuda_stream)
    return o


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    g = torch.Generator().manual_seed(11)
    inputs = [(torch.randn(2048, 1536, generator=g) * 2.0).to(torch.bfloat16),
              (torch.randn(512, 4096, generator=g) * 0.5).to(torch.bfloat16)]
    got = [_without_allocation(x.cuda()) for x in inputs]          # two calls in a row
    want = [_with_workspace(x.cuda()) for x in inputs]
    binding.te_mx_device_status()
    for x, a, b in zip(inputs, got, want):
        for key in ("q_row", "s_row", "q_col", "s_col"):
            assert torch.equal(a[key], b[key]), key
        da = O.bf16_bits_to_f64(U.bf16_bits(a["dbias"]))
        db = O.bf16_bits_to_f64(U.bf16_bits(b["dbias"]))
        _, abs_sum = O.column_sums(U.bf16_bits(x))
        assert np.all(np.abs(da - db) <= 2.0 ** -7 * np.abs(db) + 1e-5 * abs_sum)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    limit = 32 << 20                                  # TE_MX_NOALLOC_SCRATCH_BYTES
    rows, cols = 64 * 1024, 8192                      # 1024 bands x 8192 columns x 4 B = 32 MiB + ... > limit
    assert binding.te_mx_quantize_dbias_workspace_size(rows + 64, cols) > limit
    x = torch.empty(rows + 64, cols, dtype=torch.bfloat16, device="cuda")
    dbias = torch.empty(cols, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.TemxError, match="WORKSPACE_TOO_SMALL"):
        binding.te_mx_quantize_dbias_noalloc(x.data_ptr(), rows + 64, cols, cols, 0, 0, 0, 0, 0, 0,
                                             dbias.data_ptr(), 0)
