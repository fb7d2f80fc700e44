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


def _assert_same(a, b, what):
    # same kernels, same band layout, same fixed summation order: every byte equal
    for key in ("q_row", "s_row", "q_col", "s_col", "dbias"):
        assert torch.equal(a[key], b[key]), f"{what}: {key} differs"


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    g = torch.Generator().manual_seed(11)
    inputs = [(torch.randn(2048, 1536, generator=g) * 2.0).to(torch.bfloat16),
              (torch.randn(512, 4096, generator=g) * 0.5).to(torch.bfloat16)]
    got = [_without_allocation(x.cuda()) for x in inputs]          # two calls in a row
    want = [_with_workspace(x.cuda()) for x in inputs]
    binding.te_mx_device_status()
    for i, (x, a, b) in enumerate(zip(inputs, got, want)):
        _assert_same(a, b, f"call {i}")
        # and the bias gradient is within the documented bound of the exact column sums
        exact, abs_sum = O.column_sums(U.bf16_bits(x))
        da = O.bf16_bits_to_f64(U.bf16_bits(a["dbias"]))
        assert np.all(np.abs(da - exact) <= 2.0 ** -7 * np.abs(exact) + 1e-5 * abs_sum)


def test_noalloc_small_call_after_a_large_one():
    # a large call leaves band sums all over the shared scratch; a smaller call
    # after it must not pick any of them up
    g = torch.Generator().manual_seed(12)
    big = (torch.randn(8192, 2048, generator=g) * 3.0).to(torch.bfloat16).cuda()
    small = (torch.randn(96, 160, generator=g) * 0.25).to(torch.bfloat16).cuda()
    _without_allocation(big)
    a = _without_allocation(small)
    b = _with_workspace(small)
    binding.te_mx_device_status()
    _assert_same(a, b, "small after large")


def test_noalloc_size_limit():
    limit = 32 << 20                                  # TE_MX_NOALLOC_SCRATCH_BYTES
    # one 64-row band x 8M columns x 4 bytes = exactly the limit: accepted
    # (dbias only, so the input is one row of 16 MB)
    cols = limit // 4
    assert binding.te_mx_quantize_dbias_workspace_size(1, cols) == limit
    x = (torch.randn(1, cols, generator=torch.Generator().manual_seed(13)) * 5.0).to(torch.bfloat16).cuda()
    o = {k: None for k in ("q_row", "s_row", "q_col", "s_col")}
    dbias = torch.zeros(cols, dtype=torch.bfloat16, device="cuda")
    binding.te_mx_quantize_dbias_noalloc(x.data_ptr(), 1, cols, cols, 0, 0, 0, 0, 0, 0, dbias.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    binding.te_mx_device_status()
    assert torch.equal(dbias, x[0]), "the column sums of a single row are the row itself"
    # beyond the limit: refused on the host before any launch (so the small
    # buffer behind the oversized shape is never read)
    stub = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    for rows, c in ((1, cols + 32), (65, cols // 2 + 32), (64 * 1024 + 64, 8192)):
        assert binding.te_mx_quantize_dbias_workspace_size(rows, c) > limit
        with pytest.raises(binding.TemxError, match="WORKSPACE_TOO_SMALL"):
            binding.te_mx_quantize_dbias_noalloc(stub.data_ptr(), rows, c, c, 0, 0, 0, 0, 0, 0,
                                                 stub.data_ptr(), 0)
