"""Shared helpers for the GPU parity tests (marshalling between torch and numpy)."""
import numpy as np
import torch

from mxfp8_block_scaled_quantize_gb300 import binding

GUARD = 256          # canary bytes after every output buffer
CANARY = 0xA5


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def guarded_u8(rows, cols, dev="cuda"):
    """uint8 [rows, cols] view into a buffer filled with the canary, with
    GUARD spare bytes after it; returns (view, whole buffer)."""
    buf = torch.full((rows * cols + GUARD,), CANARY, dtype=torch.uint8, device=dev)
    return buf[: rows * cols].view(rows, cols), buf


def guarded_bf16(rows, cols, dev="cuda"):
    buf = torch.full((rows * cols + GUARD // 2,), 0, dtype=torch.int16, device=dev)
    buf.fill_(-0x5A5B)  # 0xA5A5 pattern
    return buf[: rows * cols].view(torch.bfloat16).view(rows, cols), buf


def check_guard(buf, n_used):
    tail = buf.view(torch.uint8)[n_used * buf.element_size():].cpu().numpy() if buf.dtype != torch.uint8 \
        else buf[n_used:].cpu().numpy()
    assert np.all(tail == CANARY), "write past the end of an output buffer"


def gpu_quantize(x: torch.Tensor, rowwise=True, colwise=True, block_2d=None):
    """Run te_mx_quantize (or, with ``block_2d`` given, te_mx_block_quantize)
    with canary-guarded outputs; returns numpy arrays and asserts no byte
    outside the documented output region changed."""
    rows, cols = x.shape
    out, bufs = {}, {}
    pr, pc = binding.te_mx_scale_pitch(cols), binding.te_mx_scale_pitch(rows)
    if rowwise:
        out["q_row"], bufs["q_row"] = guarded_u8(rows, cols)
        out["s_row"], bufs["s_row"] = guarded_u8(rows, pr)
    if colwise:
        out["q_col"], bufs["q_col"] = guarded_u8(cols, rows)
        out["s_col"], bufs["s_col"] = guarded_u8(cols, pc)
    if block_2d is None:
        binding.quantize(x, rowwise=rowwise, colwise=colwise, out=out)
    else:
        binding.block_quantize(x, block_2d=block_2d, rowwise=rowwise, colwise=colwise, out=out)
    binding.te_mx_device_status()
    res = {}
    if rowwise:
        check_guard(bufs["q_row"], rows * cols)
        check_guard(bufs["s_row"], rows * pr)
        s = out["s_row"].cpu().numpy()
        assert np.all(s[:, cols // 32:] == CANARY), "scale padding bytes were written"
        res["q_row"], res["s_row"] = out["q_row"].cpu().numpy(), s[:, : cols // 32]
    if colwise:
        check_guard(bufs["q_col"], rows * cols)
        check_guard(bufs["s_col"], cols * pc)
        s = out["s_col"].cpu().numpy()
        assert np.all(s[:, rows // 32:] == CANARY), "scale padding bytes were written"
        res["q_col"], res["s_col"] = out["q_col"].cpu().numpy(), s[:, : rows // 32]
    return res


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatching bytes; first at {i}: "
                             f"got 0x{int(got[i]):02X}, want 0x{int(want[i]):02X}")
