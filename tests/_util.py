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


_POOL = None


def oracle_pool():
    """Process pool (spawn start method, safe after CUDA is initialised) for
    oracle work that is independent per item; its workers import only the
    oracle and numpy."""
    global _POOL
    if _POOL is None:
        import multiprocessing
        import os
        from concurrent.futures import ProcessPoolExecutor
        _POOL = ProcessPoolExecutor(max_workers=max(1, min(16, (os.cpu_count() or 2) - 1)),
                                    mp_context=multiprocessing.get_context("spawn"))
    return _POOL


def band_rows(n, band, seed, extra=()):
    """One random row in every ``band``-row band of [0, n), plus the first and
    last row and ``extra`` (sorted, unique): every output tile row band is
    visited."""
    rng = np.random.default_rng(seed)
    rows = {0, n - 1, *[int(r) for r in extra if 0 <= r < n]}
    for b0 in range(0, n, band):
        rows.add(int(rng.integers(b0, min(n, b0 + band))))
    return np.array(sorted(rows), dtype=np.int64)


def check_rows_rowwise(q_dev, s_dev, x_cpu, rows, what, only_rows=False):
    """Row-wise codes and scales of the given rows, read back from the device,
    against the oracle quantisation of the same input rows (bit-exact);
    ``only_rows``: ``x_cpu`` holds just those rows, in that order."""
    from oracle import mx_oracle as O
    ri = torch.from_numpy(rows)
    q, s = O.quantize_rowwise(bf16_bits(x_cpu if only_rows else x_cpu[ri]))
    rd = ri.to(q_dev.device)
    cols = x_cpu.shape[1]
    assert_bytes_equal(q_dev[rd].cpu().numpy(), q, what + " codes")
    assert_bytes_equal(s_dev[rd][:, : cols // 32].cpu().numpy(), s, what + " scales")
    return q, s


def check_cols_colwise(q_dev, s_dev, x_cpu, cols_idx, what, dev_index=None):
    """Column-wise codes and scales (rows of the transposed copy) of the given
    input columns against the oracle (bit-exact); ``dev_index`` are the
    columns' indices in the device copy when ``x_cpu`` holds only them."""
    from oracle import mx_oracle as O
    ci = torch.from_numpy(cols_idx)
    q, s = O.quantize_colwise(bf16_bits(x_cpu[:, ci]))
    cd = torch.from_numpy(cols_idx if dev_index is None else dev_index).to(q_dev.device)
    rows = x_cpu.shape[0]
    assert_bytes_equal(q_dev[cd].cpu().numpy(), q, what + " codes")
    assert_bytes_equal(s_dev[cd][:, : rows // 32].cpu().numpy(), s, what + " scales")
    return q, s


def oracle_quantize_parallel(bits, colwise=False, slab=1024):
    """Oracle MXFP8 quantisation of a large bf16 matrix (uint16 patterns),
    computed slab by slab in the spawn pool: row slabs for the row-wise copy,
    column slabs for the column-wise copy (blocks never cross a slab)."""
    from tests import _oracle_jobs as J
    pool = oracle_pool()
    n = bits.shape[1] if colwise else bits.shape[0]
    parts = []
    for a in range(0, n, slab):
        chunk = np.ascontiguousarray(bits[:, a:a + slab] if colwise else bits[a:a + slab])
        parts.append(pool.submit(J.quantize_cols if colwise else J.quantize_rows, chunk))
    res = [p.result() for p in parts]
    return np.concatenate([q for q, _ in res]), np.concatenate([s for _, s in res])


def check_every_byte(out, x_cpu, rowwise, colwise, what):
    """Every code and scale of the device copies in ``out`` against the
    oracle (bit-exact); returns the oracle's {(q_row, s_row), (q_col, s_col)}."""
    bits = bf16_bits(x_cpu)
    rows, cols = x_cpu.shape
    ref = {}
    if rowwise:
        q, s = oracle_quantize_parallel(bits, colwise=False)
        assert_bytes_equal(out["q_row"].cpu().numpy(), q, what + " row-wise codes")
        assert_bytes_equal(out["s_row"][:, : cols // 32].cpu().numpy(), s, what + " row-wise scales")
        ref["row"] = (q, s)
    if colwise:
        q, s = oracle_quantize_parallel(bits, colwise=True)
        assert_bytes_equal(out["q_col"].cpu().numpy(), q, what + " column-wise codes")
        assert_bytes_equal(out["s_col"][:, : rows // 32].cpu().numpy(), s, what + " column-wise scales")
        ref["col"] = (q, s)
    return ref


_MOE = None


def moe_workload():
    """The MoE workload (2.7 GB of bf16 on the host), drawn once per session."""
    global _MOE
    if _MOE is None:
        from mxfp8_block_scaled_quantize_gb300 import workloads
        _MOE = workloads.make_moe()
    return _MOE
