"""GPU parity of te_mx_layernorm_quantize against the oracle.

The kernel evaluates the LayerNorm in fp32 (its header states how), the oracle
in fp64.  Statistics: |mu_gpu - mu| <= dmu and |rsigma_gpu - rsigma| <= rho
rsigma (``layernorm_stat_bounds``).  Codes and scales: every one must be the
MXFP8 quantisation of some y' within ``layernorm_error_bound`` of the exact y
(``mx_admissible``); where only one answer is admissible (all but a small
fraction of the elements, asserted) that is bit-exactness.  Covers chunk and
unit edge cases (hidden not a multiple of 64, long rows, the largest hidden),
several rows per statistics warp group (with and without codes), ragged rows,
each orientation alone, statistics only,
constant and non-finite rows, large row means, determinism, canary-guarded
outputs, and the full-size ffn input (sampled rows and 32-row bands).
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu

MAX_AMBIGUOUS = 5e-3


def make(rows, hidden, seed, mean=0.0, std=1.0, row_spread=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, hidden, generator=g) * std + mean
    if row_spread:                                    # rows of different scale and offset
        x = x * torch.exp2(torch.randint(-3, 4, (rows, 1), generator=g).float()) \
            + torch.randn(rows, 1, generator=g)
    ga = 1.0 + 0.1 * torch.randn(hidden, generator=g)
    be = 0.1 * torch.randn(hidden, generator=g)
    return x.to(torch.bfloat16), ga.to(torch.bfloat16), be.to(torch.bfloat16)


def run(x, ga, be, rowwise=True, colwise=True):
    rows, hidden = x.shape
    out, bufs = {}, {}
    pr, pc = binding.te_mx_scale_pitch(hidden), binding.te_mx_scale_pitch(rows)
    if rowwise:
        out["q_row"], bufs["q_row"] = U.guarded_u8(rows, hidden)
        out["s_row"], bufs["s_row"] = U.guarded_u8(rows, pr)
    if colwise:
        out["q_col"], bufs["q_col"] = U.guarded_u8(hidden, rows)
        out["s_col"], bufs["s_col"] = U.guarded_u8(hidden, pc)
    for key in ("mu", "rsigma"):
        buf = torch.full((rows + 64,), float("nan"), dtype=torch.float32, device="cuda")
        out[key], bufs[key] = buf[:rows], buf
    binding.layernorm_quantize(x.cuda(), ga.cuda(), be.cuda(), rowwise=rowwise, colwise=colwise, out=out)
    binding.te_mx_device_status()
    res = {}
    if rowwise:
        U.check_guard(bufs["q_row"], rows * hidden)
        U.check_guard(bufs["s_row"], rows * pr)
        s = out["s_row"].cpu().numpy()
        assert np.all(s[:, hidden // 32:] == U.CANARY)
        res["q_row"], res["s_row"] = out["q_row"].cpu().numpy(), s
    if colwise:
        U.check_guard(bufs["q_col"], rows * hidden)
        U.check_guard(bufs["s_col"], hidden * pc)
        s = out["s_col"].cpu().numpy()
        assert np.all(s[:, rows // 32:] == U.CANARY)
        res["q_col"], res["s_col"] = out["q_col"].cpu().numpy(), s
    for key in ("mu", "rsigma"):
        assert torch.isnan(bufs[key][rows:]).all(), "write past the end of " + key
        res[key] = out[key].double().cpu().numpy()
    return res


def check(x, ga, be, got, rows_idx=None, max_ambiguous=MAX_AMBIGUOUS):
    """Compare against the oracle for the rows ``rows_idx`` (default all).
    ``max_ambiguous`` caps the fraction of elements whose answer the error
    bound leaves open (None: no cap, for inputs where the bound is wide)."""
    xb, gb, bb = U.bf16_bits(x), U.bf16_bits(ga), U.bf16_bits(be)
    if rows_idx is not None:
        xb = xb[rows_idx]
    y, mu, rs = O.layernorm(xb, gb, bb)
    err = O.layernorm_error_bound(xb, gb)
    finite = np.isfinite(mu)
    if "mu" in got:
        dmu, rho = O.layernorm_stat_bounds(xb)
        gm, gr = got["mu"], got["rsigma"]
        if rows_idx is not None:
            gm, gr = gm[rows_idx], gr[rows_idx]
        assert np.all(np.abs(gm - mu)[finite] <= dmu[finite]), "mu outside its bound"
        assert np.all(np.abs(gr - rs)[finite] <= (rho * rs)[finite]), "rsigma outside its bound"
        assert not np.isfinite(gm[~finite]).any()
    n_amb = n = 0
    if "q_row" in got:
        q, s = got["q_row"], got["s_row"]
        if rows_idx is not None:
            q, s = q[rows_idx], s[rows_idx]
        ok, amb = O.mx_admissible(y, err, q, s, 1)
        if not ok.all():
            i = tuple(np.argwhere(~ok)[0])
            raise AssertionError(f"row-wise: {int((~ok).sum())} inadmissible; first {i}: code 0x{q[i]:02X} "
                                 f"scale {s[i[0], i[1] // 32]} y {y[i]!r} err {err[i]!r}")
        n_amb += int(amb.sum()); n += amb.size
    if "q_col" in got and rows_idx is None:
        ok, amb = O.mx_admissible(y, err, got["q_col"], got["s_col"], 0)
        if not ok.all():
            i = tuple(np.argwhere(~ok)[0])
            raise AssertionError(f"column-wise: {int((~ok).sum())} inadmissible; first {i}")
        n_amb += int(amb.sum()); n += amb.size
    if n and max_ambiguous is not None:
        assert n_amb <= max_ambiguous * n + 4, f"{n_amb} of {n} elements ambiguous"


@pytest.mark.parametrize("rows,hidden", [(32, 64), (64, 96), (256, 1024), (96, 4128), (128, 7168),
                                         (64, 2080), (32, 24576), (32, 24640),
                                         (32, 32768)])
def test_both_orientations(rows, hidden):
    x, ga, be = make(rows, hidden, rows * 3 + hidden)
    check(x, ga, be, run(x, ga, be))


@pytest.mark.parametrize("rows,hidden", [(10016, 512), (1312, 2048), (1248, 2016)])
def test_several_rows_per_statistics_warp(rows, hidden):
    # more rows than the statistics kernel's warp groups (one warp per row
    # under 2048 elements, four from 2048): each group reuses its two row
    # buffers; every row's statistics and a sample of code rows are checked
    x, ga, be = make(rows, hidden, rows + 2 * hidden)
    check(x, ga, be, run(x, ga, be, rowwise=False, colwise=False))
    got = run(x, ga, be)
    sample = np.sort(np.random.default_rng(rows).choice(rows, 48, replace=False))
    check(x, ga, be, {"mu": got["mu"], "rsigma": got["rsigma"]})
    check(x, ga, be, {k: v for k, v in got.items() if k in ("q_row", "s_row")}, sample)


@pytest.mark.parametrize("rows,hidden", [(1, 64), (37, 512), (100, 1056), (45, 24608)])
def test_rowwise_ragged_rows(rows, hidden):
    x, ga, be = make(rows, hidden, rows + hidden)
    check(x, ga, be, run(x, ga, be, rowwise=True, colwise=False))


def test_one_orientation_and_stats_only():
    x, ga, be = make(160, 1536, 5)
    check(x, ga, be, run(x, ga, be, rowwise=False, colwise=True))
    check(x, ga, be, run(x, ga, be, rowwise=False, colwise=False))


def test_large_row_means_and_tiny_variance():
    # |mean| >> std: the fp32 mean error bound grows with mean|x| (here ~8e-4
    # on y ~ 1), so many answers are open; every code must still be admissible
    x, ga, be = make(64, 2048, 6, mean=200.0, std=1.0, row_spread=False)
    check(x, ga, be, run(x, ga, be), max_ambiguous=None)
    x, ga, be = make(64, 1024, 7, mean=0.0, std=1e-4, row_spread=False)      # var << eps
    check(x, ga, be, run(x, ga, be))


def test_constant_and_non_finite_rows():
    x, ga, be = make(64, 512, 8)
    x[3, :] = 2.5                                  # constant row: y = beta exactly
    x[9, 100] = float("nan")
    x[40, 7] = float("inf")
    got = run(x, ga, be)
    # rsigma = 1/sqrt(eps) on the constant row makes its bound wide: no cap on
    # ambiguity, but its mean is exact (a sum of equal values), so y = beta
    # exactly and its codes must be the quantisation of beta itself
    check(x, ga, be, got, max_ambiguous=None)
    qb, sb = O.quantize_mx_values(O.bf16_bits_to_f64(U.bf16_bits(be))[None, :], 1)
    assert np.array_equal(got["q_row"][3], qb[0]) and np.array_equal(got["s_row"][3, :16], sb[0])
    s_row = got["s_row"]
    assert np.all(s_row[9, :16] == 0xFF) and np.all(s_row[40, :16] == 0xFF)
    assert np.all(got["s_col"][:, 0] == 0xFF) and np.all(got["s_col"][:, 1] == 0xFF)   # rows 9 and 40


def test_deterministic():
    x, ga, be = make(128, 3072, 9)
    a, b = run(x, ga, be), run(x, ga, be)
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_full_size_ffn_input_sampled():
    d = workloads.make_ffn()
    x = d["X"]
    ga, be = workloads.layernorm_params(x.shape[1], 410)
    got = run(x, ga, be)
    rows = x.shape[0]
    rng = np.random.default_rng(11)
    sample = np.sort(rng.choice(rows, 64, replace=False))
    sample[-1] = rows - 1
    check(x, ga, be, {k: v for k, v in got.items() if k in ("q_row", "s_row", "mu", "rsigma")}, sample)
    for band in (0, int(rng.integers(1, rows // 32 - 1)), rows // 32 - 1):   # 32-row bands, column-wise
        r = slice(32 * band, 32 * band + 32)
        xb = x[r]
        y, _, _ = O.layernorm(U.bf16_bits(xb), U.bf16_bits(ga), U.bf16_bits(be))
        err = O.layernorm_error_bound(U.bf16_bits(xb), U.bf16_bits(ga))
        ok, amb = O.mx_admissible(y, err, got["q_col"][:, r], got["s_col"][:, band:band + 1], 0)
        assert ok.all() and amb.mean() <= MAX_AMBIGUOUS
