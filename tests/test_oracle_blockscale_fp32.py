"""Pins for the Float8BlockScaling mode that keeps FP32 scales (ROCm/TransformerEngine
README, "Blockwise FP8 GEMM support on ROCm": the GEMM computed "with the FP32 scales
directly").

* the scale pair (s = fl32(amax / 448), r = fl32(1 / s)) against exact rational
  arithmetic with brute-force rounding to fp32, over every positive bf16 amax;
* the codes against exact products rounded to fp32 by brute force;
* round-trip accuracy of deq = code * s, special blocks (zero, NaN, inf), 2D
  blocks shared by both copies, colwise(X) == rowwise(X^T), ragged edges;
* the GEMM against exact rational sums and K-block linearity.
"""
from fractions import Fraction

import numpy as np
import torch

from oracle import mx_oracle as O

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
F32_MAX = Fraction(float(np.finfo(np.float32).max))


def rand_bits(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def round_f32(f: Fraction) -> float:
    """Round a positive rational to the nearest fp32 (ties to even mantissa),
    by comparing the neighbours of a first guess exactly; inf past the
    rounding boundary above the largest finite value."""
    half_ulp_max = Fraction(2) ** (127 - 24)
    if f >= F32_MAX + half_ulp_max:
        return float("inf")
    guess = np.float32(float(f))
    cands = {np.nextafter(guess, np.float32(-np.inf)), guess, np.nextafter(guess, np.float32(np.inf))}
    cands = [c for c in cands if np.isfinite(c) and c >= 0]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - f),
                                     int(np.array(c, dtype=np.float32).view(np.uint32)) & 1))
    return float(best)


def test_scale_pair_exhaustive():
    v = O.bf16_bits_to_f64(ALL_BF16)
    amax = v[np.isfinite(v) & (v > 0)]
    s, r = O.block_scale_fp32(amax)
    for a, si, ri in zip(amax, s, r):
        se = round_f32(Fraction(float(a)) / 448)
        assert float(si) == se, (a, si, se)
        re = round_f32(1 / Fraction(se)) if se > 0 else float("inf")
        re = min(re, float(F32_MAX))
        assert float(ri) == re, (a, ri, re)
    s0, r0 = O.block_scale_fp32(np.array([0.0, np.nan, np.inf]))
    assert s0[0] == 1 and r0[0] == 1 and np.isnan(s0[1:]).all() and np.isnan(r0[1:]).all()


def test_codes_are_rounded_fp32_products():
    x = rand_bits((128, 256), 7, std=3.0)
    q_row, s_row, _, _ = O.quantize_block_fp32(x, False)
    xv = O.bf16_bits_to_f64(x)
    rng = np.random.default_rng(1)
    for i, j in zip(rng.integers(0, 128, 300), rng.integers(0, 256, 300)):
        a = np.abs(xv[i, 128 * (j // 128):128 * (j // 128) + 128]).max()
        _, r = O.block_scale_fp32(np.array([a]))
        exact = Fraction(float(xv[i, j])) * Fraction(float(r[0]))
        p = round_f32(abs(exact)) * (1 if exact >= 0 else -1)
        assert q_row[i, j] == O.e4m3_encode(np.array([p]))[0], (i, j)


def test_round_trip_accuracy():
    x = rand_bits((256, 384), 3, std=4.0)
    xv = O.bf16_bits_to_f64(x)
    for two_d in (False, True):
        q_row, s_row, q_col, s_col = O.quantize_block_fp32(x, two_d)
        for q, s, ref in ((q_row, s_row, xv), (q_col, s_col, xv.T)):
            d = O.dequantize_fp32(q, s)
            # each block's true scale amax / 448, from the input alone
            ar = np.abs(ref)
            if two_d:
                blk = ar.reshape(ar.shape[0] // 128, 128, ar.shape[1] // 128, 128).max(axis=(1, 3))
                amax = np.repeat(np.repeat(blk, 128, axis=0), 128, axis=1)
            else:
                amax = np.repeat(ar.reshape(ar.shape[0], -1, 128).max(axis=2), 128, axis=1)
            sc = amax / 448.0
            # normal E4M3 range: half an ulp (2^-4 relative) plus the s * r != 1 slack;
            # below 2^-6 * s: half the subnormal step 2^-9 * s
            bound = np.maximum(ar * (2.0 ** -4 + 2.0 ** -20), sc * 2.0 ** -10 * (1 + 2.0 ** -20))
            assert np.all(np.abs(d - ref) <= bound)
            assert np.abs(O.e4m3_decode(q)).max() <= 448.0


def test_special_blocks():
    x = np.full((128, 256), 0.5)
    x[:, 128:] = 0.0
    x[3, 5] = np.nan
    x[7, 200] = np.inf
    bits = O.f64_to_bf16_bits(x)
    q_row, s_row, q_col, s_col = O.quantize_block_fp32(bits, False)
    assert np.isnan(s_row[3, 0]) and np.all(q_row[3, :128] == 0x7F)
    assert np.isnan(s_row[7, 1]) and np.all(q_row[7, 128:] == 0x7F)
    assert s_row[0, 1] == 1.0 and not q_row[0, 128:].any()              # zero block
    # amax 0.5: s = 0.5 / 448 (fp32), r = fl32(1 / s) ~ 896; 0.5 * r rounds to 448
    assert s_row[0, 0] == np.float32(0.5) / np.float32(448) and np.all(q_row[0, :128] == 0x7E)
    assert np.isnan(s_col[5, 0]) and np.all(q_col[5] == 0x7F)


def test_2d_blocks_and_transposition():
    x = rand_bits((256, 384), 5, std=2.0)
    q_row, s_row, q_col, s_col = O.quantize_block_fp32(x, True)
    assert np.array_equal(q_row.T, q_col)
    for bi in range(2):
        assert np.all(s_row[128 * bi:128 * bi + 128] == s_row[128 * bi])
    assert np.array_equal(s_row[::128], s_col[::128].T)
    xt = np.ascontiguousarray(x.T)
    qr1, sr1, qc1, sc1 = O.quantize_block_fp32(x, False)
    qr2, sr2, qc2, sc2 = O.quantize_block_fp32(xt, False)
    assert np.array_equal(qc1, qr2) and np.array_equal(sc1, sr2)


def test_ragged_edges_per_element():
    x = rand_bits((130, 200), 9, std=1.5)
    xv = O.bf16_bits_to_f64(x)
    q_row, s_row, q_col, s_col = O.quantize_block_fp32(x, False)
    for i in (0, 64, 129):
        for b in range(2):
            seg = xv[i, 128 * b:128 * b + 128]
            s, r = O.block_scale_fp32(np.array([np.abs(seg).max()]))
            assert s_row[i, b] == s[0]
            prod = (seg.astype(np.float32) * r[0]).astype(np.float64)
            assert np.array_equal(q_row[i, 128 * b:128 * b + len(seg)], O.e4m3_encode(prod).astype(np.uint8))
    seg = xv[128:, 7]                                         # partial column block: 2 rows
    s, _ = O.block_scale_fp32(np.array([np.abs(seg).max()]))
    assert s_col[7, 1] == s[0]


def test_gemm_exact_small():
    rng = np.random.default_rng(2)
    qa = rng.integers(0, 0x7F, (16, 256)).astype(np.uint8)
    qb = rng.integers(0, 0x7F, (16, 256)).astype(np.uint8)
    qa[qa == 0x7F] = 0x7E
    qb[qb == 0x7F] = 0x7E
    sa = rng.uniform(1e-3, 1.0, (16, 2)).astype(np.float32)
    sb = rng.uniform(1e-3, 1.0, (16, 2)).astype(np.float32)
    r = O.block_gemm_fp32(qa, sa, qb, sb)
    va, vb = O.e4m3_decode(qa), O.e4m3_decode(qb)
    for m, n in ((0, 0), (3, 11), (15, 15)):
        exact = sum(Fraction(float(va[m, k])) * Fraction(float(sa[m, k // 128])) *
                    Fraction(float(vb[n, k])) * Fraction(float(sb[n, k // 128])) for k in range(256))
        assert abs(Fraction(float(r["pre"][m, n])) - exact) <= Fraction(float(r["sigma"][m, n])) * Fraction(1, 1 << 40)


def test_gemm_k_block_linearity():
    x = rand_bits((64, 256), 11)
    w = rand_bits((32, 256), 12)
    qa, sa, _, _ = O.quantize_block_fp32(x, False)
    qb, sb, _, _ = O.quantize_block_fp32(w, True)
    base = O.block_gemm_fp32(qa, sa, qb, sb)["pre"]
    sa2 = sa.copy()
    sa2[:, 1] *= 2                                             # exact: a power of two
    doubled = O.block_gemm_fp32(qa, sa2, qb, sb)["pre"]
    qa1 = qa.copy()
    qa1[:, :128] = 0
    second = O.block_gemm_fp32(qa1, sa, qb, sb)["pre"]         # the second K block alone
    assert np.allclose(doubled - base, second, rtol=0, atol=1e-12 * np.abs(base).max())
