"""Pins for the Float8BlockScaling (E8M0-cast) part of the oracle.

* the scale rule against brute force (smallest power of two >= amax/448) over
  every positive bf16 value;
* hand-worked blocks;
* invariants: no element saturates, 2D blocks give transposed-identical codes,
  the largest element of each block lands in [224, 448] after rounding, a power-of-two shift
  of a block only shifts its scale;
* the MX GEMM of block-scaled operands equals the fp64 product of the
  dequantised operands built from the block definition directly.
"""
import numpy as np
import pytest
import torch

from oracle import mx_oracle as O

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def rand_bits(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_block_scale_rule_exhaustive():
    v = O.bf16_bits_to_f64(ALL_BF16)
    amax = v[np.isfinite(v) & (v > 0)]
    es = np.arange(-127, 128)
    ok = amax[:, None] <= 448.0 * np.ldexp(1.0, es)[None, :]
    brute = np.where(ok.any(axis=1), es[np.argmax(ok, axis=1)], 127)
    assert np.array_equal(O.block_scale_exponent(amax), brute)
    assert O.block_scale_exponent(0.0) == -127


def test_hand_worked_1d_block():
    # one 128-row block: amax = 3 -> 3/448 = 0.0067 -> 2^-7 = 0.0078 >= it, 2^-8 is not -> e = -7
    x = np.full((128, 128), 0.25)
    x[5, :] = 1.0
    x[5, 17] = 3.0
    x[6, :] = 0.0
    bits = O.f64_to_bf16_bits(x)
    q_row, s_row, q_col, s_col = O.quantize_block(bits, False)
    assert s_row[5, 0] == 127 - 7 and np.all(s_row[5] == 120)      # repeated over the 4 groups
    assert q_row[5, 17] == 0x7C                                     # 3 * 2^7 = 384 = 0.1111.100
    assert q_row[5, 0] == 0x70                                      # 1 * 2^7 = 128
    # a row of 0.25: 0.25/448 -> e = -10 (2^-10 = 0.00098 >= 0.000558; 2^-11 is not), 0.25 * 2^10 = 256
    assert s_row[0, 0] == 127 - 10 and q_row[0, 0] == 0x78
    assert np.all(s_row[6] == 0) and not q_row[6].any()              # zero row
    # column 17 holds 3.0: same scale; other columns amax 1.0 -> e = -8 (2^-8 = 0.0039 >= 0.00223)
    assert np.all(s_col[17] == 120) and np.all(s_col[0] == 127 - 8)


def test_no_saturation_and_top_binade():
    x = rand_bits((256, 384), 3, std=5.0)
    for two_d in (False, True):
        q_row, s_row, q_col, s_col = O.quantize_block(x, two_d)
        for q, s in ((q_row, s_row), (q_col, s_col)):
            v = np.abs(O.e4m3_decode(q))
            assert v.max() <= 448.0
            # every block's largest element scales into (224, 448]; E4M3 spacing
            # is 16 below 256, so after rounding it lies in [224, 448]
            blocks = v.reshape(v.shape[0], -1, 128).max(axis=2)
            if not two_d:
                assert np.all((blocks >= 224.0) & (blocks <= 448.0))


def test_2d_blocks_share_scale_across_copies():
    x = rand_bits((256, 256), 4)
    q_row, s_row, q_col, s_col = O.quantize_block(x, True)
    assert np.array_equal(q_col, q_row.T)
    assert np.array_equal(np.repeat(s_col, 32, axis=1), np.repeat(s_row, 32, axis=1).T)


@pytest.mark.parametrize("k", [-6, 9])
def test_power_of_two_shift_only_moves_the_scale(k):
    x = rand_bits((128, 256), 5)
    y = O.f64_to_bf16_bits(O.bf16_bits_to_f64(x) * 2.0 ** k)
    for two_d in (False, True):
        a, b = O.quantize_block(x, two_d), O.quantize_block(y, two_d)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
        assert np.array_equal(b[1].astype(int), a[1].astype(int) + k)


def test_block_scaled_gemm_equals_direct_definition():
    xa, xb = rand_bits((128, 256), 6), rand_bits((128, 256), 7, std=0.1)
    qa, sa, _, _ = O.quantize_block(xa, False)          # 1x128 activations
    qb, sb, _, _ = O.quantize_block(xb, True)           # 128x128 weights
    got = O.mx_gemm(qa, sa, qb, sb)["pre"]
    # direct: per-128 scales from the block definition, no MX layout involved
    av = O.bf16_bits_to_f64(xa); bv = O.bf16_bits_to_f64(xb)
    ea = O.block_scale_exponent(np.abs(av).reshape(128, 2, 128).max(axis=2))       # [128, 2]
    eb = O.block_scale_exponent(np.abs(bv).reshape(1, 128, 2, 128).max(axis=(1, 3)))  # [1, 2]
    da = O.e4m3_decode(O.e4m3_encode(av * np.repeat(2.0 ** -ea, 128, axis=1))) * np.repeat(2.0 ** ea, 128, axis=1)
    db = O.e4m3_decode(O.e4m3_encode(bv * np.repeat(2.0 ** -eb, 128, axis=1))) * np.repeat(2.0 ** eb, 128, axis=1)
    assert np.array_equal(got, da @ db.T)


@pytest.mark.parametrize("two_d", [False, True])
def test_partial_edge_blocks_by_loops(two_d):
    """Ragged 96 x 160 input: per-block loops over the elements present."""
    rows, cols = 96, 160
    x = rand_bits((rows, cols), 8, std=3.0)
    v = O.bf16_bits_to_f64(x)
    q_row, s_row, q_col, s_col = O.quantize_block(x, two_d)
    assert s_row.shape == (rows, cols // 32) and s_col.shape == (cols, rows // 32)
    for r in range(rows):
        for c in range(cols):
            if two_d:
                rb, cb = r // 128 * 128, c // 128 * 128
                a_r = a_c = max(abs(v[i, j]) for i in range(rb, min(rb + 128, rows))
                                for j in range(cb, min(cb + 128, cols)))
            else:
                cb, rb = c // 128 * 128, r // 128 * 128
                a_r = max(abs(v[r, j]) for j in range(cb, min(cb + 128, cols)))
                a_c = max(abs(v[i, c]) for i in range(rb, min(rb + 128, rows)))
            e_r = next(e for e in range(-127, 128) if a_r <= 448.0 * 2.0 ** e)
            e_c = next(e for e in range(-127, 128) if a_c <= 448.0 * 2.0 ** e)
            assert s_row[r, c // 32] == e_r + 127
            assert s_col[c, r // 32] == e_c + 127
            assert q_row[r, c] == O.e4m3_encode(v[r, c] * 2.0 ** -e_r)
            assert q_col[c, r] == O.e4m3_encode(v[r, c] * 2.0 ** -e_c)
        if two_d:
            break                                     # every row of a 2D block is alike: one row suffices


def test_non_finite_block():
    x = O.f64_to_bf16_bits(np.ones((128, 256)))
    x[3, 200] = 0x7FC0                                # NaN in row 3, second 128-block
    x[70, 10] = 0x7F80                                # +inf in row 70, first block
    q_row, s_row, q_col, s_col = O.quantize_block(x, False)
    assert np.all(s_row[3, 4:] == 0xFF) and np.all(q_row[3, 128:] == 0x7F)
    assert np.all(s_row[3, :4] == 127 - 8) and np.all(q_row[3, :128] == 0x78)    # 1 * 2^8 = 256
    assert np.all(s_row[70, :4] == 0xFF) and np.all(q_row[70, :128] == 0x7F)
    assert np.all(s_col[200] == 0xFF) and np.all(q_col[200] == 0x7F) and np.all(s_col[201] == 119)
    q_row, s_row, q_col, s_col = O.quantize_block(x, True)
    assert np.all(s_row == 0xFF) and np.all(q_col == 0x7F)
