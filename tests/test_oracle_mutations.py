"""Planted mistakes: break the oracle in a plausible way and check that a pin fails.

Each test patches one piece of the oracle (on the CPU, for the duration of
the test) and runs an existing pin, which must now raise AssertionError.
"""
import numpy as np
import pytest

from oracle import mx_oracle as O
from tests import test_oracle_gemm as G
from tests import test_oracle_quantize as Q


def run_all_golden():
    for blk in Q.parse_golden():
        Q.test_golden_block_rowwise(blk)
        Q.test_golden_block_colwise(blk)


def test_golden_pins_pass_unpatched():
    run_all_golden()


def test_wrong_emax_is_caught(monkeypatch):
    monkeypatch.setattr(O, "E4M3_EMAX", 7)
    with pytest.raises(AssertionError):
        run_all_golden()
    with pytest.raises(AssertionError):
        Q.test_scale_rule_exhaustive_against_brute_force()


def test_ties_away_from_zero_is_caught(monkeypatch):
    def round_half_away(v, mant_bits, emin):
        v = np.asarray(v, dtype=np.float64)
        _, p = np.frexp(v)
        quantum = np.ldexp(1.0, np.maximum(p - 1, emin) - mant_bits)
        return np.sign(v) * np.floor(np.abs(v) / quantum + 0.5) * quantum
    monkeypatch.setattr(O, "round_to_binary_format", round_half_away)
    with pytest.raises(AssertionError):
        Q.test_e4m3_encode_equals_brute_force_nearest()
    with pytest.raises(AssertionError):
        run_all_golden()


def test_lost_sign_of_zero_is_caught(monkeypatch):
    orig = O.e4m3_encode_value
    monkeypatch.setattr(O, "e4m3_encode_value", lambda r: orig(np.where(np.asarray(r) == 0, 0.0, r)))
    with pytest.raises(AssertionError):
        run_all_golden()
    with pytest.raises(AssertionError):
        Q.test_e4m3_encode_matches_library_saturating_cast()


def test_scale_with_wrong_sign_is_caught(monkeypatch):
    orig = O.mx_scale_exponent
    monkeypatch.setattr(O, "mx_scale_exponent", lambda a: -orig(a))
    with pytest.raises(AssertionError):
        run_all_golden()


def test_no_saturation_is_caught(monkeypatch):
    monkeypatch.setattr(O, "E4M3_MAX", 1e9)
    with pytest.raises(AssertionError):
        run_all_golden()


def test_wrong_scale_block_index_is_caught(monkeypatch):
    def bad_dequantize(q, s):
        q = np.asarray(q, dtype=np.uint8)
        s = np.asarray(s, dtype=np.uint8).astype(np.int64)
        scale = np.tile(np.ldexp(1.0, s - 127), (1, 32))        # k % nblocks instead of k // 32
        return O.e4m3_decode(q) * scale
    monkeypatch.setattr(O, "dequantize", bad_dequantize)
    with pytest.raises(AssertionError):
        G.test_tiny_gemm_exact_rational(8, 24, 64)


def test_dropped_bias_is_caught(monkeypatch):
    orig = O.mx_gemm
    monkeypatch.setattr(O, "mx_gemm", lambda qa, sa, qb, sb, bias=None, gelu=False: orig(qa, sa, qb, sb, None, gelu))
    with pytest.raises(AssertionError):
        G.test_tiny_gemm_exact_rational(16, 16, 32)


def test_transposed_b_is_caught(monkeypatch):
    orig_deq = O.dequantize
    calls = {"n": 0}

    def deq_second_transposed(q, s):
        calls["n"] += 1
        d = orig_deq(q, s)
        return d[::-1] if calls["n"] % 2 == 0 else d        # B's rows in the wrong order
    monkeypatch.setattr(O, "dequantize", deq_second_transposed)
    with pytest.raises(AssertionError):
        G.test_transposed_operands_are_distinguished()


def test_wrong_gelu_constant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "gelu_tanh",
                        lambda x: 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.0447 * x ** 3))))
    with pytest.raises(AssertionError):
        G.test_gelu_matches_library_and_identities()


def test_fp32_scale_mutations_are_caught(monkeypatch):
    from tests import test_oracle_blockscale_fp32 as F
    orig = O.block_scale_fp32
    # the quantisation scale used as the stored scale (448 / amax instead of amax / 448)
    monkeypatch.setattr(O, "block_scale_fp32", lambda a: tuple(reversed(orig(a))))
    with pytest.raises(AssertionError):
        F.test_scale_pair_exhaustive()
    with pytest.raises(AssertionError):
        F.test_round_trip_accuracy()
    monkeypatch.setattr(O, "block_scale_fp32", orig)
    # the K blocks' scales misaligned by one block
    orig_deq = O.dequantize_fp32
    monkeypatch.setattr(O, "dequantize_fp32", lambda q, s: orig_deq(q, np.roll(np.asarray(s), 1, axis=1)))
    with pytest.raises(AssertionError):
        F.test_gemm_exact_small()


def test_block_scale_mutations_are_caught(monkeypatch):
    from tests import test_oracle_blockscale as B
    # floor instead of ceil: the largest element of a block can then exceed 448 after scaling
    orig = O.block_scale_exponent
    monkeypatch.setattr(O, "block_scale_exponent",
                        lambda amax: np.where(np.asarray(amax) > 0, O.floor_log2(np.asarray(amax, np.float64)) - 8,
                                              -127).astype(np.int64))
    with pytest.raises(AssertionError):
        B.test_block_scale_rule_exhaustive()
    monkeypatch.setattr(O, "block_scale_exponent", orig)
    # 2D blocks requested, 1x128 / 128x1 blocks computed
    orig_qb = O.quantize_block
    monkeypatch.setattr(O, "quantize_block", lambda x, block_2d: orig_qb(x, False))
    with pytest.raises(AssertionError):
        B.test_2d_blocks_share_scale_across_copies()


def test_backward_mutations_are_caught(monkeypatch):
    from tests import test_oracle_backward as D
    # dGELU without the term from the derivative of u (only 0.5 (1 + tanh u))
    monkeypatch.setattr(O, "dgelu_tanh",
                        lambda x: 0.5 * (1 + np.tanh(np.sqrt(2 / np.pi) * (np.asarray(x, np.float64)
                                                                           + 0.044715 * np.asarray(x, np.float64) ** 3))))
    with pytest.raises(AssertionError):
        D.test_dgelu_matches_autograd()
    with pytest.raises(AssertionError):
        D.test_dgelu_matches_finite_differences()
    # bias gradient missing the last row
    monkeypatch.setattr(O, "column_sums",
                        lambda xb: (O.bf16_bits_to_f64(xb)[:-1].sum(axis=0), np.abs(O.bf16_bits_to_f64(xb)).sum(axis=0)))
    with pytest.raises(AssertionError):
        D.test_column_sums_exact()


def test_grouped_expert_index_mistake_is_caught(monkeypatch):
    # experts numbered by non-empty groups only: every group after an empty one uses the wrong weights
    def shifted(qx, sx, group_m, qw, sw, bias_bits=None, gelu=False):
        nonempty = [i for i, m in enumerate(group_m) if int(m) > 0]
        out = {"pre": None, "d": [], "aux": [] if gelu else None, "sigma": None}
        row = 0
        for j, g in enumerate(nonempty):
            m = int(group_m[g])
            r = O.mx_gemm(qx[row:row + m], sx[row:row + m], qw[j], sw[j],
                          None if bias_bits is None else bias_bits[j], gelu)
            out["d"].append(r["d"])
            if gelu:
                out["aux"].append(r["aux"])
            row += m
        out["d"] = np.concatenate(out["d"])
        if gelu:
            out["aux"] = np.concatenate(out["aux"])
        return out
    monkeypatch.setattr(O, "mx_grouped_gemm", shifted)
    with pytest.raises(AssertionError):
        G.test_grouped_equals_per_group_dense_with_empty_groups()
