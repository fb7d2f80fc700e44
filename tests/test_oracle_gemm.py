"""Pins for the oracle's GEMM, epilogues and grouped GEMM.

* exact rational arithmetic (fractions.Fraction) on tiny shapes, with operand
  values decoded through torch's float8_e4m3fn (not the oracle's decoder);
* identity-B: D reproduces the dequantised A bit-exactly;
* GELU-tanh against torch's tanh-approximate GELU and the identity
  gelu(x) - gelu(-x) = x, GELU(0) = 0;
* power-of-two scaling of A scales the pre-activation exactly;
* the grouped GEMM equals per-group dense GEMMs, with empty groups.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O


def rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def lib_decode(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("m,n,k", [(16, 16, 32), (8, 24, 64), (5, 3, 128)])
def test_tiny_gemm_exact_rational(m, n, k):
    qa, sa = O.quantize_rowwise(rand_bf16((m, k), 1 + m))
    qb, sb = O.quantize_rowwise(rand_bf16((n, k), 2 + n))
    bias = rand_bf16((n,), 3)
    av, bv = lib_decode(qa), lib_decode(qb)
    bias_v = torch.from_numpy(bias.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    out = O.mx_gemm(qa, sa, qb, sb, bias)
    for i in range(m):
        for j in range(n):
            acc = Fraction(bias_v[j])
            sig = Fraction(0)
            for kk in range(k):
                ta = Fraction(av[i, kk]) * Fraction(2) ** (int(sa[i, kk // 32]) - 127)
                tb = Fraction(bv[j, kk]) * Fraction(2) ** (int(sb[j, kk // 32]) - 127)
                acc += ta * tb
                sig += abs(ta * tb)
            assert Fraction(out["pre"][i, j]) == acc
            assert Fraction(out["sigma"][i, j]) == sig


def test_identity_b_reproduces_dequantised_a():
    k = 256
    qa, sa = O.quantize_rowwise(rand_bf16((64, k), 4, std=2.0))
    eye_bits = O.f64_to_bf16_bits(np.eye(k))
    qb, sb = O.quantize_rowwise(eye_bits)
    assert np.all(qb[np.eye(k, dtype=bool)] == 0x78)
    diag_block = np.arange(k)[:, None] // 32 == np.arange(k // 32)[None, :]
    assert np.all(sb[diag_block] == 127 - 8) and np.all(sb[~diag_block] == 0)
    out = O.mx_gemm(qa, sa, qb, sb)
    assert np.array_equal(out["d"], O.dequantize(qa, sa))


def test_gelu_matches_library_and_identities():
    x = np.linspace(-12, 12, 20001)
    lib = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    # both evaluate 0.5 x (1 + tanh u) in fp64; for x << 0 the sum 1 + tanh u
    # cancels, so they agree to a few fp64 ulps of |x| rather than of the result
    ours = O.gelu_tanh(x)
    assert np.all(np.abs(ours - lib) <= 1e-13 * np.abs(lib) + 8 * np.finfo(np.float64).eps * np.abs(x))
    assert O.gelu_tanh(0.0) == 0.0
    assert np.allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, rtol=1e-13, atol=1e-13)


def test_gelu_epilogue_zero_and_bias():
    k = 128
    qa, sa = O.quantize_rowwise(np.zeros((4, k), np.uint16))
    qb, sb = O.quantize_rowwise(rand_bf16((6, k), 8))
    out = O.mx_gemm(qa, sa, qb, sb, None, gelu=True)
    assert not out["d"].any() and not out["aux"].any()
    bias = rand_bf16((6,), 9)
    out = O.mx_gemm(qa, sa, qb, sb, bias, gelu=True)
    b = O.bf16_bits_to_f64(bias)
    lib = torch.nn.functional.gelu(torch.from_numpy(b), approximate="tanh").to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(out["d"][0], lib.to(torch.float64).numpy())
    assert np.array_equal(out["aux"][0], b)


@pytest.mark.parametrize("kexp", [-9, 4])
def test_scaling_a_by_power_of_two_scales_pre(kexp):
    x = rand_bf16((16, 256), 12)
    qa, sa = O.quantize_rowwise(x)
    qa2, sa2 = O.quantize_rowwise(O.f64_to_bf16_bits(O.bf16_bits_to_f64(x) * 2.0 ** kexp))
    qb, sb = O.quantize_rowwise(rand_bf16((8, 256), 13))
    r1 = O.mx_gemm(qa, sa, qb, sb)["pre"]
    r2 = O.mx_gemm(qa2, sa2, qb, sb)["pre"]
    assert np.array_equal(r2, r1 * 2.0 ** kexp)


def test_transposed_operands_are_distinguished():
    # D = A B^T with B row j -> column j of D: a plain check on one nonzero block
    k = 64
    a = np.zeros((3, k)); a[1, 40] = 2.0
    b = np.zeros((5, k)); b[4, 40] = 0.5
    qa, sa = O.quantize_rowwise(O.f64_to_bf16_bits(a))
    qb, sb = O.quantize_rowwise(O.f64_to_bf16_bits(b))
    d = O.mx_gemm(qa, sa, qb, sb)["d"]
    expect = np.zeros((3, 5)); expect[1, 4] = 1.0
    assert np.array_equal(d, expect)


def test_grouped_equals_per_group_dense_with_empty_groups():
    k, n = 128, 48
    group_m = [5, 0, 17, 0, 1, 9]
    total = sum(group_m)
    qx, sx = O.quantize_rowwise(rand_bf16((total, k), 20))
    w = rand_bf16((len(group_m), n, k), 21, std=0.1)
    qw = np.stack([O.quantize_rowwise(w[g])[0] for g in range(len(group_m))])
    sw = np.stack([O.quantize_rowwise(w[g])[1] for g in range(len(group_m))])
    bias = rand_bf16((len(group_m), n), 22)
    out = O.mx_grouped_gemm(qx, sx, group_m, qw, sw, bias, gelu=True)
    row = 0
    for g, m in enumerate(group_m):
        if m:
            ref = O.mx_gemm(qx[row:row + m], sx[row:row + m], qw[g], sw[g], bias[g], gelu=True)
            assert np.array_equal(out["d"][row:row + m], ref["d"])
            assert np.array_equal(out["aux"][row:row + m], ref["aux"])
        row += m


def test_fp32_accumulation_is_within_the_bound():
    # the acceptance bound admits an fp32-accumulated result of the same GEMM
    qa, sa = O.quantize_rowwise(rand_bf16((32, 1024), 30))
    qb, sb = O.quantize_rowwise(rand_bf16((32, 1024), 31, std=0.02))
    ref = O.mx_gemm(qa, sa, qb, sb)
    a32 = O.dequantize(qa, sa).astype(np.float32)
    b32 = O.dequantize(qb, sb).astype(np.float32)
    d32 = O.bf16_round((a32 @ b32.T).astype(np.float64))
    assert np.all(np.abs(d32 - ref["d"]) <= O.gemm_error_bound(ref["d"], ref["sigma"]))
