"""Pins for the backward parts of the oracle: dGELU and the bias gradient.

* dgelu_tanh against torch autograd of the tanh-approximate GELU (library
  route) and against central finite differences of gelu_tanh in fp64;
* the dGELU GEMM against the plain product of the dequantised operands and
  the derivative, and its sign/zero structure;
* column sums against exact rational sums.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O


def test_dgelu_matches_autograd():
    x = torch.linspace(-12, 12, 20001, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(x, approximate="tanh").sum().backward()
    ours = O.dgelu_tanh(x.detach().numpy())
    assert np.allclose(ours, x.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_dgelu_matches_finite_differences():
    x = np.linspace(-8, 8, 4001)
    h = 1e-5
    fd = (O.gelu_tanh(x + h) - O.gelu_tanh(x - h)) / (2 * h)
    assert np.allclose(O.dgelu_tanh(x), fd, rtol=1e-7, atol=1e-9)
    assert O.dgelu_tanh(0.0) == 0.5
    assert abs(O.dgelu_tanh(30.0) - 1.0) < 1e-12 and abs(O.dgelu_tanh(-30.0)) < 1e-12


def rand_bits(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_dgelu_gemm_is_product_with_derivative():
    qa, sa = O.quantize_rowwise(rand_bits((16, 128), 1))
    qb, sb = O.quantize_rowwise(rand_bits((24, 128), 2))
    aux = rand_bits((16, 24), 3, std=2.0)
    out = O.mx_gemm_dgelu(qa, sa, qb, sb, aux)
    plain = O.mx_gemm(qa, sa, qb, sb)["pre"]
    g = O.dgelu_tanh(O.bf16_bits_to_f64(aux))
    assert np.array_equal(out["pre"], plain * g)
    # aux = 0 -> derivative 1/2 exactly
    out0 = O.mx_gemm_dgelu(qa, sa, qb, sb, np.zeros((16, 24), np.uint16))
    assert np.array_equal(out0["pre"], plain * 0.5)


def test_column_sums_exact():
    x = rand_bits((64, 32), 4, std=3.0)
    s, a = O.column_sums(x)
    xv = O.bf16_bits_to_f64(x)
    for c in (0, 7, 31):
        assert Fraction(s[c]) == sum(Fraction(v) for v in xv[:, c])
        assert Fraction(a[c]) == sum(abs(Fraction(v)) for v in xv[:, c])


def _dgelu_decimal(x: float):
    """The tanh-form derivative evaluated with 160-digit decimal arithmetic."""
    from decimal import Decimal, getcontext
    getcontext().prec = 160
    X = Decimal(x)
    pi = Decimal("3.14159265358979323846264338327950288419716939937510582097494")
    c = (Decimal(2) / pi).sqrt()
    u = c * (X + Decimal("0.044715") * X ** 3)
    e2 = (2 * u).exp()
    t = (e2 - 1) / (e2 + 1)
    return float(Decimal("0.5") * (1 + t) + Decimal("0.5") * X * (1 - t * t) * c *
                 (1 + 3 * Decimal("0.044715") * X ** 2))


@pytest.mark.parametrize("x", [-12.0, -9.5, -7.21875, -5.0, -2.0, -0.75, 0.0, 0.5, 3.0, 8.0])
def test_dgelu_relative_accuracy_in_the_tails(x):
    ref = _dgelu_decimal(x)
    got = float(O.dgelu_tanh(x))
    assert abs(got - ref) <= 1e-13 * abs(ref) + 1e-300
