"""Pins for the LayerNorm -> MXFP8 part of the oracle.

* ``layernorm`` against torch.nn.functional.layer_norm and torch.var_mean in
  float64 (a library route), hand-worked rows, constant rows, shift invariance;
* ``layernorm_error_bound`` against fp32 evaluations of the same formula in
  several summation orders (numpy float32), including rows with a large mean;
* ``mx_admissible``: with zero error it accepts exactly the unique
  quantisation; it rejects a changed code, a changed scale and a zero of the
  wrong sign; near a rounding midpoint it accepts both neighbours;
* planted mistakes in a copy of the LayerNorm (unbiased variance, eps outside
  the square root, dropped beta) fail the torch comparison.
"""
import numpy as np
import pytest
import torch

from oracle import mx_oracle as O


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def make(rows, h, seed, mean=0.0, std=1.0):
    g = torch.Generator().manual_seed(seed)
    x = bits_of(torch.randn(rows, h, generator=g) * std + mean)
    ga = bits_of(1.0 + 0.1 * torch.randn(h, generator=g))
    be = bits_of(0.1 * torch.randn(h, generator=g))
    return x, ga, be


def f64(bits):
    return O.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("rows,h,mean", [(16, 64, 0.0), (8, 1024, 0.0), (4, 4096, 30.0)])
def test_layernorm_matches_torch_float64(rows, h, mean):
    x, ga, be = make(rows, h, rows + h, mean=mean)
    y, mu, rs = O.layernorm(x, ga, be)
    xt = torch.from_numpy(f64(x))
    want = torch.nn.functional.layer_norm(xt, (h,), torch.from_numpy(f64(ga)), torch.from_numpy(f64(be)), eps=1e-5)
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-12, atol=1e-12)
    var, m = torch.var_mean(xt, dim=1, unbiased=False)
    np.testing.assert_allclose(mu, m.numpy(), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rs, (1.0 / torch.sqrt(var + 1e-5)).numpy(), rtol=1e-12)


def test_hand_worked_row_and_constant_row():
    x = O.f64_to_bf16_bits(np.array([[1.0, 2.0, 3.0, 4.0], [5.0, 5.0, 5.0, 5.0]]))
    ga = O.f64_to_bf16_bits(np.array([1.0, 2.0, 1.0, 1.0]))
    be = O.f64_to_bf16_bits(np.array([0.0, 0.0, 0.5, -1.0]))
    y, mu, rs = O.layernorm(x, ga, be)
    # row 0: mean 2.5, deviations -1.5 -0.5 0.5 1.5, variance (2.25+0.25+0.25+2.25)/4 = 1.25
    assert mu[0] == 2.5
    assert rs[0] == 1.0 / np.sqrt(1.25 + 1e-5)
    r = rs[0]
    np.testing.assert_array_equal(y[0], [-1.5 * r, -0.5 * r * 2.0, 0.5 * r + 0.5, 1.5 * r - 1.0])
    # constant row: every deviation is 0, so y = beta exactly and rsigma = 1/sqrt(eps)
    assert mu[1] == 5.0 and rs[1] == 1.0 / np.sqrt(1e-5)
    np.testing.assert_array_equal(y[1], [0.0, 0.0, 0.5, -1.0])


def test_shift_invariance():
    g = torch.Generator().manual_seed(3)
    xi = torch.randint(-20, 20, (8, 256), generator=g).double()         # integers: x + 64 exact in bf16
    _, ga, be = make(8, 256, 4)
    y0, _, rs0 = O.layernorm(bits_of(xi), ga, be)
    y1, _, rs1 = O.layernorm(bits_of(xi + 64.0), ga, be)
    np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(rs1, rs0, rtol=1e-14)


def fp32_layernorm(x_bits, ga_bits, be_bits, order, eps=1e-5):
    """The fp32 evaluation the error bound covers, with a chosen summation order
    of depth <= 64 ('pairwise': numpy's pairwise float32 sum; 'chunks': 8
    pieces summed left to right in blocks of 32 and then combined)."""
    x = f64(x_bits).astype(np.float32)
    g = f64(ga_bits).astype(np.float32)
    b = f64(be_bits).astype(np.float32)
    h = x.shape[1]

    def rowsum(v):
        if order == "pairwise":
            return np.sum(v, axis=1, dtype=np.float32)
        acc = np.zeros(v.shape[0], np.float32)
        for c in range(0, h, 32):                        # per 32-column block, left to right
            part = np.zeros(v.shape[0], np.float32)
            for j in range(c, min(c + 32, h)):
                part = np.float32(part + v[:, j])
            acc = np.float32(acc + part)
        return acc

    mu = np.float32(rowsum(x) / np.float32(h))
    d = (x - mu[:, None]).astype(np.float32)
    var = np.float32(rowsum((d * d).astype(np.float32)) / np.float32(h))
    rs = np.float32(np.float32(1.0) / np.sqrt(np.float32(var + np.float32(eps))))
    n = (d * rs[:, None]).astype(np.float32)
    y = (n.astype(np.float64) * g.astype(np.float64) + b.astype(np.float64)).astype(np.float32)   # one rounding
    return y.astype(np.float64)


@pytest.mark.parametrize("order", ["pairwise", "chunks"])
@pytest.mark.parametrize("rows,h,mean,std", [(32, 1024, 0.0, 1.0), (16, 2048, 100.0, 1.0), (16, 512, 0.0, 1e-3),
                                             (8, 1024, 3.0, 30.0)])
def test_error_bound_covers_fp32_evaluation(order, rows, h, mean, std):
    x, ga, be = make(rows, h, 7 * rows + h, mean=mean, std=std)
    y, _, _ = O.layernorm(x, ga, be)
    e = O.layernorm_error_bound(x, ga)
    got = fp32_layernorm(x, ga, be, order)
    assert np.all(np.abs(got - y) <= e), float(np.max(np.abs(got - y) / e))


def test_admissible_with_zero_error_is_exact():
    x, ga, be = make(64, 256, 9)
    y, _, _ = O.layernorm(x, ga, be)
    for axis in (1, 0):
        q, s = O.quantize_mx_values(y, axis)
        ok, amb = O.mx_admissible(y, 0.0, q, s, axis)
        assert ok.all() and not amb.any()
        q2 = q.copy(); q2[3, 5] ^= 0x01
        ok, _ = O.mx_admissible(y, 0.0, q2, s, axis)
        assert not ok[3, 5] and ok.sum() == ok.size - 1
        s2 = s.copy(); s2[2, 1] += 1
        ok, _ = O.mx_admissible(y, 0.0, q, s2, axis)
        assert not ok[2, 32:64].any()


def test_admissible_midpoint_and_signed_zero():
    # block of 32: amax 1.0 -> exponent -8, element 1.0 + 2^-4 (times 2^8 = 272) sits midway
    # between the E4M3 neighbours 256 and 288
    y = np.zeros((1, 32))
    y[0, 0] = 1.0
    y[0, 1] = 1.0625
    y[0, 2] = 1e-9                 # positive, rounds to +0
    q, s = O.quantize_mx_values(y, 1)
    ok, amb = O.mx_admissible(y, 0.0, q, s, 1)
    assert ok.all() and not amb.any()
    q_up = q.copy(); q_up[0, 1] += 1                       # the other neighbour
    ok, _ = O.mx_admissible(y, 0.0, q_up, s, 1)
    assert not ok[0, 1]
    err = np.full(y.shape, 1e-6)
    ok, amb = O.mx_admissible(y, err, q_up, s, 1)
    assert ok[0, 1] and amb[0, 1]
    q_neg = q.copy(); q_neg[0, 2] = 0x80                   # -0 for a value that is positive
    ok, _ = O.mx_admissible(y, 1e-12, q_neg, s, 1)
    assert not ok[0, 2]


def test_admissible_non_finite_rows():
    y = np.ones((2, 64))
    y[1, 40] = np.nan
    q, s = O.quantize_mx_values(y, 1)
    ok, amb = O.mx_admissible(y, 1e-7, q, s, 1)
    assert ok.all() and s[1, 1] == 0xFF and np.all(q[1, 32:] == 0x7F)
    q2 = q.copy(); q2[1, 40] = 0x7E
    ok, _ = O.mx_admissible(y, 1e-7, q2, s, 1)
    assert not ok[1, 40]


def _mutant(kind):
    def ln(x_bits, gamma_bits, beta_bits, eps=1e-5):
        x, g, b = f64(x_bits), f64(gamma_bits), f64(beta_bits)
        mu = x.mean(axis=1)
        if kind == "unbiased":
            var = ((x - mu[:, None]) ** 2).sum(axis=1) / (x.shape[1] - 1)
        else:
            var = ((x - mu[:, None]) ** 2).mean(axis=1)
        rs = 1.0 / (np.sqrt(var) + eps) if kind == "eps_outside" else 1.0 / np.sqrt(var + eps)
        y = (x - mu[:, None]) * rs[:, None] * g
        return (y if kind == "no_beta" else y + b), mu, rs
    return ln


@pytest.mark.parametrize("kind", ["unbiased", "eps_outside", "no_beta"])
def test_planted_mistakes_fail_the_torch_pin(kind, monkeypatch):
    monkeypatch.setattr(O, "layernorm", _mutant(kind))
    with pytest.raises(AssertionError):
        test_layernorm_matches_torch_float64(16, 64, 0.0)
