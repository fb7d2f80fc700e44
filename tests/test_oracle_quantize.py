"""Pins for the oracle's quantiser: checks against facts that do not come from the oracle.

* hand-worked blocks in tests/golden/mx_blocks.txt;
* brute force over every code of the E4M3 format and every bf16 pattern;
* library routes (torch's float8_e4m3fn and bfloat16 casts);
* the invariants of the MX scale rule (power-of-two shifts, saturation,
  idempotent re-quantisation, column-wise == row-wise of the transpose).
"""
import os

import numpy as np
import pytest
import torch

from oracle import mx_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_blocks.txt")


def parse_golden(path=GOLDEN):
    blocks, cur = [], None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "block":
            cur = {"name": tok[1], "vals": [], "q": []}
        elif tok[0] == "scale":
            cur["scale"] = int(tok[1], 16)
        elif tok[0] == "elem":
            v = {"nan": float("nan"), "-0": -0.0}.get(tok[1])
            if v is None:
                v = float.fromhex(tok[1])
            n = int(tok[3][1:]) if len(tok) > 3 else 1
            cur["vals"] += [v] * n
            cur["q"] += [int(tok[2], 16)] * n
        elif tok[0] == "end":
            assert len(cur["vals"]) == 32, (cur["name"], len(cur["vals"]))
            blocks.append(cur)
    return blocks


def to_bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float64), torch.tensor(vals, dtype=torch.float64)) or any(
        np.isnan(vals)), "golden values must be exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def finite_e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


# ---------------------------------------------------------------- golden blocks

@pytest.mark.parametrize("blk", parse_golden(), ids=lambda b: b["name"])
def test_golden_block_rowwise(blk):
    bits = to_bf16_bits(blk["vals"]).reshape(1, 32)
    q, s = O.quantize_rowwise(bits)
    assert int(s[0, 0]) == blk["scale"]
    assert q[0].tolist() == blk["q"]


@pytest.mark.parametrize("blk", parse_golden(), ids=lambda b: b["name"])
def test_golden_block_colwise(blk):
    bits = to_bf16_bits(blk["vals"]).reshape(32, 1)
    q, s = O.quantize_colwise(bits)
    assert q.shape == (1, 32) and s.shape == (1, 1)
    assert int(s[0, 0]) == blk["scale"]
    assert q[0].tolist() == blk["q"]


# ---------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_matches_library_for_every_code():
    codes, lib = finite_e4m3_table()
    ours = O.e4m3_decode(codes)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                      # 0x7F and 0xFF only
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert O.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def brute_force_e4m3(v):
    """Nearest finite E4M3 code by exhaustive search, ties to the even code."""
    codes, vals = finite_e4m3_table()
    pos = (codes <= 0x7E)
    pc, pv = codes[pos].astype(np.int64), vals[pos]        # 0x00 .. 0x7E, ascending
    a = np.abs(v)[:, None]
    d = np.abs(a - pv[None, :])
    best = d.min(axis=1, keepdims=True)
    tie = d == best
    # among equally near codes prefer the one with an even mantissa (code LSB 0)
    score = np.where(tie, np.where(pc[None, :] % 2 == 0, 0, 1), 2)
    idx = np.argmin(score, axis=1)
    out = pc[idx]
    return (out | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def e4m3_probe_values():
    """Every bf16 value below 600, all E4M3 midpoints and +-1 fp64 ulp around them."""
    bf = O.bf16_bits_to_f64(ALL_BF16)
    bf = bf[np.isfinite(bf) & (np.abs(bf) < 600)]
    _, vals = finite_e4m3_table()
    pv = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pv[1:] + pv[:-1]) / 2
    mids = np.concatenate([mids, [448.0 + 16.0, 480.0, 512.0, 1e6]])
    near = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    return np.concatenate([bf, near, -near, [0.0, -0.0]])


def test_e4m3_encode_equals_brute_force_nearest():
    v = e4m3_probe_values()
    assert np.array_equal(O.e4m3_encode(v), brute_force_e4m3(v))


def test_e4m3_encode_matches_library_saturating_cast():
    v = e4m3_probe_values().astype(np.float32)        # all probe values are fp32-exact or near
    v64 = v.astype(np.float64)
    lib = torch.from_numpy(v).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v64), lib)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_library_on_fp32_inputs():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(200000, generator=g) * 10.0 ** torch.randint(-30, 30, (200000,), generator=g),
                   torch.tensor([0.0, -0.0, 3.3895313892515355e38, 3.4e38, -3.4e38, 1e-40, -1e-45])])
    lib = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = O.f64_to_bf16_bits(x.to(torch.float64).numpy())
    assert np.array_equal(ours, lib)


def test_bf16_round_midpoints_in_fp64():
    vals = O.bf16_bits_to_f64(ALL_BF16)
    vals = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2                                # exact in fp64
    lo_bits = O.f64_to_bf16_bits(lo)
    expect_mid = np.where(lo_bits % 2 == 0, lo, hi)    # ties to even
    assert np.array_equal(O.bf16_round(mid), expect_mid)
    assert np.array_equal(O.bf16_round(np.nextafter(mid, 0)), lo)
    assert np.array_equal(O.bf16_round(np.nextafter(mid, np.inf)), hi)
    assert np.isinf(O.bf16_round(2.0 ** 128))


# ---------------------------------------------------------------- scale rule

def test_scale_rule_exhaustive_against_brute_force():
    vals = O.bf16_bits_to_f64(ALL_BF16)
    amax = vals[np.isfinite(vals) & (vals > 0)]
    # brute force: the smallest e in [-127, 127] with amax * 2^-e < 512 (= 2^(8+1))
    es = np.arange(-127, 128)
    ok = amax[:, None] * np.ldexp(1.0, -es)[None, :] < 512.0
    brute = es[np.argmax(ok, axis=1)]
    assert np.array_equal(O.mx_scale_exponent(amax), brute)
    assert O.mx_scale_exponent(0.0) == -127


# ---------------------------------------------------------------- invariants

def random_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("k", [-20, -3, 1, 5, 40])
def test_power_of_two_scaling_shifts_only_the_scale(k):
    x = random_bf16((64, 256), seed=11)
    xs = O.f64_to_bf16_bits(O.bf16_bits_to_f64(x) * 2.0 ** k)   # exact
    q0, s0 = O.quantize_rowwise(x)
    q1, s1 = O.quantize_rowwise(xs)
    assert np.array_equal(q0, q1)
    assert np.array_equal(s1.astype(np.int64), s0.astype(np.int64) + k)


def test_values_beyond_range_saturate():
    x = np.clip(O.bf16_bits_to_f64(random_bf16((8, 64), seed=3)), -1.5, 1.5)
    x[:, 0] = 1.9375                     # the block amax, mantissa above 1.75 -> it saturates
    q, s = O.quantize_rowwise(O.f64_to_bf16_bits(x))
    assert np.all(q[:, 0] == 0x7E)
    assert np.all(s[:, 0] == 127 - 8)
    q_all = O.e4m3_decode(q)
    assert np.nanmax(np.abs(q_all)) == 448.0


def test_requantising_dequantised_blocks_is_idempotent():
    x = random_bf16((128, 512), seed=5, std=3.0)
    q, s = O.quantize_rowwise(x)
    deq = O.dequantize(q, s)
    bits = O.f64_to_bf16_bits(deq)
    assert np.array_equal(O.bf16_bits_to_f64(bits), deq)       # representable in bf16
    q2, s2 = O.quantize_rowwise(bits)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_colwise_is_rowwise_of_transpose():
    x = random_bf16((96, 160), seed=9)
    qc, sc = O.quantize_colwise(x)
    qr, sr = O.quantize_rowwise(np.ascontiguousarray(x.T))
    assert qc.shape == (160, 96) and sc.shape == (160, 3)
    assert np.array_equal(qc, qr) and np.array_equal(sc, sr)
    # and column c of X really is row c of the column-wise copy
    one = O.quantize_rowwise(np.ascontiguousarray(x[:, 7].reshape(1, 96)))
    assert np.array_equal(qc[7], one[0][0]) and np.array_equal(sc[7], one[1][0])


def test_zero_block_gives_zero_codes():
    x = np.zeros((2, 64), dtype=np.uint16)
    q, s = O.quantize_rowwise(x)
    assert not q.any() and not s.any()


def test_dequantised_error_within_half_e4m3_ulp():
    x = random_bf16((256, 256), seed=21)
    q, s = O.quantize_rowwise(x)
    xf = O.bf16_bits_to_f64(x)
    deq = O.dequantize(q, s)
    scale = np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
    v = np.abs(xf) / scale
    # half an ulp of E4M3 at |v| (or of the subnormal step), unless saturated
    _, p = np.frexp(v)
    ulp = np.ldexp(1.0, np.maximum(p - 1, -6) - 3)
    sat = v > 448
    err = np.abs(deq - xf) / scale
    assert np.all(err[~sat] <= ulp[~sat] / 2)
    assert np.all(np.abs(deq[sat]) / scale[sat] == 448)
