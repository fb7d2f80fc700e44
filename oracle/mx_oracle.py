"""CPU oracle for MXFP8 block-scaled quantisation and the MXFP8 GEMM.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
definition that the CUDA path is checked against.  Only the test suite, the
smoke check of the package entry point and the CPU-baseline leg of the bench
may import it.  The product path never calls it, and it shares no code with
the CUDA library: it imports numpy alone.

All arithmetic is float64 (exact for every value that occurs here: bf16 and
E4M3 values times powers of two), rounding steps are written out as
definitions, and a library primitive (numpy's matmul) is the only "fast" step.

Sources of the definitions
--------------------------
* "HipKittens MXFP8 GEMM Support", ROCm/TransformerEngine PR #566 (PR
  description and review thread): the GEMM is an MXFP8 TN GEMM with a per-K
  block scale array (``scale_K``), BIAS and GELU-AUX epilogues, K a multiple
  of 128 "for MXFP8 scaling", and the MXFP8 1D scaling mode.
* ROCm/TransformerEngine README, sections "MXFP8 support on ROCm" and
  "Blockwise FP8 GEMM support on ROCm": MX scales are E8M0 (power of two).
* leeroopedia "FP8 Training Quickstart", step on autocast recipes: E4M3 is the
  forward-pass FP8 format.
* The pages name MXFP8 but never define its numerics.  The block size (32),
  the scale rule and the element format are those of the OCP Microscaling
  Formats (MX) v1.0 specification, FP32 -> MX conversion: shared exponent
  = floor(log2(max |V_i|)) - emax(element), element = V_i / 2^shared_exp
  rounded to nearest-even in E4M3 and clamped to the largest normal (448).
  E4M3 itself is the OCP 8-bit floating point "E4M3" encoding (bias 7, no
  infinities, S.1111.111 is NaN, largest normal 448).
* GELU-tanh: the tanh approximation of GELU named on the TE "Getting
  Started" page (``approximate=True``), 0.5 x (1 + tanh(sqrt(2/pi) (x +
  0.044715 x^3))); its derivative (dGELU) for the backward epilogue named in
  ROCm/TransformerEngine README, "Blockwise FP8 GEMM support on ROCm"
  (bias/beta/DGELU epilogues).
* Float8BlockScaling (ROCm/TransformerEngine README, "Blockwise FP8 GEMM support
  on ROCm"): 1x128 blocks for activations/gradients, 128x128 blocks for
  weights, each with an FP32 scale amax / 448 that is cast to E8M0 (the
  default there).  Reading of the cast: the smallest power of two >= amax/448,
  i.e. 2^ceil(log2(amax / 448)), so that no element exceeds 448 after scaling.
* LayerNorm -> MXFP8 (LayerNormLinear / LayerNormMLP input): see the section
  of that name below.
* Bias gradient: the column sums of the output gradient (the cast_transpose_bgrad
  kernels of ROCm/TransformerEngine README, "Experimental Triton Kernels on ROCm").

Readings where the sources are silent (each one is listed in the design notes):
* amax == 0: the scale byte is 0x00 (2^-127, the smallest E8M0 value); every
  element is +-0.
* The scale exponent is clamped to [-127, 127] (E8M0's finite range).
* A negative value that rounds to zero keeps its sign (code 0x80).
* A block holding a NaN or an infinity: scale byte 0xFF (E8M0 NaN) and every
  element code 0x7F (E4M3 NaN).
* Float8BlockScaling with FP32 scales (the README's second mode): the scale is
  s = amax / 448 rounded to fp32; elements are multiplied by r = fl32(1 / s)
  in fp32 (one multiply per element, as a quantiser does) and rounded to E4M3
  (nearest even, saturating); r is capped at the largest finite fp32;
  amax == 0 gives s = r = 1.
* GELU is applied to the unrounded pre-activation; AUX is that
  pre-activation rounded to bf16.
"""
from __future__ import annotations

import numpy as np

MX_BLOCK = 32              # elements per E8M0 scale (OCP MX block size)
E4M3_EMAX = 8              # exponent of the largest E4M3 binade (448 = 1.75 * 2^8)
E4M3_MAX = 448.0
E4M3_MANT_BITS = 3
E4M3_EMIN = -6             # smallest normal exponent; subnormal step 2^-9
E4M3_BIAS = 7
E8M0_BIAS = 127
BF16_MANT_BITS = 7
BF16_EMIN = -126
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127

# --------------------------------------------------------------------------
# Exact exponent helpers
# --------------------------------------------------------------------------
# Every nonzero value handled here is a normal IEEE-754 double (the smallest
# magnitudes are bf16 subnormals, about 2^-133, far above 2^-1022), so
# floor(log2 |v|) is the double's unbiased exponent field and 2^e is the double
# with exponent field e + 1023 and a zero fraction.


def floor_log2(v) -> np.ndarray:
    """floor(log2 |v|) for normal doubles (int64); -1023 for 0."""
    bits = np.asarray(v, dtype=np.float64).view(np.uint64)
    return ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1023


def pow2(e) -> np.ndarray:
    """2.0 ** e for integer e in [-1022, 1023], exactly."""
    e = np.asarray(e, dtype=np.int64)
    return ((e + 1023).astype(np.uint64) << np.uint64(52)).view(np.float64)


# --------------------------------------------------------------------------
# Rounding to a binary floating-point format
# --------------------------------------------------------------------------


def round_to_binary_format(v, mant_bits: int, emin: int) -> np.ndarray:
    """Round float64 values to the nearest value of a binary FP format, ties to even.

    The format has ``mant_bits`` fraction bits and smallest normal exponent
    ``emin``; below 2^emin it is subnormal with step 2^(emin - mant_bits).
    It is unbounded above (overflow is the caller's business).  The sign is
    kept, so a negative value that rounds to zero gives -0.0.
    """
    v = np.asarray(v, dtype=np.float64)
    e = np.maximum(floor_log2(v), emin)   # held at emin for subnormals (and zero)
    quantum = pow2(e - mant_bits)
    # v / quantum is exact (division by a power of two); np.round is ties-to-even.
    return np.round(v / quantum) * quantum


def bf16_round(v) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64.

    Overflow goes to +-inf, as in IEEE round-to-nearest-even.
    """
    r = round_to_binary_format(v, BF16_MANT_BITS, BF16_EMIN)
    v = np.asarray(v, dtype=np.float64)
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, v), r)
    return np.where(np.isnan(v), np.nan, r)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):          # NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 to bf16 (ties to even) and return the uint16 bit patterns."""
    r = bf16_round(v).astype(np.float32)          # exact: every bf16 value is an fp32 value
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# E4M3 (OCP FP8 "E4M3") codec
# --------------------------------------------------------------------------


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 bytes to float64: sign | 4-bit exponent (bias 7) | 3-bit mantissa.

    Exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no
    infinity.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp_field = (c >> 3) & 0xF
    mant = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + mant / 8.0, exp_field - E4M3_BIAS)
    subnormal = np.ldexp(mant / 8.0, E4M3_EMIN)
    mag = np.where(exp_field == 0, subnormal, normal)
    mag = np.where((exp_field == 0xF) & ((c & 0x7) == 0x7), np.nan, mag)
    return sign * mag


def e4m3_round_saturate(v) -> np.ndarray:
    """Round float64 to the nearest E4M3 value (ties to even), then clamp to +-448.

    Rounding first and clamping after gives the saturating conversion: every
    |v| that would round above 448 becomes 448.
    """
    r = round_to_binary_format(v, E4M3_MANT_BITS, E4M3_EMIN)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def e4m3_encode_value(r) -> np.ndarray:
    """Bit pattern of an (already representable) E4M3 value; -0.0 -> 0x80."""
    r = np.asarray(r, dtype=np.float64)
    sign = np.signbit(r).astype(np.int64) << 7
    a = np.abs(r)
    e = floor_log2(a)
    is_sub = a < 2.0 ** E4M3_EMIN
    sub_mant = np.round(a / 2.0 ** (E4M3_EMIN - E4M3_MANT_BITS)).astype(np.int64)
    safe_e = np.where(is_sub | ~np.isfinite(a), 0, e)
    norm_mant = np.round((a / pow2(safe_e) - 1.0) * 8.0).astype(np.int64)
    norm_field = (safe_e + E4M3_BIAS).astype(np.int64)
    code = np.where(is_sub, sub_mant, (norm_field << 3) | norm_mant)
    return (sign | code).astype(np.uint8)


def e4m3_encode(v) -> np.ndarray:
    """float64 -> E4M3 byte: round to nearest even, saturate to +-448, keep sign of zero."""
    return e4m3_encode_value(e4m3_round_saturate(v))


# --------------------------------------------------------------------------
# MXFP8 quantisation
# --------------------------------------------------------------------------


def mx_scale_exponent(amax) -> np.ndarray:
    """Shared exponent of an MX block: floor(log2 amax) - 8, clamped to [-127, 127].

    floor(log2) is taken exactly from the exponent field (never from a log function).
    amax == 0 gives -127 (reading: the smallest E8M0 scale).
    """
    amax = np.asarray(amax, dtype=np.float64)
    e = np.clip(floor_log2(amax) - E4M3_EMAX, -E8M0_BIAS, E8M0_BIAS)
    return np.where(amax == 0.0, -E8M0_BIAS, e).astype(np.int64)


def quantize_mx(x_bits, axis: int):
    """MXFP8-quantise a bf16 matrix along ``axis`` in blocks of 32.

    ``x_bits``: uint16 bf16 patterns, shape [R, C].  Blocks are 32 consecutive
    elements along ``axis`` (1: along a row; 0: down a column), so that axis
    must have a length divisible by 32.

    Returns ``(q, s)`` laid out with the blocked axis last and contiguous:
      axis=1: q uint8 [R, C],  s uint8 [R, C/32]
      axis=0: q uint8 [C, R],  s uint8 [C, R/32]   (the transposed copy)
    where s is the E8M0 byte (exponent + 127) and q the E4M3 byte.
    """
    return quantize_mx_values(bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16)), axis)


def quantize_mx_values(x, axis: int):
    """``quantize_mx`` of real (float64) values instead of bf16 patterns."""
    x = np.asarray(x, dtype=np.float64)
    if axis == 0:
        x = x.T                                   # put the blocked axis last
    rows, n = x.shape
    if n % MX_BLOCK:
        raise ValueError(f"blocked axis length {n} is not a multiple of {MX_BLOCK}")
    blocks = x.reshape(rows, n // MX_BLOCK, MX_BLOCK)
    with np.errstate(invalid="ignore"):
        amax = np.max(np.abs(blocks), axis=2)
    bad = ~np.isfinite(amax)                      # block holds NaN or inf
    amax_f = np.where(bad, 1.0, amax)
    e = mx_scale_exponent(amax_f)
    with np.errstate(invalid="ignore", over="ignore"):
        v = blocks * pow2(-e)[:, :, None]         # exact: scaling by a power of two
        q = e4m3_encode(v)
    q = np.where(bad[:, :, None], np.uint8(0x7F), q)
    s = np.where(bad, 0xFF, e + E8M0_BIAS).astype(np.uint8)
    return q.reshape(rows, n).astype(np.uint8), s


def quantize_rowwise(x_bits):
    """Row-wise MXFP8: blocks of 32 along each row.  -> (q [R,C], s [R,C/32])."""
    return quantize_mx(x_bits, axis=1)


def quantize_colwise(x_bits):
    """Column-wise MXFP8: blocks of 32 down each column, stored transposed.

    -> (q [C,R], s [C,R/32]); row c of q is column c of X, so the copy is
    K-contiguous when X's rows are the K axis of a later GEMM (the wgrad
    operand).
    """
    return quantize_mx(x_bits, axis=0)


def block_scale_exponent(amax) -> np.ndarray:
    """Float8BlockScaling scale cast to E8M0: e = ceil(log2(amax / 448)), found
    exactly as the smallest integer e with amax <= 448 * 2^e; clamped to
    [-127, 127]; amax == 0 gives -127."""
    amax = np.asarray(amax, dtype=np.float64)
    e = floor_log2(amax) - E4M3_EMAX                 # first guess: 448 * 2^e may be below amax
    e = np.where(amax > E4M3_MAX * pow2(np.clip(e, -1000, 1000)), e + 1, e)
    e = np.clip(e, -E8M0_BIAS, E8M0_BIAS)
    return np.where(amax == 0.0, -E8M0_BIAS, e).astype(np.int64)


def quantize_block(x_bits, block_2d: bool):
    """Float8BlockScaling quantisation, E8M0-cast scales, in the MX layout.

    ``block_2d`` False: 1x128 blocks along each row (row-wise copy) and 128x1
    blocks down each column (column-wise copy).  True: 128x128 blocks; both
    copies share each block's scale.  Blocks at the right and bottom edges may
    be partial: their amax is taken over the elements present.  A block holding
    NaN or inf gets scale byte 0xFF and every code 0x7F (the MX convention).
    Returns (q_row [R,C], s_row [R,ceil(C/32)], q_col [C,R], s_col
    [C,ceil(R/32)]): the scale of a 128-block is repeated for each of its
    32-element groups, so the MX GEMM of these operands is the block-scaled GEMM.
    """
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    rows, cols = x.shape
    pr, pc = -(-rows // 128) * 128, -(-cols // 128) * 128
    xp = np.zeros((pr, pc))                  # zero padding leaves every amax unchanged
    xp[:rows, :cols] = x
    ax = np.abs(xp)
    with np.errstate(invalid="ignore"):
        if block_2d:
            amax = ax.reshape(pr // 128, 128, pc // 128, 128).max(axis=(1, 3))   # [R/128, C/128]
            a_row = np.repeat(np.repeat(amax, 128, axis=0), 4, axis=1)           # [R, C/32]
            a_col = np.repeat(np.repeat(amax.T, 128, axis=0), 4, axis=1)         # [C, R/32]
        else:
            a_row = np.repeat(ax.reshape(pr, pc // 128, 128).max(axis=2), 4, axis=1)
            a_col = np.repeat(ax.T.reshape(pc, pr // 128, 128).max(axis=2), 4, axis=1)
    out = []
    for v, a in ((xp, a_row), (xp.T, a_col)):
        bad = ~np.isfinite(a)
        e = block_scale_exponent(np.where(bad, 0.0, a))
        with np.errstate(invalid="ignore", over="ignore"):
            q = e4m3_encode(v * pow2(-np.repeat(e, 32, axis=1))).astype(np.uint8)
        q[np.repeat(bad, 32, axis=1)] = 0x7F
        s = np.where(bad, 0xFF, e + E8M0_BIAS).astype(np.uint8)
        out.append((q, s))
    (q_row, s_row), (q_col, s_col) = out
    gr, gc = -(-rows // 32), -(-cols // 32)
    return q_row[:rows, :cols], s_row[:rows, :gc], q_col[:cols, :rows], s_col[:cols, :gr]


FP32_MAX = float(np.finfo(np.float32).max)
BLOCK_EDGE = 128           # Float8BlockScaling block: 1x128, 128x1 or 128x128 elements


def block_scale_fp32(amax):
    """Float8BlockScaling with the FP32 scales kept (the README's second mode,
    "compute the GEMM with the FP32 scales directly").  Per block:
      s = fl32(amax / 448)       the FP32 scale (the dequantisation factor),
      r = fl32(1 / s)            the quantisation multiplier, at most the
                                 largest finite fp32,
    each an IEEE fp32 operation rounded to nearest even.  amax == 0 gives
    s = r = 1; a non-finite amax gives s = r = NaN (codes 0x7F).
    Returns (s, r) as float32 arrays."""
    a = np.asarray(amax, dtype=np.float32)           # exact: amax is a bf16 value
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        s = a / np.float32(E4M3_MAX)
        r = np.minimum(np.float32(1.0) / s, np.float32(FP32_MAX))
    one = np.float32(1.0)
    s = np.where(a == 0, one, s)
    r = np.where(a == 0, one, r)
    bad = ~np.isfinite(a)
    s = np.where(bad, np.float32(np.nan), s)
    r = np.where(bad, np.float32(np.nan), r)
    return s.astype(np.float32), r.astype(np.float32)


def quantize_block_fp32(x_bits, block_2d: bool):
    """Float8BlockScaling quantisation keeping FP32 scales.

    Blocks as in ``quantize_block`` (1x128 / 128x1, or 128x128 shared by both
    copies; partial edge blocks take the amax of the elements present).  Codes:
    q = E4M3_rn_satfinite(fl32(x * r)) with r from ``block_scale_fp32``
    (0x7F for a block holding NaN or inf).  Scales: one fp32 s per block and
    row of the copy, s_row [R, ceil(C/128)] and s_col [C, ceil(R/128)]; a
    128x128 block's scale is repeated over its 128 rows in both copies.
    Returns (q_row [R,C], s_row, q_col [C,R], s_col)."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    rows, cols = x.shape
    e = BLOCK_EDGE
    pr, pc = -(-rows // e) * e, -(-cols // e) * e
    xp = np.zeros((pr, pc))                  # zero padding leaves every amax unchanged
    xp[:rows, :cols] = x
    ax = np.abs(xp)
    with np.errstate(invalid="ignore"):
        if block_2d:
            amax = ax.reshape(pr // e, e, pc // e, e).max(axis=(1, 3))
            a_row = np.repeat(amax, e, axis=0)               # [R, C/128]
            a_col = np.repeat(amax.T, e, axis=0)             # [C, R/128]
        else:
            a_row = ax.reshape(pr, pc // e, e).max(axis=2)
            a_col = ax.T.reshape(pc, pr // e, e).max(axis=2)
    out = []
    for v, a in ((xp, a_row), (xp.T, a_col)):
        sc, r = block_scale_fp32(a)
        bad = ~np.isfinite(a)
        with np.errstate(invalid="ignore", over="ignore"):
            prod = v.astype(np.float32) * np.repeat(r, e, axis=1)      # fl32(x * r)
            q = e4m3_encode(prod.astype(np.float64)).astype(np.uint8)
        q[np.repeat(bad, e, axis=1)] = 0x7F
        out.append((q, sc))
    (q_row, s_row), (q_col, s_col) = out
    gr, gc = -(-rows // e), -(-cols // e)
    return q_row[:rows, :cols], s_row[:rows, :gc], q_col[:cols, :rows], s_col[:cols, :gr]


def dequantize_fp32(q, s) -> np.ndarray:
    """E4M3 bytes [R, C] with fp32 scales [R, >= ceil(C/128)] (one per row and
    128 columns) -> float64 [R, C], exactly (a 4-bit by 24-bit product)."""
    q = np.asarray(q, dtype=np.uint8)
    rows, n = q.shape
    sc = np.asarray(s, dtype=np.float32).astype(np.float64)[:, :-(-n // BLOCK_EDGE)]
    return e4m3_decode(q) * np.repeat(sc, BLOCK_EDGE, axis=1)[:, :n]


def dequantize(q, s) -> np.ndarray:
    """E4M3 bytes [R, C] with E8M0 bytes [R, C/32] -> float64 [R, C] (exact)."""
    q = np.asarray(q, dtype=np.uint8)
    s = np.asarray(s, dtype=np.uint8).astype(np.int64)
    rows, n = q.shape
    vals = e4m3_decode(q).reshape(rows, n // MX_BLOCK, MX_BLOCK)
    scale = np.where(s == 0xFF, np.nan, pow2(s - E8M0_BIAS))
    return (vals * scale[:, :, None]).reshape(rows, n)


# --------------------------------------------------------------------------
# MXFP8 GEMM and epilogues
# --------------------------------------------------------------------------


def gelu_tanh(x) -> np.ndarray:
    """GELU, tanh approximation: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def dgelu_tanh(x) -> np.ndarray:
    """d/dx of gelu_tanh: 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) u',
    u = sqrt(2/pi) (x + 0.044715 x^3), u' = sqrt(2/pi) (1 + 3 * 0.044715 x^2).

    Evaluated through the exact identities 0.5 (1 + tanh u) = 1 / (1 + E) and
    1 - tanh^2 u = 4 E / (1 + E)^2 with E = exp(-2u): the same function, but
    1 + tanh u does not cancel for u << 0 (where the derivative is ~1e-15 and
    the tanh form loses every digit in fp64)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.sqrt(2.0 / np.pi)
    u = c * (x + 0.044715 * x ** 3)
    with np.errstate(over="ignore"):
        big = np.exp(-2.0 * u)                       # E (inf for u << 0)
    s = 1.0 / (1.0 + big)                            # 0.5 (1 + tanh u)
    with np.errstate(invalid="ignore"):
        one_minus_t2 = np.where(np.isinf(big), 0.0, 4.0 * big * s * s)   # 1 - tanh^2 u
    return s + 0.5 * x * one_minus_t2 * c * (1.0 + 3.0 * 0.044715 * x ** 2)


def mx_gemm_dgelu(qa, sa, qb, sb, aux_bits):
    """MXFP8 TN GEMM with the dGELU epilogue: D = bf16(acc * dgelu_tanh(aux)),
    acc = deq(A) . deq(B)^T, aux the bf16 pre-activation saved by the forward
    GEMM (an input here).  Returns dict with d, ref (unrounded), sigma (scaled by
    |dgelu(aux)|, the error scale of the bound)."""
    a = dequantize(qa, sa)
    b = dequantize(qb, sb)
    g = dgelu_tanh(bf16_bits_to_f64(aux_bits))
    acc = a @ b.T
    sigma = (np.abs(a) @ np.abs(b).T) * np.abs(g)
    ref = acc * g
    return {"pre": ref, "d": bf16_round(ref), "sigma": sigma}


def column_sums(x_bits):
    """Bias gradient: sum over rows of a bf16 matrix (fp64, exact for the
    sizes here).  Returns (sums, sum of |x| per column)."""
    x = bf16_bits_to_f64(x_bits)
    return x.sum(axis=0), np.abs(x).sum(axis=0)


def mx_gemm(qa, sa, qb, sb, bias_bits=None, gelu: bool = False):
    """MXFP8 TN GEMM: pre = deq(A) . deq(B)^T (+ bias), then the epilogue.

    qa [M,K], sa [M,K/32]; qb [N,K], sb [N,K/32] (both K-contiguous);
    bias_bits: bf16 patterns [N] or None.

    Returns a dict of float64 arrays:
      pre   exact pre-activation (fp64 matmul of the exact dequantised operands)
      d     bf16(pre), or bf16(gelu_tanh(pre)) when ``gelu``
      aux   bf16(pre) when ``gelu``, else None
      sigma sum_k |a_k b_k| (the error scale of the acceptance bound)
    """
    a = dequantize(qa, sa)
    b = dequantize(qb, sb)
    pre = a @ b.T
    if bias_bits is not None:
        pre = pre + bf16_bits_to_f64(bias_bits)[None, :]
    sigma = np.abs(a) @ np.abs(b).T
    if gelu:
        return {"pre": pre, "d": bf16_round(gelu_tanh(pre)), "aux": bf16_round(pre), "sigma": sigma}
    return {"pre": pre, "d": bf16_round(pre), "aux": None, "sigma": sigma}


def block_gemm_fp32(qa, sa, qb, sb, bias_bits=None, gelu: bool = False):
    """Float8BlockScaling TN GEMM with the FP32 scales applied directly:
    pre = deq(A) . deq(B)^T (+ bias), deq = code * its block's fp32 scale
    (``dequantize_fp32``; the K blocks are 128 long), then the epilogue as in
    ``mx_gemm``.  Returns the same dict."""
    a = dequantize_fp32(qa, sa)
    b = dequantize_fp32(qb, sb)
    pre = a @ b.T
    if bias_bits is not None:
        pre = pre + bf16_bits_to_f64(bias_bits)[None, :]
    sigma = np.abs(a) @ np.abs(b).T
    if gelu:
        return {"pre": pre, "d": bf16_round(gelu_tanh(pre)), "aux": bf16_round(pre), "sigma": sigma}
    return {"pre": pre, "d": bf16_round(pre), "aux": None, "sigma": sigma}


def mx_grouped_gemm(qx, sx, group_m, qw, sw, bias_bits=None, gelu: bool = False):
    """Grouped MXFP8 GEMM (MoE experts): for each group g with m_g > 0,
    D[rows of g] = epilogue(X_g . W_g^T (+ bias_g)).

    qx [sum m, K], sx [sum m, K/32] hold the groups' rows back to back in group
    order; qw [G, N, K], sw [G, N, K/32]; bias_bits [G, N] or None.  Empty
    groups contribute nothing.  Returns dict of float64 [sum m, N] arrays as
    ``mx_gemm`` does (aux None without gelu).
    """
    group_m = [int(m) for m in group_m]
    total = sum(group_m)
    n = qw.shape[1]
    out = {"pre": np.zeros((total, n)), "d": np.zeros((total, n)),
           "aux": np.zeros((total, n)) if gelu else None, "sigma": np.zeros((total, n))}
    row = 0
    for g, m in enumerate(group_m):
        if m == 0:
            continue
        bias = None if bias_bits is None else bias_bits[g]
        r = mx_gemm(qx[row:row + m], sx[row:row + m], qw[g], sw[g], bias, gelu)
        for key in ("pre", "d", "sigma"):
            out[key][row:row + m] = r[key]
        if gelu:
            out["aux"][row:row + m] = r["aux"]
        row += m
    return out


# --------------------------------------------------------------------------
# Acceptance bound
# --------------------------------------------------------------------------

REL_TOL = 2.0 ** -7
SIGMA_TOL = 1e-5


def gemm_error_bound(ref, sigma) -> np.ndarray:
    """Per-element bound |gpu - ref| <= 2^-7 |ref| + 1e-5 sum_k |a_k b_k|."""
    return REL_TOL * np.abs(ref) + SIGMA_TOL * np.asarray(sigma)


# --------------------------------------------------------------------------
# LayerNorm -> MXFP8 (the input quantisation of LayerNormLinear / LayerNormMLP)
# --------------------------------------------------------------------------
#
# LayerNorm as named on the TE pages: te.LayerNorm is a drop-in replacement of
# torch.nn.LayerNorm (leeroopedia "FP8 Training Quickstart", step on module
# replacement), with parameters 'scale' (gamma) and 'bias' (beta) and epsilon
# 1e-5 (TE "Getting Started" JAX page, layer configuration); LayerNormLinear /
# LayerNormDenseGeneral / LayerNormMLP fuse it with the Linear that consumes
# its output.  Over each row (the hidden axis):
#   mu = mean(x),  var = mean((x - mu)^2)  (biased),  rsigma = 1/sqrt(var + eps)
#   y  = (x - mu) * rsigma * gamma + beta.
# Reading: the fused quantiser takes y itself (no bf16 rounding between the
# norm and the quantiser) and MXFP8-quantises it with the rule above.

LAYERNORM_EPS = 1e-5


def layernorm(x_bits, gamma_bits, beta_bits, eps: float = LAYERNORM_EPS):
    """fp64 LayerNorm of a bf16 matrix [R, H] over each row.
    Returns (y [R, H], mu [R], rsigma [R])."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    g = bf16_bits_to_f64(np.asarray(gamma_bits, dtype=np.uint16))
    b = bf16_bits_to_f64(np.asarray(beta_bits, dtype=np.uint16))
    with np.errstate(invalid="ignore", over="ignore"):
        mu = x.mean(axis=1)
        var = ((x - mu[:, None]) ** 2).mean(axis=1)
        rsigma = 1.0 / np.sqrt(var + eps)
        y = (x - mu[:, None]) * rsigma[:, None] * g[None, :] + b[None, :]
    return y, mu, rsigma


FP32_U = 2.0 ** -24        # unit roundoff of fp32
LN_SUM_DEPTH = 64          # longest chain of fp32 additions in any row sum of the GPU


def layernorm_stat_bounds(x_bits, eps: float = LAYERNORM_EPS, depth: int = LN_SUM_DEPTH):
    """Bounds on the fp32 statistics of a row (the evaluation described under
    ``layernorm_error_bound``): |mu_fp32 - mu| <= dmu and
    |rsigma_fp32 - rsigma| <= rho * rsigma.  Returns (dmu [R], rho [R])."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    u = FP32_U
    with np.errstate(invalid="ignore", over="ignore"):
        mean_abs = np.abs(x).mean(axis=1)
        mu = x.mean(axis=1)
        var = ((x - mu[:, None]) ** 2).mean(axis=1)
        dmu = (depth + 1) * u * mean_abs                                  # sum error + the division
        rho = 0.5 * ((depth + 5) * u + dmu ** 2 / (var + eps)) + 2 * u    # var, +eps, sqrt, reciprocal
    return dmu, rho


def layernorm_error_bound(x_bits, gamma_bits, eps: float = LAYERNORM_EPS, depth: int = LN_SUM_DEPTH):
    """Per-element bound E on |y_fp32 - y| for a LayerNorm evaluated in fp32 as:
    mu = fl(S / H), S = sum of x with at most ``depth`` additions on any path;
    var = fl(S2 / H), S2 = sum of the squares of fl(x - mu), same depth, each
    square rounded on its own or fused into the addition that accumulates it
    (one rounding fewer, inside the same bound); rsigma =
    fl(1 / fl(sqrt(fl(var + eps)))); y = fl(fl(fl(x - mu) * rsigma) * gamma +
    beta) with one rounding (fused multiply-add).  Standard forward error
    analysis (each fl() a relative error of at most u = 2^-24, a sum of depth d
    at most d u sum|terms|), first-order terms times 1.05 for the rest."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    g = np.abs(bf16_bits_to_f64(np.asarray(gamma_bits, dtype=np.uint16)))
    u = FP32_U
    dmu, rho = layernorm_stat_bounds(x_bits, eps, depth)
    with np.errstate(invalid="ignore", over="ignore"):
        mu = x.mean(axis=1)
        var = ((x - mu[:, None]) ** 2).mean(axis=1)
        r = 1.0 / np.sqrt(var + eps)
        y_abs = np.abs((x - mu[:, None]) * r[:, None]) * g[None, :]
        e = (g[None, :] * r[:, None] * (dmu[:, None] * (1 + rho[:, None] + 2 * u)
                                        + np.abs(x - mu[:, None]) * (rho[:, None] + 2 * u)))
        return 1.05 * (e + u * (y_abs + np.abs(e)))


def mx_admissible(y, err, q, s, axis: int):
    """Is (q, s) the MX quantisation (``quantize_mx_values``) of some y' with
    |y' - y| <= err element-wise?  The test for a quantiser whose input is
    computed in a lower precision than the oracle's.

    ``y``, ``err``: float64 [R, C]; (q, s) laid out as ``quantize_mx_values``
    returns them for ``axis``.  Returns (ok, ambiguous), boolean arrays shaped
    like q: ``ok`` that the code and its block's scale are admissible,
    ``ambiguous`` that more than one (scale, code) is admissible there (outside
    these, ``ok`` means the answer equals the unique one).
    """
    y = np.asarray(y, dtype=np.float64)
    err = np.broadcast_to(np.asarray(err, dtype=np.float64), y.shape)
    if axis == 0:
        y, err = y.T, err.T
    rows, n = y.shape
    nb = n // MX_BLOCK
    yb = y.reshape(rows, nb, MX_BLOCK)
    eb = err.reshape(rows, nb, MX_BLOCK)
    q = np.asarray(q, dtype=np.uint8).reshape(rows, nb, MX_BLOCK)
    s = np.asarray(s, dtype=np.uint8)[:, :nb].astype(np.int64)
    with np.errstate(invalid="ignore", over="ignore"):
        bad = ~np.isfinite(np.max(np.abs(yb) + eb, axis=2))
        a_lo = np.max(np.maximum(np.abs(yb) - eb, 0.0), axis=2)
        a_hi = np.max(np.abs(yb) + eb, axis=2)
        e_lo = mx_scale_exponent(np.where(bad, 1.0, a_lo))
        e_hi = mx_scale_exponent(np.where(bad, 1.0, a_hi))
        e = s - E8M0_BIAS
        scale_ok = np.where(bad, s == 0xFF, (e >= e_lo) & (e <= e_hi))
        e_use = np.where(bad | ~scale_ok, 0, e)[:, :, None]
        v_lo = (yb - eb) * pow2(-e_use)
        v_hi = (yb + eb) * pow2(-e_use)
        c_lo = e4m3_decode(e4m3_encode(np.where(bad[:, :, None], 0.0, v_lo)))
        c_hi = e4m3_decode(e4m3_encode(np.where(bad[:, :, None], 0.0, v_hi)))
        got = e4m3_decode(q)
        sign_ok = np.where(v_lo > 0, (q & 0x80) == 0, np.where(v_hi < 0, (q & 0x80) != 0, True))
        code_ok = (got >= c_lo) & (got <= c_hi) & sign_ok
    code_ok = np.where(bad[:, :, None], q == 0x7F, code_ok)
    ok = code_ok & np.broadcast_to(scale_ok[:, :, None], code_ok.shape)
    amb = (c_lo != c_hi) | np.broadcast_to((e_lo != e_hi)[:, :, None], code_ok.shape)
    amb = amb & ~bad[:, :, None]
    return ok.reshape(rows, n), amb.reshape(rows, n)


# --------------------------------------------------------------------------
# Grouped wgrad for MoE experts (the second expert GEMM of training)
# --------------------------------------------------------------------------
#
# Expert e owns rows [R_e, R_e + m_e) of the token-major activations X and of
# the output gradient dY (ROCm/TransformerEngine README, "Single-Launch Grouped
# GEMM Backends on ROCm": one launch over the experts of a MoE layer).  Its weight gradient
# is dW_e = dY_e^T X_e, a TN GEMM whose reduction axis is the expert's tokens,
# so both operands are column-wise MXFP8 copies of dY_e and X_e, blocked
# along tokens.  Blocks must not cross an expert boundary, so each expert's
# tokens are zero-padded to Kp_e = round_up(m_e, 128) (128 tokens = one K-step
# of the GEMM).  Layout (reading: any layout that keeps experts apart works;
# this one keeps each expert's operand a strided slice of one array):
#   codes : q[c][P_e + t],  P_e = sum_{e' < e} Kp_e'          (t < Kp_e)
#   scales: s[c][Q_e + b],  Q_e = sum_{e' < e} round_up(Kp_e' / 32, 16)   (b < Kp_e / 32)
# (scale rows start on 16-byte boundaries, the alignment of a tensor copy).
# Padding tokens are zeros: their blocks get scale 0x00 and code 0.

WGRAD_PAD = 128


def grouped_layout(group_m, pad: int = WGRAD_PAD):
    """(Kp [G], P [G], Q [G], total codes width, total scale width)."""
    m = np.asarray(group_m, dtype=np.int64)
    kp = -(-m // pad) * pad
    P = np.concatenate([[0], np.cumsum(kp)[:-1]]) if len(m) else np.zeros(0, np.int64)
    sw = -(-(kp // MX_BLOCK) // 16) * 16
    Q = np.concatenate([[0], np.cumsum(sw)[:-1]]) if len(m) else np.zeros(0, np.int64)
    return kp, P.astype(np.int64), Q.astype(np.int64), int(kp.sum()), int(sw.sum())


def quantize_colwise_grouped(x_bits, group_m, pad: int = WGRAD_PAD):
    """Per-expert column-wise MXFP8 of the token-major matrix x [T, C] (bf16
    bits), each expert zero-padded to Kp_e tokens.  Returns (q [C, TP], s [C,
    TS]) in the layout above; scale bytes between Kp_e / 32 and the next
    16-byte boundary are 0 here (they are never read)."""
    x = np.asarray(x_bits, dtype=np.uint16)
    cols = x.shape[1]
    kp, P, Q, tp, ts = grouped_layout(group_m, pad)
    q = np.zeros((cols, tp), np.uint8)
    s = np.zeros((cols, ts), np.uint8)
    r = 0
    for e, m in enumerate(int(v) for v in group_m):
        if kp[e] == 0:
            continue
        xe = np.zeros((kp[e], cols), np.uint16)               # bf16 +0 padding
        xe[:m] = x[r:r + m]
        qe, se = quantize_colwise(xe)
        q[:, P[e]:P[e] + kp[e]] = qe
        s[:, Q[e]:Q[e] + kp[e] // MX_BLOCK] = se
        r += m
    return q, s


def mx_grouped_wgrad(qa, sa, qb, sb, group_m, pad: int = WGRAD_PAD) -> dict:
    """dW_e = deq(A_e) deq(B_e)^T for every expert, A = the grouped column-wise
    copy of dY ([N, TP]), B that of X ([K, TP]).  Returns {"d": [G, N, K]
    (bf16-rounded), "pre": fp64, "sigma": [G, N, K]}; an expert without tokens
    gets zeros."""
    kp, P, Q, _, _ = grouped_layout(group_m, pad)
    G, n, k = len(kp), qa.shape[0], qb.shape[0]
    pre = np.zeros((G, n, k))
    sigma = np.zeros((G, n, k))
    for e in range(G):
        if kp[e] == 0:
            continue
        nb = kp[e] // MX_BLOCK
        r = mx_gemm(qa[:, P[e]:P[e] + kp[e]], sa[:, Q[e]:Q[e] + nb], qb[:, P[e]:P[e] + kp[e]], sb[:, Q[e]:Q[e] + nb])
        pre[e], sigma[e] = r["pre"], r["sigma"]
    return {"pre": pre, "d": bf16_round(pre), "sigma": sigma}
