"""Oracle work items run in a spawn process pool by the full-size parity tests.

Imports numpy and the oracle only (no torch, no CUDA library), so the worker
processes start quickly and never touch the GPU.
"""
from oracle import mx_oracle as O


def quantize_rows(bits):
    """Row-wise MXFP8 of a slab of rows: (q, s)."""
    return O.quantize_rowwise(bits)


def quantize_cols(bits):
    """Column-wise MXFP8 of a slab of columns: (q, s) of the transposed copy."""
    return O.quantize_colwise(bits)


def gemm_rows(qa, sa, qb, sb, bias_bits, gelu):
    """Oracle GEMM of a few rows of A against all of B: (d, aux, sigma)."""
    r = O.mx_gemm(qa, sa, qb, sb, bias_bits, gelu)
    return r["d"], r["aux"], r["sigma"]
