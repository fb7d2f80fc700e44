"""Seeded synthetic inputs for the FP8-Linear workloads (shared by tests, bench, smoke).

This module only draws random numbers: it holds none of the quantisation or
GEMM arithmetic.  Every tensor is drawn in fp32 on the CPU from its own
``torch.Generator`` seed, scaled, and rounded once to bf16 (the operands of an
FP8 Linear are bf16 before quantisation).

Workloads (shapes R x C are row-major; GEMMs are TN: D[M,N] = A[M,K] . B[N,K]^T):

* ``tiny``    A[256x256], B[256x256] N(0,1) and bias[256] N(0,1), all from one
              generator seeded 0 (drawn in that order).
* ``qkv``     GPT decoder QKV projection, batch 32 x seq 128 x hidden 1024:
              X[4096x1024] N(0,1), W[3072x1024] N(0,0.02^2), bias N(0,0.02^2).
* ``fc1``     LayerNormMLP FC1: X[4096x1024] N(0,1) with 1% of its K columns
              (10) scaled x64, W1[4096x1024] N(0,0.02^2), bias[4096]
              N(0,0.02^2), dY[4096x4096] N(0,1e-3^2) for the wgrad.
* ``ffn``     large dense FFN, 8192 tokens, hidden 7168, ffn 18432:
              X[8192x7168] N(0,1) with 0.5% of columns (36) scaled x32,
              W[18432x7168] N(0,0.01^2), bias N(0,0.01^2),
              dY[8192x18432] N(0,1e-4^2).
* ``moe``     16384 tokens routed top-8 over 128 experts; per-expert row
              counts from Zipf(1.1) popularity (4 experts forced empty),
              X[131072x4096] N(0,1) in expert-sorted order,
              W[128x1536x4096] N(0,0.02^2), no bias, GELU-tanh + AUX.

Seeds: workload index x 100 + tensor index (qkv 200.., fc1 300.., ffn 400..,
moe 500..).
"""
from __future__ import annotations

import math

import torch

_CHUNK_ELEMS = 1 << 24


def normal_bf16(shape, std: float, seed: int, mean: float = 0.0) -> torch.Tensor:
    """N(mean, std^2) drawn in fp32 from ``seed`` (in 16M-element chunks), rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    numel = math.prod(shape)
    out = torch.empty(numel, dtype=torch.bfloat16)
    for start in range(0, numel, _CHUNK_ELEMS):
        n = min(_CHUNK_ELEMS, numel - start)
        out[start:start + n] = (torch.randn(n, generator=g) * std + mean).to(torch.bfloat16)
    return out.view(*shape)


def normal_bf16_outlier_cols(rows: int, cols: int, std: float, frac: float,
                             factor: float, seed: int, col_seed: int):
    """N(0, std^2) with round(frac * cols) columns multiplied by ``factor`` in fp32.

    The outlier columns are ``randperm(cols)[:n]`` from ``col_seed``.  Returns
    (bf16 tensor, sorted outlier column indices).
    """
    n_out = round(frac * cols)
    cols_idx = torch.randperm(cols, generator=torch.Generator().manual_seed(col_seed))[:n_out]
    mult = torch.ones(cols)
    mult[cols_idx] = factor
    g = torch.Generator().manual_seed(seed)
    out = torch.empty(rows, cols, dtype=torch.bfloat16)
    step = max(1, _CHUNK_ELEMS // cols)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = (torch.randn(r1 - r0, cols, generator=g) * std * mult).to(torch.bfloat16)
    return out, torch.sort(cols_idx).values


def moe_group_sizes(tokens: int = 16384, experts: int = 128, top_k: int = 8,
                    zipf_s: float = 1.1, n_empty: int = 4, seed: int = 500) -> torch.Tensor:
    """Per-expert row counts for top-k routing with Zipf(s) expert popularity.

    Popularity p_r ~ r^-s over a seeded permutation of the experts; ``n_empty``
    seeded experts get p = 0.  Each token draws ``top_k`` distinct experts
    (sampling without replacement), so the counts sum to tokens * top_k and no
    expert can exceed ``tokens``.  Returns int32 [experts].
    """
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(experts, generator=g)
    p = torch.empty(experts, dtype=torch.float64)
    p[order] = torch.arange(1, experts + 1, dtype=torch.float64) ** (-zipf_s)
    p[torch.randperm(experts, generator=g)[:n_empty]] = 0.0
    picks = torch.multinomial(p.expand(tokens, experts), top_k, replacement=False, generator=g)
    counts = torch.bincount(picks.flatten(), minlength=experts).to(torch.int32)
    assert int(counts.sum()) == tokens * top_k
    return counts


# ---------------------------------------------------------------------------
# Workload registry
# ---------------------------------------------------------------------------

WORKLOADS = {
    "tiny": dict(M=256, N=256, K=256),
    "qkv": dict(M=4096, N=3072, K=1024, tokens=4096),
    "fc1": dict(M=4096, N=4096, K=1024, tokens=4096),
    "ffn": dict(M=8192, N=18432, K=7168, tokens=8192),
    "moe": dict(tokens=16384, experts=128, top_k=8, N=1536, K=4096),
}


def make_moe_wgrad():
    """Expert wgrad of the MoE layer: the routing and X of ``make_moe`` and an
    output gradient dY [sum m_e x 1536] N(0, 1e-3^2) (the gradient scale of the
    fc1 workload; the MoE workload names none)."""
    d = make_moe()
    total = int(d["group_m"].sum())
    return {"group_m": d["group_m"], "X": d["X"], "dY": normal_bf16((total, 1536), 1e-3, 503)}


def layernorm_params(hidden: int, seed: int):
    """LayerNorm scale (gamma) and bias (beta), bf16 [hidden]: N(1, 0.1^2) and
    N(0, 0.1^2) (trained-looking values instead of the 1 / 0 initialisation)."""
    return normal_bf16((hidden,), 0.1, seed, mean=1.0), normal_bf16((hidden,), 0.1, seed + 1)


def make_tiny():
    """A, B [256x256] and bias [256], N(0,1), one generator seeded 0."""
    g = torch.Generator().manual_seed(0)
    a = torch.randn(256, 256, generator=g).to(torch.bfloat16)
    b = torch.randn(256, 256, generator=g).to(torch.bfloat16)
    bias = torch.randn(256, generator=g).to(torch.bfloat16)
    return {"A": a, "B": b, "bias": bias}


def make_qkv():
    return {"X": normal_bf16((4096, 1024), 1.0, 200),
            "W": normal_bf16((3072, 1024), 0.02, 201),
            "bias": normal_bf16((3072,), 0.02, 202)}


def make_fc1():
    x, cols = normal_bf16_outlier_cols(4096, 1024, 1.0, 0.01, 64.0, 300, 304)
    return {"X": x, "outlier_cols": cols,
            "W": normal_bf16((4096, 1024), 0.02, 301),
            "bias": normal_bf16((4096,), 0.02, 302),
            "dY": normal_bf16((4096, 4096), 1e-3, 303)}


def make_ffn():
    x, cols = normal_bf16_outlier_cols(8192, 7168, 1.0, 0.005, 32.0, 400, 404)
    return {"X": x, "outlier_cols": cols,
            "W": normal_bf16((18432, 7168), 0.01, 401),
            "bias": normal_bf16((18432,), 0.01, 402),
            "dY": normal_bf16((8192, 18432), 1e-4, 403)}


def make_moe():
    counts = moe_group_sizes(seed=500)
    total = int(counts.sum())
    return {"group_m": counts,
            "X": normal_bf16((total, 4096), 1.0, 501),
            "W": normal_bf16((128, 1536, 4096), 0.02, 502)}


MAKERS = {"tiny": make_tiny, "qkv": make_qkv, "fc1": make_fc1, "ffn": make_ffn, "moe": make_moe}
