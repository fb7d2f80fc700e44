"""GPU parity of te_mx_gemm_fp32_scales (the Float8BlockScaling GEMM with FP32
scales applied directly) against the oracle's ``block_gemm_fp32``, within the
GEMM acceptance bound, on operands quantised by te_mx_block_quantize_fp32
(checked bit-exact against the oracle first).

Covers 1Dx2D (weight blocks 128x128) and 1Dx1D scaling, the single-CTA and
CTA-pair tile paths, K with a partial last scale group, ragged M and N, every
epilogue (none, bias, GELU+AUX, bias+GELU+AUX, dGELU), block scales that differ
by orders of magnitude between K blocks, and the full-size ffn fprop (sampled).
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U
from tests.test_gemm_gpu import assert_within_bound, to_f64

pytestmark = pytest.mark.gpu


def randn_bf16(rows, cols, seed, std=1.0, block_spread=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * std
    if block_spread:     # K blocks of very different magnitude: exercises the per-block FP32 scales
        x = x * torch.exp2(torch.randint(-6, 7, (1, (cols + 127) // 128), generator=g).float()).repeat_interleave(128, 1)[:, :cols]
    return x.to(torch.bfloat16)


def quantize_checked(x_cpu, block_2d):
    q = binding.block_quantize_fp32(x_cpu.cuda(), block_2d=block_2d, rowwise=True, colwise=False)
    q_row, s_row, _, _ = O.quantize_block_fp32(U.bf16_bits(x_cpu), block_2d)
    U.assert_bytes_equal(q["q_row"].cpu().numpy(), q_row, "codes")
    n = s_row.shape[1]
    assert np.array_equal(q["s_row"][:, :n].cpu().numpy().view(np.uint32), s_row.view(np.uint32)), "scales"
    return q, (q_row, s_row)


def check(M, N, K, w_2d, epi, seed, spread=False):
    x = randn_bf16(M, K, seed, 1.0, block_spread=spread)
    w = randn_bf16(N, K, seed + 1, 0.05, block_spread=spread)
    qx, (oqx, osx) = quantize_checked(x, False)
    qw, (oqw, osw) = quantize_checked(w, w_2d)
    bias = aux_in = None
    if epi in ("bias", "bias_gelu"):
        bias = (torch.randn(N, generator=torch.Generator().manual_seed(seed + 2)) * 0.5).to(torch.bfloat16)
    if epi == "dgelu":
        aux_in = torch.randn(M, N, generator=torch.Generator().manual_seed(seed + 3)).to(torch.bfloat16)
    gelu = epi in ("gelu", "bias_gelu")
    d, aux = binding.gemm_fp32_scales(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], w_2d,
                                      bias=None if bias is None else bias.cuda(), gelu=gelu,
                                      dgelu_aux=None if aux_in is None else aux_in.cuda())
    binding.te_mx_device_status()
    ref = O.block_gemm_fp32(oqx, osx, oqw, osw, None if bias is None else U.bf16_bits(bias), gelu)
    if epi == "dgelu":
        g = O.dgelu_tanh(O.bf16_bits_to_f64(U.bf16_bits(aux_in)))
        assert_within_bound(to_f64(d), O.bf16_round(ref["pre"] * g), ref["sigma"] * np.abs(g), "dgelu D")
        return
    assert_within_bound(to_f64(d), ref["d"], ref["sigma"], "D")
    if gelu:
        assert_within_bound(to_f64(aux), ref["aux"], ref["sigma"], "AUX")


@pytest.mark.parametrize("w_2d", [True, False])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 256, 256), (384, 512, 640), (200, 272, 1024)])
def test_single_cta_tiles(M, N, K, w_2d):
    check(M, N, K, w_2d, "none", M + N + K + w_2d)


@pytest.mark.parametrize("w_2d", [True, False])
@pytest.mark.parametrize("M,N,K", [(2048, 2560, 1024), (1936, 2576, 640)])
def test_pair_tiles(M, N, K, w_2d):
    check(M, N, K, w_2d, "bias_gelu", M + N + K + 7 * w_2d)


@pytest.mark.parametrize("epi", ["bias", "gelu", "bias_gelu", "dgelu"])
def test_epilogues(epi):
    check(384, 512, 768, True, epi, 50 + len(epi))


@pytest.mark.parametrize("w_2d", [True, False])
def test_block_scales_spread_over_k(w_2d):
    check(512, 512, 1536, w_2d, "none", 60 + w_2d, spread=True)
    check(2048, 2560, 1024, w_2d, "none", 62 + w_2d, spread=True)


def test_full_size_ffn_fprop_sampled():
    d = workloads.make_ffn()
    x, w, b = d["X"], d["W"], d["bias"]
    qx = binding.block_quantize_fp32(x.cuda(), block_2d=False)
    qw = binding.block_quantize_fp32(w.cuda(), block_2d=True)
    dd, aux = binding.gemm_fp32_scales(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"], True, bias=b.cuda(),
                                       gelu=True)
    binding.te_mx_device_status()
    rng = np.random.default_rng(70)
    rows = np.sort(rng.choice(x.shape[0], 24, replace=False))
    ox = O.quantize_block_fp32(U.bf16_bits(x[rows]), False)     # 1D blocks: a row's scales are its own
    rt = torch.as_tensor(rows).cuda()
    for band in sorted(set(rng.choice(w.shape[0] // 128, 3, replace=False).tolist()) | {w.shape[0] // 128 - 1}):
        # a 128-row band of W holds whole 2D blocks
        kw = O.quantize_block_fp32(U.bf16_bits(w[128 * band:128 * band + 128]), True)
        loc = np.sort(rng.choice(128, 32, replace=False))
        cols = 128 * band + loc
        ref = O.block_gemm_fp32(ox[0], ox[1], kw[0][loc], kw[1][loc], U.bf16_bits(b)[cols], True)
        ct = torch.as_tensor(cols).cuda()
        assert_within_bound(to_f64(dd[rt][:, ct]), ref["d"], ref["sigma"], f"ffn D (sampled, band {band})")
        assert_within_bound(to_f64(aux[rt][:, ct]), ref["aux"], ref["sigma"], f"ffn AUX (sampled, band {band})")
