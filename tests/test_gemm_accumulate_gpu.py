"""GPU parity of the accumulating fp32 epilogue (TE_MX_EPI_ACCUMULATE_F32 of
te_mx_gemm, and the accumulate flag of te_mx_grouped_gemm_wgrad): D (fp32) +=
deq(A) deq(B)^T.  Acceptance: |gpu - (D_in + pre)| <= 2^-7 |pre| + 1e-5 sum|a b|
+ 2^-23 |D_in + pre| (the GEMM bound plus the fp32 rounding of the sum), pre
the oracle's exact product.  Both GEMM paths (single CTA and CTA pairs),
repeated accumulation, a canary after D, and experts without tokens left
bit-identical."""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding
from oracle import mx_oracle as O
from tests import _util as U
from tests.test_gemm_gpu import rand_bits, upload

pytestmark = pytest.mark.gpu


def bound(pre, sigma, total):
    return O.gemm_error_bound(pre, sigma) + 2.0 ** -23 * np.abs(total)


def check(got, want, pre, sigma, what):
    err = np.abs(got - want)
    b = bound(pre, sigma, want)
    if not np.all(err <= b):
        i = tuple(np.argwhere(~(err <= b))[0])
        raise AssertionError(f"{what}: {int((~(err <= b)).sum())} outside; first {i}: gpu {got[i]} want {want[i]}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 272, 384), (4096, 512, 256)])
def test_dense_accumulate(M, N, K):
    qa, sa = O.quantize_rowwise(rand_bits((M, K), 50 + M, outlier_cols=[1]))
    qb, sb = O.quantize_rowwise(rand_bits((N, K), 51 + N, std=0.05))
    ref = O.mx_gemm(qa, sa, qb, sb)
    g = torch.Generator().manual_seed(52)
    d_in = (torch.randn(M, N, generator=g) * 3.0).float()
    buf = torch.full((M * N + 64,), -7.25, dtype=torch.float32, device="cuda")
    d = buf[:M * N].view(M, N)
    d.copy_(d_in.cuda())
    A, SA = upload(qa, sa)
    B, SB = upload(qb, sb)
    binding.gemm(A, SA, B, SB, accumulate=d)
    binding.te_mx_device_status()
    assert torch.all(buf[M * N:] == -7.25), "write past the end of D"
    want = d_in.double().numpy() + ref["pre"]
    check(d.double().cpu().numpy(), want, ref["pre"], ref["sigma"], "D")
    binding.gemm(A, SA, B, SB, accumulate=d)                   # twice: D_in + 2 pre
    binding.te_mx_device_status()
    want2 = d_in.double().numpy() + 2 * ref["pre"]
    check(d.double().cpu().numpy(), want2, 2 * ref["pre"], 2 * ref["sigma"] + np.abs(ref["pre"]) * 2.0 ** -22, "D twice")


def test_grouped_wgrad_accumulate():
    group_m = [0, 100, 300, 0, 129]
    M, N = 256, 384
    dy = rand_bits((sum(group_m), M), 60, std=0.5)
    x = rand_bits((sum(group_m), N), 61)
    qa, sa = O.quantize_colwise_grouped(dy, group_m)
    qb, sb = O.quantize_colwise_grouped(x, group_m)
    ref = O.mx_grouped_wgrad(qa, sa, qb, sb, group_m)
    total, G = sum(group_m), len(group_m)
    wq, ws = binding.te_mx_grouped_code_width(total, G), binding.te_mx_grouped_scale_width(total, G)

    def up(q, s, rows):
        qd = torch.zeros(rows, wq, dtype=torch.uint8)
        qd[:, :q.shape[1]] = torch.from_numpy(q)
        sd = torch.zeros(rows, ws, dtype=torch.uint8)
        sd[:, :s.shape[1]] = torch.from_numpy(s)
        return {"q": qd.cuda(), "s": sd.cuda()}
    g = torch.Generator().manual_seed(62)
    d_in = torch.randn(G, M, N, generator=g).float()
    d = d_in.cuda()
    gm = torch.tensor(group_m, dtype=torch.int32, device="cuda")
    binding.grouped_gemm_wgrad(gm, total, up(qa, sa, M), up(qb, sb, N), out=d, accumulate=True)
    binding.te_mx_device_status()
    got = d.double().cpu().numpy()
    for e, m in enumerate(group_m):
        if m == 0:
            assert torch.equal(d[e].cpu(), d_in[e]), f"expert {e} without tokens changed"
            continue
        want = d_in[e].double().numpy() + ref["pre"][e]
        check(got[e], want, ref["pre"][e], ref["sigma"][e], f"dW[{e}]")
