"""GPU parity of the grouped wgrad path (te_mx_quantize_colwise_grouped and
te_mx_grouped_gemm_wgrad) against the oracle.

* the per-expert column-wise quantiser bit-exactly (codes and real scale
  bytes), ragged / empty / tiny experts, canaries in every byte the layout
  does not own;
* the grouped wgrad GEMM on oracle-quantised operands within the GEMM bound
  (|gpu - oracle| <= 2^-7 |oracle| + 1e-5 sum |a b|), zeros for experts without
  tokens, M and N not multiples of the tile;
* both GPU stages together; device-side argument errors write nothing;
* the full-size MoE wgrad on sampled outputs (exact sums over whole experts).
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U
from tests.test_gemm_gpu import assert_within_bound, to_f64

pytestmark = pytest.mark.gpu


def rand_bf16(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


def gm_dev(group_m):
    return torch.tensor(group_m, dtype=torch.int32, device="cuda")


def gpu_grouped_colwise(x_cpu, group_m):
    total, cols = x_cpu.shape
    G = len(group_m)
    wq, ws = binding.te_mx_grouped_code_width(total, G), binding.te_mx_grouped_scale_width(total, G)
    out = {"q": torch.full((cols, wq), U.CANARY, dtype=torch.uint8, device="cuda"),
           "s": torch.full((cols, ws), U.CANARY, dtype=torch.uint8, device="cuda")}
    binding.quantize_colwise_grouped(x_cpu.cuda(), gm_dev(group_m), out=out)
    binding.te_mx_device_status()
    return out["q"].cpu().numpy(), out["s"].cpu().numpy()


def check_grouped_colwise(x_cpu, group_m):
    q, s = gpu_grouped_colwise(x_cpu, group_m)
    wq, ws = O.quantize_colwise_grouped(U.bf16_bits(x_cpu), group_m)
    kp, P, Q, tp, ts = O.grouped_layout(group_m)
    U.assert_bytes_equal(q[:, :tp], wq, "codes")
    assert np.all(q[:, tp:] == U.CANARY), "codes written past the layout"
    owned = np.zeros(s.shape[1], bool)
    for e in range(len(group_m)):
        owned[Q[e]:Q[e] + kp[e] // 32] = True
    U.assert_bytes_equal(s[:, owned], ws[:, owned[:ts]], "scales")
    assert np.all(s[:, ~owned] == U.CANARY), "scale bytes outside the experts' blocks were written"


@pytest.mark.parametrize("group_m,cols", [([100], 64), ([0, 5, 128, 300, 1], 96), ([31, 32, 33, 0, 0, 7], 256),
                                          ([1000, 0, 513, 64], 1024)])
def test_grouped_colwise_quantize(group_m, cols):
    check_grouped_colwise(rand_bf16(sum(group_m), cols, sum(group_m) + cols, std=2.0), group_m)


def test_grouped_colwise_many_experts_and_specials():
    rng = np.random.default_rng(3)
    group_m = rng.integers(0, 200, 70).tolist()
    x = rand_bf16(sum(group_m), 128, 9)
    x[5, 3] = float("nan")
    x[17, :] = 0.0
    check_grouped_colwise(x, group_m)


def run_wgrad(qa, sa, qb, sb, group_m, M, N):
    """Upload oracle operands (pitches = the host bounds) and run the GEMM."""
    total, G = sum(group_m), len(group_m)
    wq, ws = binding.te_mx_grouped_code_width(total, G), binding.te_mx_grouped_scale_width(total, G)

    def up(q, s, rows):
        qd = torch.zeros(rows, wq, dtype=torch.uint8)
        qd[:, :q.shape[1]] = torch.from_numpy(q)
        sd = torch.full((rows, ws), 0xFF, dtype=torch.uint8)          # unused scale bytes: E8M0 NaN
        sd[:, :s.shape[1]] = torch.from_numpy(s)
        kp, P, Q, _, _ = O.grouped_layout(group_m)
        for e in range(G):                                           # gaps between experts' scales: NaN too
            sd[:, Q[e] + kp[e] // 32:(Q[e + 1] if e + 1 < G else ws)] = 0xFF
        return {"q": qd.cuda(), "s": sd.cuda()}
    dy, x = up(qa, sa, M), up(qb, sb, N)
    d, dbuf = U.guarded_bf16(G * M, N)
    binding.grouped_gemm_wgrad(gm_dev(group_m), total, dy, x, out=d.view(G, M, N))
    binding.te_mx_device_status()
    U.check_guard(dbuf, G * M * N)
    return to_f64(d).reshape(G, M, N)


@pytest.mark.parametrize("group_m,M,N", [([256], 256, 256), ([0, 100, 128, 300, 1], 256, 512),
                                         ([33, 0, 700], 320, 272), ([5, 9, 0, 2000, 64, 128], 512, 256)])
def test_grouped_wgrad_gemm(group_m, M, N):
    dy = U.bf16_bits(rand_bf16(sum(group_m), M, 11 + M, std=0.5))
    x = U.bf16_bits(rand_bf16(sum(group_m), N, 12 + N))
    qa, sa = O.quantize_colwise_grouped(dy, group_m)
    qb, sb = O.quantize_colwise_grouped(x, group_m)
    got = run_wgrad(qa, sa, qb, sb, group_m, M, N)
    ref = O.mx_grouped_wgrad(qa, sa, qb, sb, group_m)
    for e, m in enumerate(group_m):
        if m == 0:
            assert not got[e].any(), f"expert {e} without tokens is not zero"
        assert_within_bound(got[e], ref["d"][e], ref["sigma"][e], f"dW[{e}]")


def test_gpu_quantiser_feeds_gpu_wgrad():
    group_m = [77, 0, 300, 129]
    M, N = 256, 384
    dy_t, x_t = rand_bf16(sum(group_m), M, 21, std=0.3), rand_bf16(sum(group_m), N, 22)
    g = gm_dev(group_m)
    dy = binding.quantize_colwise_grouped(dy_t.cuda(), g)
    x = binding.quantize_colwise_grouped(x_t.cuda(), g)
    d = binding.grouped_gemm_wgrad(g, sum(group_m), dy, x)
    binding.te_mx_device_status()
    qa, sa = O.quantize_colwise_grouped(U.bf16_bits(dy_t), group_m)
    qb, sb = O.quantize_colwise_grouped(U.bf16_bits(x_t), group_m)
    ref = O.mx_grouped_wgrad(qa, sa, qb, sb, group_m)
    got = to_f64(d)
    for e in range(len(group_m)):
        assert_within_bound(got[e], ref["d"][e], ref["sigma"][e], f"dW[{e}]")


def test_device_side_errors_write_nothing():
    x = rand_bf16(200, 64, 5).cuda()
    for bad in ([50, -1, 10], [150, 100]):                       # a negative count; a sum above total_m
        g = gm_dev(bad)
        out = {"q": torch.full((64, 1024), 7, dtype=torch.uint8, device="cuda"),
               "s": torch.full((64, 64), 7, dtype=torch.uint8, device="cuda")}
        binding.quantize_colwise_grouped(x, g, out=out)
        with pytest.raises(binding.TemxError, match="INVALID_ARG"):
            binding.te_mx_device_status()
        assert torch.all(out["q"] == 7) and torch.all(out["s"] == 7)
    # a layout wider than the given pitch
    g = gm_dev([100, 100])
    out = {"q": torch.full((64, 128), 7, dtype=torch.uint8, device="cuda"),
           "s": torch.full((64, 16), 7, dtype=torch.uint8, device="cuda")}
    binding.quantize_colwise_grouped(x, g, out=out)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_device_status()
    assert torch.all(out["q"] == 7)
    dy = {"q": torch.zeros(256, 128, dtype=torch.uint8, device="cuda"),
          "s": torch.zeros(256, 16, dtype=torch.uint8, device="cuda")}
    xx = {"q": torch.zeros(256, 128, dtype=torch.uint8, device="cuda"),
          "s": torch.zeros(256, 16, dtype=torch.uint8, device="cuda")}
    d = torch.full((2, 256, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    binding.grouped_gemm_wgrad(g, 200, dy, xx, out=d)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_device_status()
    assert torch.all(d == 3.0)


def test_full_size_moe_wgrad_sampled():
    w = workloads.make_moe_wgrad()
    group_m = w["group_m"].tolist()
    g = w["group_m"].to(torch.int32).cuda()
    total = sum(group_m)
    dy = binding.quantize_colwise_grouped(w["dY"].cuda(), g)
    x = binding.quantize_colwise_grouped(w["X"].cuda(), g)
    d = binding.grouped_gemm_wgrad(g, total, dy, x)
    binding.te_mx_device_status()
    rng = np.random.default_rng(7)
    nz = [e for e, m in enumerate(group_m) if m > 0]
    experts = sorted({nz[0], max(nz, key=lambda e: group_m[e]), int(rng.choice(nz)), nz[-1]})
    experts += [e for e, m in enumerate(group_m) if m == 0][:1]
    starts = np.concatenate([[0], np.cumsum(group_m)])
    for e in experts:
        r0, m = starts[e], group_m[e]
        rows = np.sort(rng.choice(1536, 12, replace=False))
        cols = np.sort(rng.choice(4096, 12, replace=False))
        got = d[e].cpu()[torch.from_numpy(rows)][:, torch.from_numpy(cols)].double().numpy()
        if m == 0:
            assert not got.any()
            continue
        qa, sa = O.quantize_colwise(np.ascontiguousarray(
            np.pad(U.bf16_bits(w["dY"][r0:r0 + m][:, torch.from_numpy(rows)]), ((0, -m % 128), (0, 0)))))
        qb, sb = O.quantize_colwise(np.ascontiguousarray(
            np.pad(U.bf16_bits(w["X"][r0:r0 + m][:, torch.from_numpy(cols)]), ((0, -m % 128), (0, 0)))))
        # the GPU quantiser's own operands for these rows / columns, bit-exact
        kp, P, Q, _, _ = O.grouped_layout(group_m)
        U.assert_bytes_equal(dy["q"][torch.from_numpy(rows)][:, P[e]:P[e] + kp[e]].cpu().numpy(), qa, "dY codes")
        U.assert_bytes_equal(x["q"][torch.from_numpy(cols)][:, P[e]:P[e] + kp[e]].cpu().numpy(), qb, "X codes")
        ref = O.mx_gemm(qa, sa, qb, sb)
        assert_within_bound(got, ref["d"], ref["sigma"], f"dW[{e}] sampled")
