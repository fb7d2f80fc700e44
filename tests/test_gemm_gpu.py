"""GPU parity of te_mx_gemm / te_mx_grouped_gemm against the fp64 oracle.

Acceptance (element-wise, no exceptions): |gpu - oracle| <= 2^-7 |oracle| +
1e-5 sum_k |a_k b_k|, oracle = the epilogue of the fp64 product of the same
dequantised operands (rounded to bf16).  Operands for the small cases are
quantised by the oracle and uploaded, so these tests do not depend on the GPU
quantiser; the full-size cases run the GPU quantiser, check every byte of
the operand used in full and the sampled rows of the other bit-exactly, and
check one row in every 256-row band of the output.  Scale-pitch padding is filled with 0xFF (an E8M0
NaN) to prove it is never used, and every output has a canary tail.
"""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding, workloads
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu


def rand_bits(shape, seed, std=1.0, outlier_cols=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * std
    if outlier_cols is not None:
        x[..., outlier_cols] *= 64.0
    return U.bf16_bits(x.to(torch.bfloat16))


def upload(q, s):
    """Oracle codes/scales -> device tensors; scale padding = 0xFF."""
    pitch = binding.te_mx_scale_pitch(q.shape[1])
    sp = np.full((q.shape[0], pitch), 0xFF, np.uint8)
    sp[:, : s.shape[1]] = s
    return torch.from_numpy(q).cuda(), torch.from_numpy(sp).cuda()


def run_gemm(qa, sa, qb, sb, bias_bits=None, gelu=False):
    M, N = qa.shape[0], qb.shape[0]
    d, dbuf = U.guarded_bf16(M, N)
    aux, abuf = U.guarded_bf16(M, N) if gelu else (None, None)
    bias = U.from_bits(bias_bits).cuda() if bias_bits is not None else None
    binding.gemm(qa, sa, qb, sb, bias=bias, gelu=gelu, out=(d, aux))
    binding.te_mx_device_status()
    U.check_guard(dbuf, M * N)
    if gelu:
        U.check_guard(abuf, M * N)
    return d, aux


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def assert_within_bound(got, ref, sigma, what):
    err = np.abs(got - ref)
    bound = O.gemm_error_bound(ref, sigma)
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the bound; first {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r} bound {bound[i]!r}")


def check_dense(M, N, K, bias, gelu, seed, b_std=0.05):
    a_bits = rand_bits((M, K), seed, outlier_cols=[3, K // 2])
    b_bits = rand_bits((N, K), seed + 1, std=b_std)
    qa, sa = O.quantize_rowwise(a_bits)
    qb, sb = O.quantize_rowwise(b_bits)
    bias_bits = rand_bits((N,), seed + 2, std=0.5) if bias else None
    d, aux = run_gemm(*upload(qa, sa), *upload(qb, sb), bias_bits, gelu)
    ref = O.mx_gemm(qa, sa, qb, sb, bias_bits, gelu)
    assert_within_bound(to_f64(d), ref["d"], ref["sigma"], "D")
    if gelu:
        assert_within_bound(to_f64(aux), ref["aux"], ref["sigma"], "AUX")


@pytest.mark.parametrize("m,k", [(128, 256), (200, 640)])
def test_identity_b_is_bit_exact(m, k):
    # B = I: every B block is one 1.0 -> D must equal the dequantised A exactly
    qa, sa = O.quantize_rowwise(rand_bits((m, k), 40, std=3.0))
    qb, sb = O.quantize_rowwise(O.f64_to_bf16_bits(np.eye(k)))
    d, _ = run_gemm(*upload(qa, sa), *upload(qb, sb))
    want = O.dequantize(qa, sa)
    got = to_f64(d)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} mismatches, first {i}: gpu {got[i]} want {want[i]}")


def test_single_nonzero_block_scales():
    # one nonzero K-block per row of A with distinct scales: checks that each
    # row and each K-block reads its own scale byte
    m, n, k = 128, 256, 512
    a = np.zeros((m, k))
    rng = np.random.default_rng(1)
    for r in range(m):
        blk = r % (k // 32)
        a[r, 32 * blk:32 * blk + 32] = rng.standard_normal(32) * 2.0 ** (r % 17 - 8)
    b = rng.standard_normal((n, k)) * 2.0 ** (np.arange(n) % 13 - 6)[:, None]
    qa, sa = O.quantize_rowwise(O.f64_to_bf16_bits(a))
    qb, sb = O.quantize_rowwise(O.f64_to_bf16_bits(b))
    d, _ = run_gemm(*upload(qa, sa), *upload(qb, sb))
    ref = O.mx_gemm(qa, sa, qb, sb)
    assert_within_bound(to_f64(d), ref["d"], ref["sigma"], "D")


@pytest.mark.parametrize("M,N,K,bias,gelu", [
    (128, 256, 128, False, False),
    (256, 256, 256, True, False),
    (200, 96, 384, False, True),
    (333, 528, 640, True, True),
    (1, 16, 128, True, False),
    (130, 272, 1024, False, False),
    (1024, 1024, 2048, True, True),
    (640, 3072, 1024, True, False),
])
def test_dense_vs_oracle(M, N, K, bias, gelu):
    check_dense(M, N, K, bias, gelu, seed=M + N + K)


# Shapes with M >= 256 run on CTA pairs (cta_group::2); the last two give
# every CTA pair several tiles.
@pytest.mark.parametrize("M,N,K,bias,gelu", [
    (2048, 2560, 256, True, True),
    (2000, 2624, 640, False, False),
    (2304, 2304, 384, True, False),
    (10240, 512, 256, True, True),
    (20480, 256, 128, True, False),
])
def test_dense_pair_tiles_vs_oracle(M, N, K, bias, gelu):
    check_dense(M, N, K, bias, gelu, seed=M + N + K + 1)


# K of 16 or more K-steps: two MMA issuers take alternate K-steps.  An odd
# number of K-steps (K = 17 x 128) makes the owner of a tile's first K-step
# alternate from tile to tile, so each issuer both waits for the other's first
# K-step and is waited for; the CTA pairs take several tiles each.
@pytest.mark.parametrize("M,N,K,bias,gelu", [
    (4096, 2048, 2176, True, True),
    (2304, 1280, 2048, False, False),
    (200, 528, 2176, True, False),
])
def test_dense_two_issuers_vs_oracle(M, N, K, bias, gelu):
    check_dense(M, N, K, bias, gelu, seed=M + N + K + 2)


def test_identity_b_pair_tiles_is_bit_exact():
    m, k = 2048, 2560
    qa, sa = O.quantize_rowwise(rand_bits((m, k), 41, std=3.0))
    qb, sb = O.quantize_rowwise(O.f64_to_bf16_bits(np.eye(k)))
    d, _ = run_gemm(*upload(qa, sa), *upload(qb, sb))
    want = O.dequantize(qa, sa)
    got = to_f64(d)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} mismatches, first {i}: gpu {got[i]} want {want[i]}")


def test_gelu_of_zero_and_of_bias():
    # A = 0: pre = bias, D = GELU(bias), AUX = bias; with no bias D = AUX = 0
    m, n, k = 128, 256, 256
    qa, sa = O.quantize_rowwise(np.zeros((m, k), np.uint16))
    qb, sb = O.quantize_rowwise(rand_bits((n, k), 50))
    bias_bits = rand_bits((n,), 51, std=2.0)
    d, aux = run_gemm(*upload(qa, sa), *upload(qb, sb), None, True)
    assert not to_f64(d).any() and not to_f64(aux).any()
    d, aux = run_gemm(*upload(qa, sa), *upload(qb, sb), bias_bits, True)
    ref = O.mx_gemm(qa, sa, qb, sb, bias_bits, True)
    assert np.array_equal(to_f64(aux), ref["aux"])
    assert np.all(np.abs(to_f64(d) - ref["d"]) <= 2.0 ** -7 * np.abs(ref["d"]))


def test_tiny_workload_end_to_end():
    d = workloads.make_tiny()
    a, b = d["A"].cuda(), d["B"].cuda()
    qa = binding.quantize(a, rowwise=True, colwise=True)
    qb = binding.quantize(b, rowwise=True, colwise=False)
    ra, rb = O.quantize_rowwise(U.bf16_bits(d["A"])), O.quantize_rowwise(U.bf16_bits(d["B"]))
    ca = O.quantize_colwise(U.bf16_bits(d["A"]))
    U.assert_bytes_equal(qa["q_row"].cpu().numpy(), ra[0], "A row codes")
    U.assert_bytes_equal(qa["s_row"].cpu().numpy()[:, :8], ra[1], "A row scales")
    U.assert_bytes_equal(qa["q_col"].cpu().numpy(), ca[0], "A col codes")
    U.assert_bytes_equal(qa["s_col"].cpu().numpy()[:, :8], ca[1], "A col scales")
    U.assert_bytes_equal(qb["q_row"].cpu().numpy(), rb[0], "B row codes")
    bias_bits = U.bf16_bits(d["bias"])
    out, _ = binding.gemm(qa["q_row"], qa["s_row"], qb["q_row"], qb["s_row"], bias=d["bias"].cuda())
    binding.te_mx_device_status()
    ref = O.mx_gemm(ra[0], ra[1], rb[0], rb[1], bias_bits)
    assert_within_bound(to_f64(out), ref["d"], ref["sigma"], "D")


# ---------------------------------------------------------------- grouped

def run_grouped(group_m, total_m, N, K, bias, gelu, seed):
    G = len(group_m)
    x_bits = rand_bits((total_m, K), seed)
    w_bits = rand_bits((G, N, K), seed + 1, std=0.05)
    qx, sx = O.quantize_rowwise(x_bits)
    qw, sw = O.quantize_rowwise(w_bits.reshape(G * N, K))
    bias_bits = rand_bits((G, N), seed + 2, std=0.5) if bias else None
    dqx, dsx = upload(qx, sx)
    dqw, dsw = upload(qw, sw)
    gm = torch.tensor(group_m, dtype=torch.int32, device="cuda")
    d, dbuf = U.guarded_bf16(total_m, N)
    aux, abuf = U.guarded_bf16(total_m, N) if gelu else (None, None)
    bias_t = U.from_bits(bias_bits).cuda() if bias else None
    binding.grouped_gemm(gm, dqx, dsx, dqw.view(G, N, K), dsw, bias=bias_t, gelu=gelu, out=(d, aux))
    return (qx, sx, qw.reshape(G, N, K), sw.reshape(G, N, -1), bias_bits), (d, dbuf, aux, abuf)


@pytest.mark.parametrize("group_m,N,K,bias,gelu", [
    ([0, 5, 130, 0, 256, 77], 160, 256, True, True),
    ([700, 0, 1, 513, 900, 0, 300], 256, 256, True, True),        # >= 2048 rows: CTA pairs
    ([300], 256, 512, False, False),
    ([700, 0, 513, 900, 300], 256, 2176, True, True),               # two MMA issuers, odd K-steps
    ([1, 0, 0, 129, 127, 128, 0, 2], 272, 384, True, False),
])
def test_grouped_vs_oracle(group_m, N, K, bias, gelu):
    used = sum(group_m)
    total_m = used + 40                                  # 40 spare rows stay untouched
    (qx, sx, qw, sw, bias_bits), (d, dbuf, aux, abuf) = run_grouped(group_m, total_m, N, K, bias, gelu, 7 * N + K)
    binding.te_mx_device_status()
    ref = O.mx_grouped_gemm(qx[:used], sx[:used], group_m, qw, sw, bias_bits, gelu)
    dd = to_f64(d)
    assert_within_bound(dd[:used], ref["d"], ref["sigma"], "D")
    canary = 0xA5A5
    assert np.all(U.bf16_bits(d[used:]) == canary), "rows past sum(m) were written"
    U.check_guard(dbuf, total_m * N)
    if gelu:
        assert_within_bound(to_f64(aux)[:used], ref["aux"], ref["sigma"], "AUX")
        assert np.all(U.bf16_bits(aux[used:]) == canary)


def test_grouped_all_empty():
    (_, _, _, _, _), (d, dbuf, _, _) = run_grouped([0, 0, 0], 64, 128, 128, False, False, 3)
    binding.te_mx_device_status()
    assert np.all(U.bf16_bits(d) == 0xA5A5)


def test_grouped_sizes_beyond_total_are_reported_and_clamped():
    (_, _, _, _, _), (d, dbuf, _, _) = run_grouped([100, 100], 150, 128, 128, False, False, 5)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_device_status()
    U.check_guard(dbuf, 150 * 128)
    binding.te_mx_device_status()          # the status word was cleared


# ---------------------------------------------------------------- full-size workloads
#
# The GPU quantiser's operands are checked bit-exactly first, every byte of
# the operand that the oracle GEMM uses in full (B) and the sampled rows of A.
# The oracle GEMM then runs on the oracle's own codes, which those checks
# showed to be identical, so a quantiser error cannot hide inside the GEMM
# tolerance and no oracle input comes from the GPU.  Rows: one random row in
# every 256-row band (the row extent of a CTA-pair tile) plus the edges, so
# every output tile row band of the persistent tile walk is checked, each
# sampled row across all N columns (every n-tile).


def check_sampled(d, aux, rows, qa_rows, sa_rows, qb, sb, bias_bits, gelu, what):
    ri = torch.from_numpy(rows).cuda()
    got_d = to_f64(d[ri])
    got_aux = to_f64(aux[ri]) if gelu else None
    from tests import _oracle_jobs as J
    pool = U.oracle_pool()
    step = 8
    futs = [(r0, pool.submit(J.gemm_rows, qa_rows[r0:r0 + step], sa_rows[r0:r0 + step], qb, sb, bias_bits, gelu))
            for r0 in range(0, len(rows), step)]
    for r0, f in futs:
        rd, raux, sigma = f.result()
        assert_within_bound(got_d[r0:r0 + step], rd, sigma, f"{what} D (rows {rows[r0]}..)")
        if gelu:
            assert_within_bound(got_aux[r0:r0 + step], raux, sigma, f"{what} AUX (rows {rows[r0]}..)")


def fprop_check(x_cpu, w_cpu, bias_cpu, gelu, seed, what):
    x, w = x_cpu.cuda(), w_cpu.cuda()
    qx = binding.quantize(x, rowwise=True)
    qw = binding.quantize(w, rowwise=True)
    d, aux = binding.gemm(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"],
                          bias=None if bias_cpu is None else bias_cpu.cuda(), gelu=gelu)
    binding.te_mx_device_status()
    rows = U.band_rows(x_cpu.shape[0], 256, seed, extra=(127, 128, 255, 256))
    qa, sa = U.check_rows_rowwise(qx["q_row"], qx["s_row"], x_cpu, rows, what + " X (sampled rows)")
    qb, sb = U.check_every_byte(qw, w_cpu, True, False, what + " W")["row"]
    check_sampled(d, aux, rows, qa, sa, qb, sb, None if bias_cpu is None else U.bf16_bits(bias_cpu), gelu, what)


def wgrad_check(dy_cpu, x_cpu, seed, what):
    # dW[N_out x K_in] = dY^T X over T tokens: A = colwise(dY) [N_out x T], B = colwise(X) [K_in x T]
    dy, x = dy_cpu.cuda(), x_cpu.cuda()
    qdy = binding.quantize(dy, rowwise=False, colwise=True)
    qx = binding.quantize(x, rowwise=False, colwise=True)
    dw, _ = binding.gemm(qdy["q_col"], qdy["s_col"], qx["q_col"], qx["s_col"])
    binding.te_mx_device_status()
    rows = U.band_rows(dy_cpu.shape[1], 256, seed, extra=(127, 128, 255, 256))
    qa, sa = U.check_cols_colwise(qdy["q_col"], qdy["s_col"], dy_cpu, rows, what + " dY (sampled columns)")
    qb, sb = U.check_every_byte(qx, x_cpu, False, True, what + " X")["col"]
    check_sampled(dw, None, rows, qa, sa, qb, sb, None, False, what)


def test_full_size_qkv():
    d = workloads.make_qkv()
    fprop_check(d["X"], d["W"], d["bias"], False, 1, "qkv fprop")


def test_full_size_fc1_fprop_and_wgrad():
    d = workloads.make_fc1()
    fprop_check(d["X"], d["W"], d["bias"], True, 2, "fc1 fprop")
    wgrad_check(d["dY"], d["X"], 3, "fc1 wgrad")


def test_full_size_ffn_fprop_and_wgrad():
    d = workloads.make_ffn()
    fprop_check(d["X"], d["W"], d["bias"], True, 4, "ffn fprop")
    wgrad_check(d["dY"], d["X"], 5, "ffn wgrad")


def test_full_size_moe_grouped():
    # the first and the last row of every non-empty expert (and one row in
    # every 256-row band of the concatenated rows), each against its expert's
    # weights; every code of X and W checked bit-exactly first
    from tests import _oracle_jobs as J
    d = U.moe_workload()
    counts = d["group_m"].numpy()
    G, N, K = 128, 1536, 4096
    x, w = d["X"].cuda(), d["W"].view(G * N, K).cuda()
    qx = binding.quantize(x, rowwise=True)
    qw = binding.quantize(w, rowwise=True)
    gm = d["group_m"].cuda()
    out, aux = binding.grouped_gemm(gm, qx["q_row"], qx["s_row"], qw["q_row"].view(G, N, K), qw["s_row"],
                                    gelu=True)
    binding.te_mx_device_status()
    del x, w
    qwo, swo = U.check_every_byte(qw, d["W"].view(G * N, K), True, False, "moe W")["row"]
    del qw
    starts = np.concatenate([[0], np.cumsum(counts)])
    total = int(starts[-1])
    ends = {int(starts[g + 1]) - 1 for g in range(G) if counts[g]}
    rows = U.band_rows(total, 256, 6, extra={int(starts[g]) for g in range(G) if counts[g]} | ends)
    qa, sa = U.check_rows_rowwise(qx["q_row"], qx["s_row"], d["X"], rows, "moe X (sampled rows)")
    got_d = to_f64(out[torch.from_numpy(rows).cuda()])
    got_aux = to_f64(aux[torch.from_numpy(rows).cuda()])
    group_of = np.searchsorted(starts, rows, side="right") - 1
    pool = U.oracle_pool()
    futs = []
    for g in np.unique(group_of):
        sel = np.nonzero(group_of == g)[0]
        wq, ws = qwo[g * N:(g + 1) * N], swo[g * N:(g + 1) * N]
        futs.append((g, sel, pool.submit(J.gemm_rows, qa[sel], sa[sel], wq, ws, None, True)))
    assert len(futs) == int((counts > 0).sum())
    for g, sel, f in futs:
        rd, raux, sigma = f.result()
        what = f"moe expert {g} (m={counts[g]}, rows {rows[sel][0]}..{rows[sel][-1]})"
        assert_within_bound(got_d[sel], rd, sigma, what + " D")
        assert_within_bound(got_aux[sel], raux, sigma, what + " AUX")


# ---------------------------------------------------------------- backward: dGELU epilogue, dgrad

@pytest.mark.parametrize("M,N,K", [(200, 96, 384), (333, 528, 640), (2048, 2560, 256)])
def test_dgelu_epilogue_vs_oracle(M, N, K):
    qa, sa = O.quantize_rowwise(rand_bits((M, K), M + 5))
    qb, sb = O.quantize_rowwise(rand_bits((N, K), N + 6, std=0.05))
    aux_bits = rand_bits((M, N), K + 7, std=2.0)
    aux_bits[:, :3] = O.f64_to_bf16_bits(np.array([-30.0, 0.0, 30.0]))       # saturated ends and 0
    aux = U.from_bits(aux_bits).cuda()
    d, dbuf = U.guarded_bf16(M, N)
    ga, gsa = upload(qa, sa)
    gb, gsb = upload(qb, sb)
    binding.gemm(ga, gsa, gb, gsb, out=(d, None), dgelu_aux=aux)
    binding.te_mx_device_status()
    U.check_guard(dbuf, M * N)
    ref = O.mx_gemm_dgelu(qa, sa, qb, sb, aux_bits)
    assert_within_bound(to_f64(d), ref["d"], ref["sigma"], "dGELU D")


def test_grouped_dgelu_vs_oracle():
    group_m, N, K = [0, 130, 1, 256, 77], 160, 256
    total = sum(group_m)
    G = len(group_m)
    qx, sx = O.quantize_rowwise(rand_bits((total, K), 61))
    qw, sw = O.quantize_rowwise(rand_bits((G * N, K), 62, std=0.05))
    aux_bits = rand_bits((total, N), 63, std=2.0)
    dqx, dsx = upload(qx, sx)
    dqw, dsw = upload(qw, sw)
    gm = torch.tensor(group_m, dtype=torch.int32, device="cuda")
    d, _ = binding.grouped_gemm(gm, dqx, dsx, dqw.view(G, N, K), dsw, dgelu_aux=U.from_bits(aux_bits).cuda())
    binding.te_mx_device_status()
    row = 0
    for g, m in enumerate(group_m):
        if m:
            ref = O.mx_gemm_dgelu(qx[row:row + m], sx[row:row + m], qw[g * N:(g + 1) * N], sw[g * N:(g + 1) * N],
                                  aux_bits[row:row + m])
            assert_within_bound(to_f64(d)[row:row + m], ref["d"], ref["sigma"], f"group {g}")
        row += m


def test_full_size_fc1_dgrad_on_colwise_weight():
    # dX[T x H] = dY[T x F] . W1[F x H]: A = row-wise dY (K = F), B = column-wise W1 = W1^T quantised along F
    d = workloads.make_fc1()
    dy, w = d["dY"].cuda(), d["W"].cuda()
    qdy = binding.quantize(dy, rowwise=True)
    qw = binding.quantize(w, rowwise=False, colwise=True)
    dx, _ = binding.gemm(qdy["q_row"], qdy["s_row"], qw["q_col"], qw["s_col"])
    binding.te_mx_device_status()
    rows = U.band_rows(d["dY"].shape[0], 256, 8)
    qa, sa = U.check_rows_rowwise(qdy["q_row"], qdy["s_row"], d["dY"], rows, "fc1 dY (sampled rows)")
    qb, sb = U.check_every_byte(qw, d["W"], False, True, "fc1 W1")["col"]
    check_sampled(dx, None, rows, qa, sa, qb, sb, None, False, "fc1 dgrad")
