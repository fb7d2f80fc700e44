"""Pins for the grouped-wgrad part of the oracle (per-expert column-wise
quantisation with zero-padded experts, and dW_e = dY_e^T X_e).

* the layout against hand-computed offsets;
* one expert alone equals quantize_colwise of the zero-padded matrix;
* per-block brute force on ragged experts (block amax and codes by loops);
* padding columns are zero codes with scale 0x00;
* dW_e equals an explicit sum over the expert's own (unpadded) tokens of
  outer products of dequantised values, written with loops;
* an expert without tokens gets zeros; a planted offset mistake is caught.
"""
import numpy as np
import pytest
import torch

from oracle import mx_oracle as O


def rand_bits(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_layout_by_hand():
    kp, P, Q, tp, ts = O.grouped_layout([0, 5, 128, 300, 1])
    assert kp.tolist() == [0, 128, 128, 384, 128]
    assert P.tolist() == [0, 0, 128, 256, 640]
    # scale widths 0, 4->16, 4->16, 12->16, 4->16
    assert Q.tolist() == [0, 0, 16, 32, 48]
    assert (tp, ts) == (768, 64)


def test_single_expert_equals_padded_colwise():
    x = rand_bits((200, 96), 1)
    q, s = O.quantize_colwise_grouped(x, [200])
    xp = np.zeros((256, 96), np.uint16)
    xp[:200] = x
    qw, sw = O.quantize_colwise(xp)
    assert np.array_equal(q, qw) and np.array_equal(s[:, :8], sw)
    assert not s[:, 8:].any()


def test_brute_force_ragged_experts():
    group_m = [40, 0, 7, 129, 32]
    x = rand_bits((sum(group_m), 64), 2, std=3.0)
    v = O.bf16_bits_to_f64(x)
    q, s = O.quantize_colwise_grouped(x, group_m)
    kp, P, Q, _, _ = O.grouped_layout(group_m)
    r0 = 0
    for e, m in enumerate(group_m):
        for c in range(64):
            for b in range(kp[e] // 32):
                rows = [r0 + t for t in range(32 * b, 32 * b + 32) if t < m]
                amax = max((abs(v[r, c]) for r in rows), default=0.0)
                want_s = 0 if amax == 0 else max(int(np.floor(np.log2(amax))) - 8 + 127, 0)
                assert s[c, Q[e] + b] == want_s
                for t in range(32 * b, 32 * b + 32):
                    val = v[r0 + t, c] if t < m else 0.0
                    assert q[c, P[e] + t] == O.e4m3_encode(val * 2.0 ** -(want_s - 127))
        r0 += m


def test_wgrad_equals_sum_over_own_tokens():
    group_m = [33, 0, 100, 1]
    N, K = 48, 64
    dy = rand_bits((sum(group_m), N), 3, std=0.5)
    x = rand_bits((sum(group_m), K), 4)
    qa, sa = O.quantize_colwise_grouped(dy, group_m)
    qb, sb = O.quantize_colwise_grouped(x, group_m)
    got = O.mx_grouped_wgrad(qa, sa, qb, sb, group_m)
    kp, P, Q, _, _ = O.grouped_layout(group_m)
    r0 = 0
    for e, m in enumerate(group_m):
        want = np.zeros((N, K))
        if m:
            nb = kp[e] // 32
            da = O.dequantize(qa[:, P[e]:P[e] + kp[e]], sa[:, Q[e]:Q[e] + nb])     # [N, Kp]
            db = O.dequantize(qb[:, P[e]:P[e] + kp[e]], sb[:, Q[e]:Q[e] + nb])     # [K, Kp]
            assert not da[:, m:].any() and not db[:, m:].any()                     # padding is zero
            for t in range(m):                                                    # only the expert's tokens
                want += np.outer(da[:, t], db[:, t])
        np.testing.assert_allclose(got["pre"][e], want, rtol=1e-12, atol=1e-300)
        r0 += m
    assert not got["pre"][1].any()


def test_planted_offset_mistake_is_caught(monkeypatch):
    real = O.grouped_layout

    def shifted(group_m, pad=O.WGRAD_PAD):
        kp, P, Q, tp, ts = real(group_m, pad)
        return kp, P, np.roll(Q, 1) * 0, tp, ts          # every expert's scales at column 0
    monkeypatch.setattr(O, "grouped_layout", shifted)
    with pytest.raises(AssertionError):
        test_brute_force_ragged_experts()
