"""Pins for the fp64 oracle: values the pages print, closed forms, invariants, independent
library routines and finite differences.  None of these retypes the oracle's formulas.

Pages: "FlashAttention and online softmax" (ML Systems lesson 4) -- "Lesson4" below.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rng_inputs(seed, B, H, n_q, n_kv, d, dv=None):
    g = np.random.default_rng(seed)
    dv = d if dv is None else dv
    q = g.standard_normal((B, H, n_q, d))
    k = g.standard_normal((B, H, n_kv, d))
    v = g.standard_normal((B, H, n_kv, dv))
    do = g.standard_normal((B, H, n_q, dv))
    return q, k, v, do


# ---------------------------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------------------------

def test_online_scalar_example_lesson4_small_numbers():
    g = load("online_scalar_1_2_then_4.json")
    b1, b2 = g["blocks"]
    x = np.array(b1 + b2)
    v = np.zeros_like(x)                      # values do not enter l
    m, l, o, tr = A.online_softmax(x, v, [(0, 2), (2, 3)])
    p = g["printed"]
    nd = g["printed_decimals"]
    assert round(tr[0][1], nd) == p["l_after_block1"]
    assert round(tr[1][0], nd) == p["factor_block2"]
    assert round(tr[1][0] * tr[0][1], nd) == p["rescaled_old_sum"]
    assert m == p["m_final"]
    assert round(l, nd) == p["l_final"]
    # closed form 1 + e^-2 + e^-3
    assert abs(l - (1 + math.exp(-2) + math.exp(-3))) < 1e-15


def test_worked_example_a_online_by_hand():
    g = load("worked_example_a.json")
    x = np.log(np.array(g["x_exp"]))
    v = np.array(g["v"])
    m, l, o, tr = A.online_softmax(x, v, [tuple(b) for b in g["blocks"]])
    for (f, lj, oj), want in zip(tr, g["per_block"]):
        assert abs(f - want["factor"]) < 1e-15
        assert abs(lj - want["l"]) < 1e-14
        assert abs(oj - want["o_tilde"]) < 1e-14
    assert abs(o / l - 44 / 15) < 1e-14
    assert abs(m + math.log(l) - math.log(15)) < 1e-14
    # the oracle's plain definition agrees with the page's hand computation too
    o_def, lse_def, _ = A.forward_head(x[None, :1] * 0 + 1.0, x[:, None], v[:, None], 1.0, False)
    assert abs(o_def[0, 0] - 44 / 15) < 1e-14
    assert abs(lse_def[0] - math.log(15)) < 1e-14


def test_worked_example_b_merge():
    g = load("worked_example_b_merge.json")
    o, lse = A.merge(np.array([4 / 3]), math.log(3), np.array([10 / 3]), math.log(12))
    assert abs(lse - math.log(15)) < 1e-14
    assert abs(o[0] - 44 / 15) < 1e-14
    assert abs(math.exp(math.log(3) - lse) - g["merged"]["w_A"]) < 1e-15
    assert abs(math.exp(math.log(12) - lse) - g["merged"]["w_B"]) < 1e-15
    assert abs(o[0] - 7 / 3) > 0.5            # the plain average is wrong


def test_check_yourself_q1_q2():
    g = load("check_yourself.json")
    q1 = g["q1"]
    s = q1["state"]
    m, l, o, f = A.online_step(s["m"], s["l"], s["o_tilde"], q1["block_scores"], q1["block_values"])
    e2 = math.exp(-2)
    assert m == 5.0
    assert abs(l - (1 + 3 * e2)) < 1e-15 and round(l, 3) == q1["answer"]["l_printed"]
    assert abs(o - (1 + 5 * e2)) < 1e-15 and round(float(o), 3) == q1["answer"]["o_tilde_printed"]
    assert round(float(o) / l, 3) == q1["answer"]["output_printed"]
    q2 = g["q2"]
    o, lse = A.merge(np.array([1.0]), math.log(2), np.array([4.0]), math.log(6))
    assert abs(lse - math.log(8)) < 1e-15
    assert abs(o[0] - 3.25) < 1e-15


def test_quick_checks_factor_and_merge():
    g = load("quick_checks.json")
    # the state after a block with max 3, then a block whose largest score is 5
    m, l, o, f = A.online_step(-np.inf, 0.0, 0.0, [3.0], [0.0])
    m, l, o, f = A.online_step(m, l, o, [5.0, 1.0], [0.0, 0.0])
    assert abs(f - math.exp(3 - 5)) < 1e-16
    o, lse = A.merge(np.array([2.0]), math.log(1), np.array([5.0]), math.log(3))
    assert abs(o[0] - 17 / 4) < 1e-15 and abs(lse - math.log(4)) < 1e-15


# ---------------------------------------------------------------------------------------------
# The theorem: online recurrence == three-pass softmax, any block split
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_online_equals_three_pass_random_splits(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 300))
    x = g.standard_normal(n) * (1 + 10 * seed)
    v = g.standard_normal((n, 5))
    cuts = sorted(set(g.integers(0, n + 1, size=int(g.integers(0, 12))).tolist()) | {0, n})
    bounds = list(zip(cuts[:-1], cuts[1:]))
    m, l, o, _ = A.online_softmax(x, v, bounds)
    p, m3, l3 = A.three_pass_softmax(x[None, :])
    assert m == m3[0]
    np.testing.assert_allclose(o / l, (p @ v)[0], rtol=0, atol=1e-13)
    assert abs((m + math.log(l)) - A.lse_from(m3, l3)[0]) < 1e-12


def test_page_numpy_tiled_check_n100_d32():
    """Lesson4 §5 'In code': a tiled pass over N=100 (not a multiple of the 16 tile), d=32
    must match the plain definition to 1e-12, causal and not."""
    g = np.random.default_rng(0)
    Q, K, V = (g.normal(size=(100, 32)) for _ in range(3))
    tau = 1 / math.sqrt(32)
    for causal in (False, True):
        o_ref, lse_ref, _ = A.forward_head(Q, K, V, tau, causal)
        for i in range(100):
            x = tau * (K @ Q[i])
            n_vis = i + 1 if causal else 100
            bounds = [(j, min(j + 16, n_vis)) for j in range(0, n_vis, 16)]
            m, l, o, _ = A.online_softmax(x, V, bounds)
            assert np.abs(o / l - o_ref[i]).max() < 1e-12
            assert abs(m + math.log(l) - lse_ref[i]) < 1e-12


def test_huge_scores_do_not_overflow():
    """Lesson4 §2: the naive e^x overflows past 89 in fp32; the safe and online forms do not."""
    x = np.array([1000.0, 999.0, 10.0, 1001.0])
    v = np.array([[1.0], [2.0], [3.0], [4.0]])
    p, m, l = A.three_pass_softmax(x[None, :])
    assert np.isfinite(p).all() and m[0] == 1001.0
    mo, lo, oo, _ = A.online_softmax(x, v, [(0, 1), (1, 3), (3, 4)])
    np.testing.assert_allclose(oo / lo, (p @ v)[0], atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Forward: independent library routines and invariants
# ---------------------------------------------------------------------------------------------

def _sdpa64(q, k, v, scale, causal):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal,
                                                         scale=scale)
    return o.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 3, 37, 37, 16), (1, 2, 130, 130, 64), (1, 1, 5, 9, 8)])
def test_forward_vs_torch_sdpa_fp64(shape, causal):
    B, H, nq, nkv, d = shape
    if causal and nq != nkv:
        pytest.skip("causal is defined for N_q == N_kv")
    q, k, v, _ = rng_inputs(7, B, H, nq, nkv, d)
    tau = 1 / math.sqrt(d)
    o, lse = A.forward(q, k, v, tau, causal)
    np.testing.assert_allclose(o, _sdpa64(q, k, v, tau, causal), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_vs_scipy_softmax_logsumexp(causal):
    from scipy.special import logsumexp, softmax
    q, k, v, _ = rng_inputs(3, 1, 2, 50, 50, 12)
    tau = 0.37
    o, lse = A.forward(q, k, v, tau, causal)
    for h in range(2):
        s = tau * q[0, h] @ k[0, h].T
        if causal:
            s = s + np.triu(np.full((50, 50), -np.inf), 1)
        np.testing.assert_allclose(lse[0, h], logsumexp(s, axis=1), atol=1e-12)
        np.testing.assert_allclose(o[0, h], softmax(s, axis=1) @ v[0, h], atol=1e-12)


def test_rows_of_p_sum_to_one():
    q, k, v, _ = rng_inputs(5, 1, 1, 64, 80, 16)
    for causal in (False,):
        _, _, p = A.forward_head(q[0, 0], k[0, 0], v[0, 0], 0.25, causal)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    q, k, v, _ = rng_inputs(6, 1, 1, 64, 64, 16)
    _, _, p = A.forward_head(q[0, 0], k[0, 0], v[0, 0], 0.25, True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert (np.triu(p, 1) == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_o_equal_v(causal):
    q, k, _, _ = rng_inputs(8, 1, 2, 40, 40, 8)
    row = np.arange(8.0) - 3.5
    v = np.broadcast_to(row, (1, 2, 40, 8)).copy()
    o, _ = A.forward(q, k, v, 0.5, causal)
    np.testing.assert_allclose(o, v[:, :, :40], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_is_uniform_average(causal):
    _, k, v, _ = rng_inputs(9, 1, 1, 30, 30, 6)
    q = np.zeros((1, 1, 30, 6))
    o, lse = A.forward(q, k, v, 1.0, causal)
    for i in range(30):
        n = i + 1 if causal else 30
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-13


def test_identical_keys_uniform_and_shifted_lse():
    q, _, v, _ = rng_inputs(10, 1, 1, 12, 20, 4)
    k1 = np.random.default_rng(1).standard_normal(4)
    k = np.broadcast_to(k1, (1, 1, 20, 4)).copy()
    tau = 0.3
    o, lse = A.forward(q, k, v, tau, False)
    for i in range(12):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, i] - (tau * q[0, 0, i] @ k1 + math.log(20))) < 1e-12


def test_causal_row0_sees_only_key0():
    q, k, v, _ = rng_inputs(11, 1, 1, 16, 16, 8)
    tau = 0.2
    o, lse = A.forward(q, k, v, tau, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert abs(lse[0, 0, 0] - tau * q[0, 0, 0] @ k[0, 0, 0]) < 1e-14


def test_empty_key_set():
    q = np.ones((1, 1, 3, 4))
    k = np.zeros((1, 1, 0, 4))
    v = np.zeros((1, 1, 0, 4))
    o, lse = A.forward(q, k, v, 1.0, False)
    assert (o == 0).all() and np.isneginf(lse).all()
    o, lse = A.merge(np.zeros(2), -np.inf, np.zeros(2), -np.inf)
    assert (o == 0).all() and lse == -np.inf
    o, lse = A.merge(np.array([1.0, 2.0]), 0.5, np.zeros(2), -np.inf)
    assert (o == [1.0, 2.0]).all() and lse == 0.5


def test_forward_rows_matches_full_head():
    q, k, v, _ = rng_inputs(12, 1, 1, 70, 70, 8)
    o, lse, _ = A.forward_head(q[0, 0], k[0, 0], v[0, 0], 0.4, True)
    idx = np.array([0, 5, 33, 69])
    o2, lse2 = A.forward_rows(q[0, 0, idx], idx, k[0, 0], v[0, 0], 0.4, True)
    np.testing.assert_allclose(o2, o[idx], atol=1e-15)
    np.testing.assert_allclose(lse2, lse[idx], atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Backward: finite differences, torch autograd, the D identity
# ---------------------------------------------------------------------------------------------

def _loss(q, k, v, do, tau, causal):
    o, _ = A.forward(q, k, v, tau, causal)
    return float((do * o).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 5, 5, 3), (1, 2, 8, 8, 4), (1, 1, 3, 7, 2)])
def test_backward_central_finite_differences(shape, causal):
    B, H, nq, nkv, d = shape
    if causal and nq != nkv:
        pytest.skip("causal is defined for N_q == N_kv")
    q, k, v, do = rng_inputs(13, B, H, nq, nkv, d)
    tau = 0.7
    dq, dk, dv, _ = A.backward(q, k, v, do, tau, causal)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, tau, causal)
            x[idx] = old - h
            lm = _loss(q, k, v, do, tau, causal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        scale = max(1.0, np.abs(g).max())
        assert np.abs(num - g).max() / scale < 1e-7


@pytest.mark.parametrize("causal", [False, True])
def test_backward_vs_torch_autograd_fp64(causal):
    q, k, v, do = rng_inputs(14, 2, 2, 48, 48, 16)
    tau = 0.25
    dq, dk, dv, _ = A.backward(q, k, v, do, tau, causal)
    tq, tk, tv = (torch.from_numpy(a.copy()).requires_grad_() for a in (q, k, v))
    s = tau * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(48, 48, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sampled_equals_full_head(causal):
    q, k, v, do = rng_inputs(18, 1, 1, 90, 90, 8)
    dq, dk, dv, _ = A.backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.3, causal)
    qr, kr = np.array([0, 7, 50, 89]), np.array([0, 1, 44, 89])
    sq, sk, sv = A.backward_sampled(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.3, causal, qr, kr, block=32)
    np.testing.assert_allclose(sq, dq[qr], atol=1e-13)
    np.testing.assert_allclose(sk, dk[kr], atol=1e-13)
    np.testing.assert_allclose(sv, dv[kr], atol=1e-13)


def test_D_identity_rowsum_do_o():
    """Lesson4 §3 'Backward pass', step 3: D_i = sum_j P_ij dP_ij = dO_i . O_i."""
    q, k, v, do = rng_inputs(15, 1, 3, 33, 33, 8)
    for causal in (False, True):
        o, _ = A.forward(q, k, v, 0.3, causal)
        _, _, _, D = A.backward(q, k, v, do, 0.3, causal)
        np.testing.assert_allclose(D, (do * o).sum(axis=-1), atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Split-KV decode
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("n_kv,n_splits", [(512, 8), (1000, 7), (37, 64), (64, 1), (5, 5)])
def test_decode_partials_merge_equals_full_row(n_kv, n_splits):
    q, k, v, _ = rng_inputs(16, 1, 1, 1, n_kv, 16)
    tau = 0.25
    m, l, o = A.decode_partials(q[0, 0], k[0, 0], v[0, 0], tau, n_splits)
    out, lse = A.decode_merge(m, l, o)
    o_ref, lse_ref = A.decode(q, k, v, tau)
    np.testing.assert_allclose(out, o_ref[0, 0, 0], atol=1e-13)
    assert abs(lse - lse_ref[0, 0, 0]) < 1e-12
    # the same result by folding the pairwise (o, lse) merge over the chunks
    acc_o, acc_lse = np.zeros(16), -np.inf
    for c in range(n_splits):
        if np.isfinite(m[c]):
            acc_o, acc_lse = A.merge(acc_o, acc_lse, o[c] / l[c], m[c] + math.log(l[c]))
        else:
            acc_o, acc_lse = A.merge(acc_o, acc_lse, np.zeros(16), -np.inf)
    np.testing.assert_allclose(acc_o, o_ref[0, 0, 0], atol=1e-13)


def test_merge_is_associative_and_order_free():
    g = np.random.default_rng(17)
    parts = [(g.standard_normal(3), float(g.standard_normal() * 5)) for _ in range(5)]
    def fold(seq):
        o, lse = np.zeros(3), -np.inf
        for po, pl in seq:
            o, lse = A.merge(o, lse, po, pl)
        return o, lse
    o1, l1 = fold(parts)
    o2, l2 = fold(parts[::-1])
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    assert abs(l1 - l2) < 1e-13
    w = np.exp(np.array([p[1] for p in parts]) - l1)
    assert abs(w.sum() - 1) < 1e-14                     # merge weights sum to 1


# ---------------------------------------------------------------------------- FP8 forward
# e4m3 codes: 1 sign, 4 exponent (bias 7), 3 mantissa bits; subnormals; S.1111.111 is NaN.
E4M3_HAND = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0x40: 2.0, 0xC0: -2.0, 0x3C: 1.5, 0x7E: 448.0,
             0xFE: -448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x30: 0.5,
             0x77: 240.0, 0x1F: 1.875 * 2.0 ** -4}


def test_e4m3_hand_values():
    for code, val in E4M3_HAND.items():
        got = A.decode_e4m3(np.array([code]))[0]
        assert got == val, (hex(code), got, val)
    assert np.isnan(A.decode_e4m3(np.array([0x7F, 0xFF]))).all()


def test_e4m3_all_codes_match_torch_float8():
    """Every code against an independent decoder (torch's float8_e4m3fn upcast)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    mine = A.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert np.array_equal(mine[~nan], ref[~nan])


def _fp8_case(seed, B=1, H=2, N=40, d=16):
    g = np.random.default_rng(seed)
    codes = [g.integers(0, 256, size=(B, H, N, d), dtype=np.uint8) for _ in range(3)]
    for c in codes:                       # no NaN codes
        c[(c & 0x7F) == 0x7F] = 0x38
    return codes


def test_forward_fp8_scales_act_where_they_belong():
    """descale_v scales O and leaves lse; descale_q and descale_k act like the softmax scale;
    a swapped or dropped scale fails one of these."""
    q8, k8, v8 = _fp8_case(3)
    tau = 0.05
    o1, l1 = A.forward_fp8(q8, k8, v8, tau, 1.0, 1.0, 1.0, causal=True)
    o2, l2 = A.forward_fp8(q8, k8, v8, tau, 1.0, 1.0, 2.0, causal=True)
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)
    o3, l3 = A.forward_fp8(q8, k8, v8, tau, 0.5, 1.0, 1.0, causal=True)
    o4, l4 = A.forward_fp8(q8, k8, v8, tau * 0.5, 1.0, 1.0, 1.0, causal=True)
    o5, l5 = A.forward_fp8(q8, k8, v8, tau, 1.0, 0.5, 1.0, causal=True)
    np.testing.assert_allclose(o3, o4, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o5, o4, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l3, l4, rtol=1e-12)
    np.testing.assert_allclose(l5, l4, rtol=1e-12)


def test_forward_fp8_equals_torch_sdpa_on_dequantized_values():
    import torch
    q8, k8, v8 = _fp8_case(4)
    sq, sk, sv, tau = 0.02, 0.03, 0.5, 0.25
    o, lse = A.forward_fp8(q8, k8, v8, tau, sq, sk, sv, causal=False)
    deq = lambda c, s: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64) * s
    qt, kt, vt = deq(q8, sq), deq(k8, sk), deq(v8, sv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=tau)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-10, atol=1e-12)
    lse_ref = torch.logsumexp(tau * qt @ kt.transpose(-1, -2), dim=-1)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=1e-12)


# ---------------------------------------------------------------------------- sliding window
def _qkv(seed, B=1, H=2, N=37, d=8):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, H, N, d)) for _ in range(4)]


def test_window_special_cases_reduce_to_causal_and_full():
    q, k, v, _ = _qkv(1)
    for (left, right), causal in (((-1, 0), True), ((-1, -1), False), ((40, 40), False), ((36, 0), True)):
        o, lse = A.forward_window(q, k, v, 0.3, left, right)
        o_ref, lse_ref = A.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-14)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


def test_window_zero_width_returns_own_value():
    q, k, v, _ = _qkv(2)
    o, lse = A.forward_window(q, k, v, 0.3, 0, 0)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bhnd,bhnd->bhn", q, k), atol=1e-14)


@pytest.mark.parametrize("left,right", [(5, 0), (3, 7), (0, 4), (10, -1)])
def test_window_vs_torch_sdpa_boolean_mask(left, right):
    import torch
    q, k, v, _ = _qkv(3)
    o, lse = A.forward_window(q, k, v, 0.3, left, right)
    N = q.shape[2]
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    mask = torch.ones(N, N, dtype=torch.bool)
    if left >= 0:
        mask &= j >= i - left
    if right >= 0:
        mask &= j <= i + right
    qt, kt, vt = (torch.from_numpy(t) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-13)
    s = (0.3 * qt @ kt.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-13)


@pytest.mark.parametrize("left,right", [(6, 0), (2, 5)])
def test_window_backward_vs_torch_autograd(left, right):
    import torch
    q, k, v, do = _qkv(4, N=29)
    dq, dk, dv = A.backward_window(q, k, v, do, 0.3, left, right)
    N = q.shape[2]
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    mask = (j >= i - left) & ((j <= i + right) if right >= 0 else torch.ones_like(j, dtype=torch.bool))
    qt, kt, vt = (torch.from_numpy(t).requires_grad_() for t in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def test_window_rows_match_full_head():
    q, k, v, _ = _qkv(5, N=50)
    rows = np.array([0, 3, 17, 49])
    for left, right in ((4, 0), (7, 3), (-1, 2)):
        o, lse, _ = A.forward_window_head(q[0, 1], k[0, 1], v[0, 1], 0.3, left, right)
        o_r, lse_r = A.forward_window_rows(q[0, 1, rows], rows, k[0, 1], v[0, 1], 0.3, left, right)
        np.testing.assert_allclose(o_r, o[rows], atol=1e-14)
        np.testing.assert_allclose(lse_r, lse[rows], atol=1e-14)


# ---------------------------------------------------------------------------- block-sparse
def _elem_mask_torch(bm, n, block, causal):
    """Element mask built independently of the oracle: repeat each block entry block x block."""
    import torch
    m = torch.from_numpy(np.asarray(bm).astype(bool))
    m = m.repeat_interleave(block, 0).repeat_interleave(block, 1)[:n, :n]
    if causal:
        m = m & torch.ones(n, n, dtype=torch.bool).tril()
    return m


BS_MASK = np.array([[1, 0, 0, 1, 0, 1, 0, 1, 1, 0],
                    [1, 1, 0, 0, 0, 0, 1, 0, 0, 1],
                    [0, 1, 1, 0, 1, 0, 0, 0, 1, 0],
                    [1, 0, 0, 1, 0, 0, 0, 1, 0, 0],
                    [0, 0, 1, 0, 1, 1, 0, 0, 0, 1],
                    [1, 0, 0, 0, 0, 1, 1, 0, 1, 0],
                    [0, 1, 0, 1, 0, 0, 1, 0, 0, 0],
                    [0, 0, 0, 0, 1, 0, 1, 1, 0, 1],
                    [1, 0, 1, 0, 0, 0, 0, 0, 1, 0],
                    [0, 1, 0, 0, 1, 0, 0, 1, 0, 1]], dtype=np.uint8)   # not symmetric, full diagonal


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_vs_torch_sdpa_boolean_mask(causal):
    import torch
    q, k, v, _ = _qkv(6, N=37)                       # block 4: ten blocks, the last one ragged
    o, lse = A.forward_block_sparse(q, k, v, 0.3, BS_MASK, causal, block=4)
    mask = _elem_mask_torch(BS_MASK, 37, 4, causal)
    qt, kt, vt = (torch.from_numpy(t) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-13)
    s = (0.3 * qt @ kt.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-13)


def test_block_sparse_all_ones_reduces_to_plain_attention():
    q, k, v, _ = _qkv(7, N=37)
    ones = np.ones((10, 10), dtype=np.uint8)
    for causal in (False, True):
        o, lse = A.forward_block_sparse(q, k, v, 0.3, ones, causal, block=4)
        o_ref, lse_ref = A.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, o_ref, atol=1e-14)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-13)


def test_block_diagonal_mask_is_attention_within_each_segment():
    q, k, v, _ = _qkv(8, N=37)
    eye = np.eye(10, dtype=np.uint8)
    o, lse = A.forward_block_sparse(q, k, v, 0.3, eye, False, block=4)
    for a in range(0, 37, 4):
        b = min(a + 4, 37)
        o_ref, lse_ref = A.forward(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], 0.3, False)
        np.testing.assert_allclose(o[:, :, a:b], o_ref, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, a:b], lse_ref, atol=1e-13)


def test_block_sparse_empty_block_row_gives_zero_and_neg_inf():
    q, k, v, do = _qkv(9, N=20)
    bm = np.ones((5, 5), dtype=np.uint8)
    bm[2] = 0                                          # queries 8..11 see nothing
    o, lse = A.forward_block_sparse(q, k, v, 0.3, bm, False, block=4)
    assert (o[:, :, 8:12] == 0).all() and np.isneginf(lse[:, :, 8:12]).all()
    assert np.isfinite(lse[:, :, :8]).all() and np.isfinite(lse[:, :, 12:]).all()
    dq, dk, dv = A.backward_block_sparse(q, k, v, do, 0.3, bm, False, block=4)
    assert (dq[:, :, 8:12] == 0).all()
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


def test_block_sparse_per_head_masks():
    q, k, v, _ = _qkv(10, B=2, H=2, N=37)
    g = np.random.default_rng(3)
    per = (g.random((2, 2, 10, 10)) < 0.5).astype(np.uint8)
    per[..., np.arange(10), np.arange(10)] = 1
    o, lse = A.forward_block_sparse(q, k, v, 0.3, per, True, block=4)
    for b in range(2):
        for h in range(2):
            o1, lse1 = A.forward_block_sparse(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                              0.3, per[b, h], True, block=4)
            np.testing.assert_array_equal(o[b, h], o1[0, 0])
            np.testing.assert_array_equal(lse[b, h], lse1[0, 0])


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_backward_vs_torch_autograd(causal):
    import torch
    q, k, v, do = _qkv(11, N=29)                     # every row sees its own diagonal block
    dq, dk, dv = A.backward_block_sparse(q, k, v, do, 0.3, BS_MASK[:8, :8], causal, block=4)
    mask = _elem_mask_torch(BS_MASK[:8, :8], 29, 4, causal)
    qt, kt, vt = (torch.from_numpy(t).requires_grad_() for t in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=0.3)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def test_block_sparse_rows_match_full_head():
    q, k, v, _ = _qkv(12, N=37)
    rows = np.array([0, 5, 17, 36])
    for causal in (False, True):
        o, lse, _ = A.forward_block_sparse_head(q[0, 1], k[0, 1], v[0, 1], 0.3, BS_MASK, 4, causal)
        o_r, lse_r = A.forward_block_sparse_rows(q[0, 1, rows], rows, k[0, 1], v[0, 1], 0.3, BS_MASK,
                                                 causal, block=4)
        np.testing.assert_allclose(o_r, o[rows], atol=1e-14)
        np.testing.assert_allclose(lse_r, lse[rows], atol=1e-14)
