"""Pin strength: plant a plausible mistake in the oracle (a dropped term, a wrong sign or index,
a transposed operand) and check that at least one pin in ``test_oracle`` fails.

Mistakes are planted on the CPU, in the oracle module, by monkeypatching one function at a time.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
import tests.test_oracle as P

NEG_INF = -np.inf


def _scores_no_scale(q, k, scale, causal):
    s = q @ k.T
    if causal:
        i = np.arange(s.shape[0])[:, None]
        j = np.arange(s.shape[1])[None, :]
        s = np.where(j <= i, s, NEG_INF)
    return s


def _scores_mask(pred):
    def f(q, k, scale, causal):
        s = scale * (q @ k.T)
        if causal:
            i = np.arange(s.shape[0])[:, None]
            j = np.arange(s.shape[1])[None, :]
            s = np.where(pred(i, j), s, NEG_INF)
        return s
    return f


def _scores_transposed(q, k, scale, causal):
    s = scale * (k @ q.T).T.T if q.shape[0] == k.shape[0] else scale * (q @ k.T)[:, ::-1]
    if causal:
        i = np.arange(s.shape[0])[:, None]
        j = np.arange(s.shape[1])[None, :]
        s = np.where(j <= i, s, NEG_INF)
    return s


def _softmax_no_max(s):
    e = np.exp(s)
    l = e.sum(axis=-1)
    return e / l[..., None], np.zeros(s.shape[:-1]), l


def _softmax_two_pass_wrong_sum(s):
    m = s.max(axis=-1)
    e = np.exp(s - m[..., None])
    l = np.exp(s).sum(axis=-1)            # sum taken without the max shift
    return e / l[..., None], m, l


def _lse_drop_m(m, l):
    return np.log(l)


def _bwd(variant):
    def f(q, k, v, do, scale, causal):
        _, _, p = A.forward_head(q, k, v, scale, causal)
        dv = p.T @ do if variant != "dv_transposed" else (p @ do if p.shape[0] == p.shape[1] else p.T @ do * 2)
        dp = do @ v.T
        D = (p * dp).sum(axis=-1) if variant != "D_rowsum_dp" else dp.sum(axis=-1)
        ds = p * (dp - D[:, None]) if variant != "ds_sign" else p * (D[:, None] - dp)
        dq = scale * (ds @ k)
        dk = scale * (ds.T @ q) if variant != "dk_no_scale" else ds.T @ q
        return dq, dk, dv, D
    return f


def _online_step_no_o_rescale(m_prev, l_prev, o_prev, x_blk, v_blk):
    x_blk = np.asarray(x_blk, float)
    v_blk = np.asarray(v_blk, float)
    m_new = max(m_prev, float(x_blk.max()))
    f = math.exp(m_prev - m_new) if m_prev != NEG_INF else 0.0
    w = np.exp(x_blk - m_new)
    return m_new, f * l_prev + w.sum(), o_prev + np.tensordot(w, v_blk, axes=(0, 0)), f


def _merge_plain_average(o_a, lse_a, o_b, lse_b):
    if lse_a == NEG_INF:
        return np.asarray(o_b, float), lse_b
    if lse_b == NEG_INF:
        return np.asarray(o_a, float), lse_a
    return (np.asarray(o_a) + np.asarray(o_b)) / 2, float(np.logaddexp(lse_a, lse_b))


def _decode_merge_linear_weights(m, l, o):
    m = np.asarray(m, float)
    live = np.isfinite(m)
    mm = m[live].max()
    w = np.where(live, np.where(live, m, mm) - mm + 1.0, 0.0)   # forgot the exponential
    l_tot = (w * np.asarray(l)).sum()
    return (w[:, None] * np.asarray(o)).sum(axis=0) / l_tot, mm + math.log(l_tot)


def _e4m3_bias8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 8.0))
    return sign * np.where((e == 0xF) & (m == 0x7), np.nan, mag)


def _e4m3_no_subnormals(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    mag = (1.0 + m / 8.0) * np.exp2(e - 7.0)                      # implicit 1 for e == 0 too
    return sign * np.where((e == 0xF) & (m == 0x7), np.nan, mag)


_forward_fp8_orig = A.forward_fp8


def _fp8_swapped_scales(q8, k8, v8, scale, dq, dk, dv, causal=False):
    return _forward_fp8_orig(q8, k8, v8, scale, dv, dk, dq, causal)


def _window_off_by_one(n_q, n_kv, left, right):
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    vis = np.ones((n_q, n_kv), dtype=bool)
    if left >= 0:
        vis &= j > i - left                                      # drops the window's first key
    if right >= 0:
        vis &= j <= i + right
    return vis


def _window_sides_swapped(n_q, n_kv, left, right):
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    vis = np.ones((n_q, n_kv), dtype=bool)
    if right >= 0:
        vis &= j >= i - right
    if left >= 0:
        vis &= j <= i + left
    return vis


def _block_visible_transposed(block_mask, n_q, n_kv, block, causal):
    bm = np.asarray(block_mask).astype(bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    vis = bm[j // block, i // block]                             # mask indexed (key, query)
    return vis & (j <= i) if causal else vis


def _block_visible_no_causal(block_mask, n_q, n_kv, block, causal):
    bm = np.asarray(block_mask).astype(bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    return bm[i // block, j // block]                            # drops the causal part


# the pins each mutation is run against (any failing one is a catch)
FWD_PINS = [
    lambda: P.test_forward_vs_torch_sdpa_fp64((2, 3, 37, 37, 16), False),
    lambda: P.test_forward_vs_torch_sdpa_fp64((2, 3, 37, 37, 16), True),
    lambda: P.test_forward_vs_scipy_softmax_logsumexp(False),
    lambda: P.test_forward_vs_scipy_softmax_logsumexp(True),
    P.test_causal_row0_sees_only_key0,
    P.test_rows_of_p_sum_to_one,
    P.test_huge_scores_do_not_overflow,
    lambda: P.test_zero_query_is_uniform_average(True),
    P.test_identical_keys_uniform_and_shifted_lse,
]
BWD_PINS = [
    lambda: P.test_backward_central_finite_differences((1, 2, 8, 8, 4), False),
    lambda: P.test_backward_central_finite_differences((1, 2, 8, 8, 4), True),
    lambda: P.test_backward_vs_torch_autograd_fp64(False),
]
METHOD_PINS = [
    P.test_worked_example_a_online_by_hand,
    P.test_worked_example_b_merge,
    P.test_check_yourself_q1_q2,
    P.test_quick_checks_factor_and_merge,
    lambda: P.test_decode_partials_merge_equals_full_row(1000, 7),
]

FP8_PINS = [
    P.test_e4m3_hand_values,
    P.test_e4m3_all_codes_match_torch_float8,
    P.test_forward_fp8_scales_act_where_they_belong,
    P.test_forward_fp8_equals_torch_sdpa_on_dequantized_values,
]

WINDOW_PINS = [
    P.test_window_special_cases_reduce_to_causal_and_full,
    P.test_window_zero_width_returns_own_value,
    lambda: P.test_window_vs_torch_sdpa_boolean_mask(3, 7),
    lambda: P.test_window_backward_vs_torch_autograd(2, 5),
]

BLOCK_PINS = [
    lambda: P.test_block_sparse_vs_torch_sdpa_boolean_mask(False),
    lambda: P.test_block_sparse_vs_torch_sdpa_boolean_mask(True),
    P.test_block_sparse_all_ones_reduces_to_plain_attention,
    P.test_block_diagonal_mask_is_attention_within_each_segment,
]

MUTATIONS = [
    ("scores", _scores_no_scale, FWD_PINS),
    ("scores", _scores_mask(lambda i, j: j < i), FWD_PINS),
    ("scores", _scores_mask(lambda i, j: j >= i), FWD_PINS),
    ("scores", _scores_transposed, FWD_PINS),
    ("three_pass_softmax", _softmax_no_max, FWD_PINS),
    ("three_pass_softmax", _softmax_two_pass_wrong_sum, FWD_PINS),
    ("lse_from", _lse_drop_m, FWD_PINS),
    ("backward_head", _bwd("D_rowsum_dp"), BWD_PINS),
    ("backward_head", _bwd("ds_sign"), BWD_PINS),
    ("backward_head", _bwd("dk_no_scale"), BWD_PINS),
    ("backward_head", _bwd("dv_transposed"), BWD_PINS),
    ("online_step", _online_step_no_o_rescale, METHOD_PINS),
    ("merge", _merge_plain_average, METHOD_PINS),
    ("decode_merge", _decode_merge_linear_weights, METHOD_PINS),
    ("decode_e4m3", _e4m3_bias8, FP8_PINS),
    ("decode_e4m3", _e4m3_no_subnormals, FP8_PINS),
    ("forward_fp8", _fp8_swapped_scales, FP8_PINS),
    ("window_visible", _window_off_by_one, WINDOW_PINS),
    ("window_visible", _window_sides_swapped, WINDOW_PINS),
    ("block_visible", _block_visible_transposed, BLOCK_PINS),
    ("block_visible", _block_visible_no_causal, BLOCK_PINS),
]


@pytest.mark.parametrize("idx", range(len(MUTATIONS)))
def test_planted_mistake_is_caught(idx, monkeypatch):
    name, fn, pins = MUTATIONS[idx]
    monkeypatch.setattr(A, name, fn)
    caught = 0
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, FloatingPointError, ValueError):
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake in {name} ({fn.__name__})"
