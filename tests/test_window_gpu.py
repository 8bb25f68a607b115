"""Sliding-window attention parity: forward and backward through the C ABI against the fp64
oracle's plain definition under the window (query i sees keys i - left .. i + right), the
special cases that reduce to the causal and unmasked kernels, and a long-sequence window sampled
at full size."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import (assert_grad_close, assert_lse_close, assert_o_close, cuda, poisoned,
                              require_gpu)

pytestmark = pytest.mark.gpu


def run_fwd(x, left, right, scale):
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned(q.shape[:3], torch.float32)
    fa.fa_fwd_window(q, k, v, o, lse, scale, left, right)
    fa.fa_sync_status()
    return o, lse


# (B, H, N, d, left, right)
FWD_CASES = [
    (1, 2, 1000, 128, 100, 0),        # causal sliding window
    (1, 2, 700, 64, 50, 50),          # symmetric band
    (2, 2, 777, 128, 5, 0),           # window much narrower than a tile
    (1, 2, 1000, 128, 300, -1),       # bounded on the left only
    (1, 1, 640, 64, -1, 130),         # bounded on the right only
    (1, 2, 513, 128, 700, 3),         # window wider than the sequence on the left
    (1, 1, 256, 128, 127, 128),       # edges exactly on tile boundaries
    (1, 2, 2500, 64, 600, 0),         # many key tiles per query tile at d = 64
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "x".join(map(str, c[:4])) + f"_w{c[4]}_{c[5]}")
def test_window_forward_matches_oracle(case):
    require_gpu()
    B, H, N, d, left, right = case
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, N, N, d, seed=500 + N + left, with_do=False)
    o, lse = run_fwd(x, left, right, scale)
    o_ref, lse_ref = A.forward_window(x["q"], x["k"], x["v"], scale, left, right)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def test_window_zero_width_returns_v():
    require_gpu()
    x = inputs.make_qkv(1, 2, 300, 300, 128, seed=4, with_do=False)
    o, lse = run_fwd(x, 0, 0, 128 ** -0.5)
    assert torch.equal(o.cpu(), x["v"])


@pytest.mark.parametrize("causal,d,N", [(True, 128, 1000), (False, 128, 1000), (True, 128, 2500),
                                          (False, 128, 2500), (True, 64, 4500), (False, 64, 2200)])
def test_window_special_cases_equal_the_plain_kernels(causal, d, N):
    """(-1, 0) is the causal mask and (-1, -1) no mask: the windowed kernel must reproduce the
    causal / unmasked kernel bit for bit (same tiles, same arithmetic).  At 1000 tokens the
    plain call runs the persistent forward; the longer heads run the one-CTA-per-item kernel,
    whose P hand-off is a named barrier where the windowed kernel's is an mbarrier."""
    require_gpu()
    x = inputs.make_qkv(2, 3, N, N, d, seed=6, with_do=False)
    o_w, lse_w = run_fwd(x, -1, 0 if causal else -1, d ** -0.5)
    o, lse = fa.forward(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), causal=causal, scale=d ** -0.5)
    assert torch.equal(o_w, o)
    assert torch.equal(lse_w, lse)


BWD_CASES = [
    (1, 2, 1000, 128, 100, 0),
    (1, 2, 700, 64, 50, 50),
    (2, 1, 777, 128, 5, 0),
    (1, 2, 600, 128, -1, 200),
    (1, 2, 2500, 64, 600, 0),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "x".join(map(str, c[:4])) + f"_w{c[4]}_{c[5]}")
def test_window_backward_matches_oracle(case):
    require_gpu()
    B, H, N, d, left, right = case
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, N, N, d, seed=800 + N + left)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward_window(q, k, v, left, right, scale=scale)
    dq, dk, dv = fa.backward_window(q, k, v, o, lse, do, left, right, scale=scale)
    fa.fa_sync_status()
    rq, rk, rv = A.backward_window(x["q"], x["k"], x["v"], x["do"], scale, left, right)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_window_backward_causal_special_case_equals_causal_kernel():
    require_gpu()
    x = inputs.make_qkv(1, 2, 640, 640, 128, seed=10)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    g_w = fa.backward_window(q, k, v, o, lse, do, -1, 0)
    g_c = fa.backward(q, k, v, o, lse, do, causal=True)
    for a, b in zip(g_w, g_c):
        assert torch.equal(a, b)


def test_window_long_sequence_sampled_rows():
    """1 x 16 x 16384 x 128 under a 1024-key causal window (the long-context shape), launched
    as the benchmark launches it; the oracle checks sampled rows of sampled heads."""
    require_gpu()
    B, H, N, d, left = 1, 16, 16384, 128, 1024
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, N, N, d, seed=1003, with_do=False)
    o, lse = run_fwd(x, left, 0, scale)
    o, lse = o.cpu(), lse.cpu()
    g = np.random.default_rng(9)
    for h in (0, 9, 15):
        rows = np.sort(g.choice(N, size=40, replace=False))
        rows[0], rows[-1] = 0, N - 1
        o_ref, lse_ref = A.forward_window_rows(x["q"][0, h, rows], rows, x["k"][0, h], x["v"][0, h],
                                               scale, left, 0)
        assert_o_close(o[0, h, rows], o_ref)
        assert_lse_close(lse[0, h, rows], lse_ref)
