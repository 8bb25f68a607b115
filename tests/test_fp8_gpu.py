"""FP8 forward parity: the CUDA path (e4m3 Q, K, V with one scale each) against the fp64 oracle's
attention of the dequantized tensors.

Accuracy bar (derived from the arithmetic, not fitted).  Scores are sums of exact e4m3 code
products in fp32, so S matches the oracle to fp32 rounding.  The only coarse step is the e4m3
rounding of each weight w_j = 2^{(s_j - m) tau' + 4} before the P V product: to nearest, so
|dw_j| <= 2^-4 w_j where e4m3 is normal (w_j >= 2^-6) and |dw_j| <= 2^-10 below.  O is
normalised by the unrounded sum l >= max_j w_j >= 2^4, so per output element

  |O_gpu - O| <= sum_j max(2^-4 P_j, 2^-14 max_i P_i) |V_j|  +  2^-8 |O|  (bf16 output)  + 1e-5

with P the exact attention weights of the row.  The roundings are to nearest and independent,
so the mean error must also sit well below the mean bound (a biased rounding, such as
truncation, would not).  lse uses the unrounded weights: max-abs 1e-3, as for bf16."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import LSE_TOL, assert_lse_close, poisoned, require_gpu

pytestmark = pytest.mark.gpu


def dequant(x, s):
    return A.decode_e4m3(x.cpu().numpy()) * s


def run_fp8(x, causal, scale):
    q8, k8, v8 = (x[n].cuda() for n in ("q8", "k8", "v8"))
    B, H, n_q, d = q8.shape
    o = poisoned((B, H, n_q, d), torch.bfloat16)
    lse = poisoned((B, H, n_q), torch.float32)
    fa.fa_fwd_fp8(q8, k8, v8, o, lse, scale, x["descale_q"], x["descale_k"], x["descale_v"], causal)
    fa.fa_sync_status()
    return o.cpu().double().numpy(), lse


def bound_rows(q, k, v, rows, scale, causal):
    """Per-element error bound for query rows ``rows`` of one head (fp64 inputs)."""
    s = scale * (q[rows] @ k.T)
    if causal:
        s = np.where(np.arange(k.shape[0])[None, :] <= np.asarray(rows)[:, None], s, -np.inf)
    if k.shape[0] == 0:
        return np.zeros((len(rows), v.shape[1]))
    mx = s.max(axis=1, keepdims=True)
    p = np.exp(s - mx)
    p /= p.sum(axis=1, keepdims=True)
    wbound = np.maximum(2.0 ** -4 * p, 2.0 ** -14 * p.max(axis=1, keepdims=True))
    return wbound @ np.abs(v)


def check_head(o_gpu, o_ref, q, k, v, rows, scale, causal):
    bound = bound_rows(q, k, v, rows, scale, causal) + 2.0 ** -8 * np.abs(o_ref) + 1e-5
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all()
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert worst <= 1.0, f"O error exceeds the e4m3 bound (ratio {worst:.3f})"
    if err.size > 1000:
        assert err.mean() <= 0.25 * bound.mean(), (err.mean(), bound.mean())


# (B, H, N_q, N_kv, causal)
CASES = [
    (1, 2, 1000, 1000, False),
    (1, 2, 1000, 1000, True),
    (2, 2, 513, 513, True),
    (1, 3, 300, 700, False),
    (1, 1, 128, 128, False),
    (1, 2, 77, 5, False),            # fewer keys than a tile
    (1, 1, 260, 0, False),           # no keys: O = 0, lse = -inf
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) + ("_c" if c[4] else ""))
def test_fp8_forward_within_e4m3_bound(case):
    require_gpu()
    B, H, n_q, n_kv, causal = case
    d = 128
    scale = d ** -0.5
    x = inputs.make_qkv_fp8(B, H, n_q, n_kv, d, seed=60 + n_q + n_kv)
    o, lse = run_fp8(x, causal, scale)
    o_ref, lse_ref = A.forward_fp8(x["q8"], x["k8"], x["v8"], scale, x["descale_q"], x["descale_k"],
                                   x["descale_v"], causal)
    assert_lse_close(lse, lse_ref)
    q, k, v = (dequant(x[n], x["descale_" + n[0]]) for n in ("q8", "k8", "v8"))
    for b in range(B):
        for h in range(H):
            check_head(o[b, h], o_ref[b, h], q[b, h], k[b, h], v[b, h], np.arange(n_q), scale, causal)


def test_fp8_forward_large_scores():
    """Peaked rows: Q and K scaled up so most rows are dominated by a few keys (the running max
    jumps and weights span the whole e4m3 range)."""
    require_gpu()
    x = inputs.make_qkv_fp8(1, 2, 640, 640, 128, seed=8)
    scale = 4 * 128 ** -0.5
    o, lse = run_fp8(x, False, scale)
    o_ref, lse_ref = A.forward_fp8(x["q8"], x["k8"], x["v8"], scale, x["descale_q"], x["descale_k"],
                                   x["descale_v"], False)
    assert_lse_close(lse, lse_ref)
    q, k, v = (dequant(x[n], x["descale_" + n[0]]) for n in ("q8", "k8", "v8"))
    for h in range(2):
        check_head(o[0, h], o_ref[0, h], q[0, h], k[0, h], v[0, h], np.arange(640), scale, False)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_full_size_sampled_rows(causal):
    """The 4x32x4096x128 workload in fp8, launched as the benchmark launches it; the oracle
    checks sampled rows of sampled heads."""
    require_gpu()
    B, H, N, d = 4, 32, 4096, 128
    scale = d ** -0.5
    x = inputs.make_qkv_fp8(B, H, N, N, d, seed=1002)
    o, lse = run_fp8(x, causal, scale)
    lse = lse.cpu().numpy()
    g = np.random.default_rng(5)
    for b, h in [(0, 0), (1, 17), (3, 31)]:
        rows = np.sort(g.choice(N, size=48, replace=False))
        rows[0], rows[-1] = 0, N - 1
        q, k, v = (dequant(x[n][b, h], x["descale_" + n[0]]) for n in ("q8", "k8", "v8"))
        o_ref, lse_ref = A.forward_rows(q[rows], rows, k, v, scale, causal)
        assert np.max(np.abs(lse[b, h, rows] - lse_ref)) <= LSE_TOL
        check_head(o[b, h, rows], o_ref, q, k, v, rows, scale, causal)


def test_fp8_scale_factors_enter_where_they_should():
    """Doubling descale_v doubles O exactly (a power of two) and leaves lse; halving descale_q
    equals halving the softmax scale."""
    require_gpu()
    x = inputs.make_qkv_fp8(1, 2, 300, 300, 128, seed=3)
    scale = 128 ** -0.5
    o1, l1 = run_fp8(x, True, scale)
    o2, l2 = run_fp8(dict(x, descale_v=2 * x["descale_v"]), True, scale)
    assert np.array_equal(o2, 2 * o1)
    assert torch.equal(l1, l2)
    o3, l3 = run_fp8(dict(x, descale_q=0.5 * x["descale_q"]), True, scale)
    o4, l4 = run_fp8(x, True, 0.5 * scale)
    assert np.array_equal(o3, o4)
    assert torch.equal(l3, l4)
