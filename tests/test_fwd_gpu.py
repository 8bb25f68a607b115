"""Forward pass parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import (assert_lse_close, assert_o_close, cuda, poisoned, require_gpu)

pytestmark = pytest.mark.gpu


def run_fwd(q, k, v, causal, scale):
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned(q.shape[:3], torch.float32)
    fa.fa_fwd(q, k, v, o, lse, scale, causal)
    fa.fa_sync_status()
    return o, lse


# (B, H, N_q, N_kv, d, causal): several tiles, ragged tails, N_q != N_kv, single rows
SHAPES = [
    (1, 1, 128, 128, 64, False),
    (1, 2, 100, 100, 64, True),
    (1, 2, 100, 100, 128, False),
    (2, 3, 257, 257, 128, True),
    (1, 2, 1000, 1000, 64, True),
    (1, 2, 1000, 1000, 128, True),
    (1, 1, 200, 333, 128, False),
    (1, 1, 333, 200, 64, False),
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 700, 128, False),
    (1, 1, 129, 129, 128, True),
    (2, 2, 384, 384, 64, False),
    (1, 1, 640, 640, 128, False),
    (3, 4, 700, 700, 128, True),     # 12 heads: causal items ordered across a full and a partial group
    (3, 3, 300, 300, 64, True),      # 9 heads, d = 64
    # one-CTA-per-item kernel with an empty second query tile in the last item (its MMA thread
    # has no work for more steps than the K/V ring is deep)
    (1, 2, 2100, 2100, 128, True),
    (1, 1, 4224, 4224, 64, False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fwd_matches_oracle(shape):
    require_gpu()
    B, H, nq, nkv, d, causal = shape
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=7 + nq + d, with_do=False)
    scale = d ** -0.5
    o, lse = run_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), causal, scale)
    o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], scale, causal)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def test_fwd_tiny_workload_exact_check():
    require_gpu()
    w = inputs.TINY
    x = inputs.make_workload(w, with_do=False)
    o, lse = run_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), w.causal, w.scale)
    o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], w.scale, w.causal)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def test_fwd_gpt2m_workload_all_heads():
    require_gpu()
    w = inputs.GPT2M
    x = inputs.make_workload(w, with_do=False)
    o, lse = run_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), w.causal, w.scale)
    o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], w.scale, w.causal)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def _sampled_rows_check(w, heads, rows_per_head=24, seed=0):
    x = inputs.make_workload(w, with_do=False)
    o, lse = run_fwd(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), w.causal, w.scale)
    g = np.random.default_rng(seed)
    n = w.N_q
    fixed = np.array([0, 1, 2, 127, 128, n // 2, n - 129, n - 2, n - 1])
    o_c, lse_c = o.cpu(), lse.cpu()
    for bh in heads:
        b, h = divmod(bh, w.H)
        rows = np.unique(np.concatenate([fixed, g.integers(0, n, rows_per_head)]))
        o_ref, lse_ref = A.forward_rows(x["q"][b, h, rows], rows, x["k"][b, h], x["v"][b, h],
                                        w.scale, w.causal)
        assert_o_close(o_c[b, h, rows], o_ref)
        assert_lse_close(lse_c[b, h, rows], lse_ref)
    return o


@pytest.mark.parametrize("w", [inputs.HEADLINE, inputs.HEADLINE_CAUSAL], ids=lambda w: w.name)
def test_fwd_headline_workload_sampled_rows(w):
    require_gpu()
    _sampled_rows_check(w, heads=[0, 37, 64, w.B * w.H - 1])


def test_fwd_long_workload_with_outliers_sampled_rows():
    require_gpu()
    _sampled_rows_check(inputs.LONG, heads=[0, 9, 15], rows_per_head=32)


def test_fwd_empty_key_set_gives_zero_and_neg_inf():
    require_gpu()
    q = cuda(torch.randn(1, 2, 70, 64).to(torch.bfloat16))
    k = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = run_fwd(q, k, k, False, 0.125)
    assert (o.float() == 0).all()
    assert torch.isneginf(lse).all()


def test_fwd_is_deterministic():
    require_gpu()
    x = inputs.make_qkv(2, 4, 600, 600, 128, seed=3, with_do=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o1, l1 = run_fwd(q, k, v, True, 0.1)
    o2, l2 = run_fwd(q, k, v, True, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_respects_stream():
    require_gpu()
    x = inputs.make_qkv(1, 2, 300, 300, 64, seed=4, with_do=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    s = torch.cuda.Stream()
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned(q.shape[:3], torch.float32)
    with torch.cuda.stream(s):
        fa.fa_fwd(q, k, v, o, lse, 0.125, False)
    s.synchronize()
    o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], 0.125, False)
    assert_o_close(o, o_ref)


@pytest.mark.parametrize("causal,d,N", [(c, d, n) for c in (False, True) for d in (64, 128)
                                          for n in (1000, 2000)] + [(True, 64, 3500)])
def test_fwd_short_heads_many_items_per_cta(causal, d, N):
    """Short heads (up to 32 key tiles causal at d = 64, 16 causal or at d = 64, 8 otherwise)
    run on the persistent forward, each CTA taking several work items (4 x 32 heads x 2 to 7
    query pairs): it must agree bit for bit with the one-CTA-per-item kernel, which the windowed
    entry point runs for the same mask, and with the oracle on sampled heads.  (2000 unmasked at
    d = 128 runs the one-CTA-per-item kernel on both sides.)"""
    require_gpu()
    B, H = 4, 32
    x = inputs.make_qkv(B, H, N, N, d, seed=77 + d, with_do=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    scale = d ** -0.5
    o, lse = run_fwd(q, k, v, causal, scale)
    o_w = poisoned(q.shape, torch.bfloat16)
    lse_w = poisoned(q.shape[:3], torch.float32)
    fa.fa_fwd_window(q, k, v, o_w, lse_w, scale, -1, 0 if causal else -1)
    fa.fa_sync_status()
    assert torch.equal(o, o_w) and torch.equal(lse, lse_w)
    for b, h in ((0, 0), (2, 17), (3, 31)):
        o_ref, lse_ref = A.forward(x["q"][b:b + 1, h:h + 1], x["k"][b:b + 1, h:h + 1],
                                   x["v"][b:b + 1, h:h + 1], scale, causal)
        assert_o_close(o[b:b + 1, h:h + 1], o_ref)
        assert_lse_close(lse[b:b + 1, h:h + 1], lse_ref)
