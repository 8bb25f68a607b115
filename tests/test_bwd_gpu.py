"""Backward pass parity: dQ, dK, dV from the CUDA path (through the C ABI) against the fp64
oracle.  The GPU backward consumes the GPU forward's own O and lse; the oracle uses its own."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_grad_close, cuda, poisoned, require_gpu

pytestmark = pytest.mark.gpu


def run_fwd_bwd(x, causal, scale):
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned(q.shape[:3], torch.float32)
    fa.fa_fwd(q, k, v, o, lse, scale, causal)
    B, H, nq, d = q.shape
    ws = torch.full((fa.fa_bwd_workspace_size(B, H, nq, k.shape[2], d),), 255, dtype=torch.uint8,
                    device="cuda")                       # garbage on entry must not matter
    dq = poisoned(q.shape, torch.bfloat16)
    dk = poisoned(k.shape, torch.bfloat16)
    dv = poisoned(v.shape, torch.bfloat16)
    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, scale, causal)
    fa.fa_sync_status()
    return dq, dk, dv


SHAPES = [
    (1, 1, 128, 128, 64, False),
    (1, 1, 128, 128, 128, False),
    (1, 2, 100, 100, 64, True),
    (1, 2, 100, 100, 128, True),
    (2, 2, 257, 257, 128, True),
    (1, 2, 300, 300, 64, False),
    (1, 1, 200, 333, 128, False),
    (1, 1, 333, 200, 64, False),
    (1, 2, 1000, 1000, 128, True),
    (1, 1, 1, 130, 128, False),
    (1, 1, 640, 640, 64, True),
    (3, 4, 700, 700, 128, True),     # 12 heads: causal items ordered across a full and a partial group
    (3, 3, 300, 300, 64, True),      # 9 heads, d = 64
    (1, 2, 77, 1000, 64, False),
    # longer heads on the one-CTA-per-key-tile kernels: 33 query steps with a ragged last one
    # (d = 128, causal), 18 key tiles of 128-query steps (d = 64)
    (1, 2, 2100, 2100, 128, True),
    (1, 1, 2304, 2304, 64, False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_matches_oracle(shape):
    require_gpu()
    B, H, nq, nkv, d, causal = shape
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=11 + nq + d)
    scale = d ** -0.5
    dq, dk, dv = run_fwd_bwd(x, causal, scale)
    rq, rk, rv, _ = A.backward(x["q"], x["k"], x["v"], x["do"], scale, causal)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_bwd_tiny_workload():
    require_gpu()
    w = inputs.TINY
    x = inputs.make_workload(w)
    dq, dk, dv = run_fwd_bwd(x, w.causal, w.scale)
    rq, rk, rv, _ = A.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_bwd_gpt2m_workload_all_heads():
    require_gpu()
    w = inputs.GPT2M
    x = inputs.make_workload(w)
    dq, dk, dv = run_fwd_bwd(x, w.causal, w.scale)
    rq, rk, rv, _ = A.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def _sampled_heads(w, heads, n_rows=48, seed=1):
    x = inputs.make_workload(w)
    dq, dk, dv = run_fwd_bwd(x, w.causal, w.scale)
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    g = np.random.default_rng(seed)
    n = w.N_q
    fixed = np.array([0, 1, 127, 128, n // 2, n - 1])
    for bh in heads:
        b, h = divmod(bh, w.H)
        qr = np.unique(np.concatenate([fixed, g.integers(0, n, n_rows)]))
        kr = np.unique(np.concatenate([fixed, g.integers(0, w.N_kv, n_rows)]))
        rq, rk, rv = A.backward_sampled(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h],
                                        w.scale, w.causal, qr, kr)
        # relative to the largest magnitude of the whole tensor of this head
        full_q = np.abs(dq[b, h].double().numpy()).max()
        full_k = np.abs(dk[b, h].double().numpy()).max()
        full_v = np.abs(dv[b, h].double().numpy()).max()
        for got, ref, name, s in ((dq[b, h, qr], rq, "dQ", full_q), (dk[b, h, kr], rk, "dK", full_k),
                                  (dv[b, h, kr], rv, "dV", full_v)):
            got = got.double().numpy()
            assert np.isfinite(got).all()
            err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
            assert err <= 2e-2, f"{name} head {bh}: rel err {err:.3e}"


@pytest.mark.parametrize("w", [inputs.HEADLINE, inputs.HEADLINE_CAUSAL], ids=lambda w: w.name)
def test_bwd_headline_workload_sampled(w):
    require_gpu()
    _sampled_heads(w, heads=[0, 77, w.B * w.H - 1])


def test_bwd_long_workload_with_outliers_sampled():
    require_gpu()
    _sampled_heads(inputs.LONG, heads=[0, 15], n_rows=24)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [300, 512, 1000])
def test_bwd_short_heads_many_items_per_cta(causal, N):
    """Short heads at d = 64 (up to 4 key tiles, or 8 with causal) run on the persistent
    backward, each CTA taking several (head, key tile) items (4 x 32 heads x 3, 4 or 8 key
    tiles): dK and dV must agree bit for bit with the one-CTA-per-tile kernel (which the windowed
    entry point runs for the same mask), dQ (summed across key tiles in a run-dependent order)
    within the tolerance, and all three with the oracle on sampled heads.  (1000 unmasked runs
    the one-CTA-per-tile kernel on both sides.)"""
    require_gpu()
    B, H, d = 4, 32, 64
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, N, N, d, seed=61 + N)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    dq_w, dk_w, dv_w = fa.backward_window(q, k, v, o, lse, do, -1, 0 if causal else -1, scale=scale)
    fa.fa_sync_status()
    assert torch.equal(dk, dk_w) and torch.equal(dv, dv_w)
    assert_grad_close(dq, dq_w.double().cpu().numpy(), "dQ")
    for b, h in ((0, 0), (1, 13), (3, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv, _ = A.backward(x["q"][sl], x["k"][sl], x["v"][sl], x["do"][sl], scale, causal)
        assert_grad_close(dq[sl], rq, "dQ")
        assert_grad_close(dk[sl], rk, "dK")
        assert_grad_close(dv[sl], rv, "dV")


@pytest.mark.parametrize("d,nkv", [(64, 300), (64, 1500), (128, 700)])
def test_bwd_without_queries_gives_zero_dk_dv(d, nkv):
    """N_q = 0: no query sees any key, so dK = dV = 0 everywhere (the persistent backward at
    d = 64 with 3 key tiles, bwd_main_kernel otherwise); outputs start as NaN so an unwritten
    element fails."""
    require_gpu()
    g = torch.Generator().manual_seed(40 + d)
    k, v = (cuda(torch.randn(2, 3, nkv, d, generator=g).to(torch.bfloat16)) for _ in range(2))
    q = torch.empty(2, 3, 0, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, 3, 0, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(fa.fa_bwd_workspace_size(2, 3, 0, nkv, d), 256), dtype=torch.uint8,
                     device="cuda")
    dk, dv = poisoned(k.shape, torch.bfloat16), poisoned(v.shape, torch.bfloat16)
    fa.fa_bwd(q, k, v, q, lse, q, q, dk, dv, ws, d ** -0.5, False)
    fa.fa_sync_status()
    assert (dk.float() == 0).all() and (dv.float() == 0).all()


def test_bwd_dk_dv_deterministic():
    require_gpu()
    x = inputs.make_qkv(1, 2, 512, 512, 128, seed=5)
    a = run_fwd_bwd(x, True, 0.1)
    b = run_fwd_bwd(x, True, 0.1)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_long_workload_needs_no_n_by_n_buffer():
    """1 x 16 x 16384 x 128 causal, forward + backward through the C ABI: the caller's buffers
    (inputs, outputs, the O(N d) workspace) are all the memory the path touches -- far below one
    N x N score matrix per head -- and the calls allocate nothing on the device."""
    require_gpu()
    w = inputs.LONG
    x = {k: v.cuda() for k, v in inputs.make_workload(w).items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:3], dtype=torch.float32, device="cuda")
    grads = [torch.empty_like(x["q"]) for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N_q, w.N_kv, w.d), dtype=torch.uint8,
                     device="cuda")
    caller_bytes = sum(t.numel() * t.element_size() for t in [*x.values(), o, lse, *grads, ws])
    n_by_n_bf16 = w.B * w.H * w.N_q * w.N_kv * 2
    assert caller_bytes < n_by_n_bf16 / 8
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, w.scale, True)
    fa.fa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], *grads, ws, w.scale, True)
    fa.fa_sync_status()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_before - free_after < (64 << 20), (free_before, free_after)
    assert all(torch.isfinite(t.float()).all() for t in (o, *grads))
