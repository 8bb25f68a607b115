"""Block-sparse attention parity: forward and backward through the C ABI against the fp64
oracle's plain definition under the block mask (query i sees key j iff block (i/128, j/128) is
set, and j <= i with causal), the special cases that reduce to the plain kernels, rows that see
no key, per-head masks, and a long-sequence pattern sampled at full size."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import (assert_grad_close, assert_lse_close, assert_o_close, cuda, poisoned,
                              require_gpu)

pytestmark = pytest.mark.gpu
BLK = fa.BLOCK_SIZE


def nblocks(n):
    return (n + BLK - 1) // BLK


def run_fwd(x, mask, causal, scale):
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned(q.shape[:3], torch.float32)
    fa.fa_fwd_block_sparse(q, k, v, o, lse, scale, cuda(mask), causal)
    fa.fa_sync_status()
    return o, lse


# (B, H, N_q, N_kv, d, causal, mask seed, per-head)
FWD_CASES = [
    (1, 2, 1000, 1000, 128, False, 1, False),
    (1, 2, 1000, 1000, 128, True, 2, False),
    (2, 2, 700, 500, 64, False, 3, False),     # N_q != N_kv, ragged last blocks
    (2, 3, 640, 640, 128, True, 4, True),      # one pattern per head
    (1, 2, 1300, 1300, 64, True, 5, False),
    (1, 1, 200, 1500, 128, False, 6, True),
]


def _mask(case):
    B, H, nq, nkv, d, causal, seed, per_head = case
    return inputs.make_block_mask(nblocks(nq), nblocks(nkv), seed, band=0, n_global=1, p_random=0.35,
                                  heads=(B, H) if per_head else None)


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("_c" if c[5] else "") + ("_ph" if c[7] else ""))
def test_block_sparse_forward_matches_oracle(case):
    require_gpu()
    B, H, nq, nkv, d, causal, seed, _ = case
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=900 + seed, with_do=False)
    mask = _mask(case)
    o, lse = run_fwd(x, mask, causal, scale)
    o_ref, lse_ref = A.forward_block_sparse(x["q"], x["k"], x["v"], scale, mask.numpy(), causal)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_all_ones_mask_equals_the_plain_kernels(causal, d):
    """Every block set: the block-sparse kernels stream the same tiles in the same order as the
    plain ones, so O, lse, dK and dV agree bit for bit (dQ sums over key tiles through L2 in a
    run-dependent order, so it is compared with the tolerance)."""
    require_gpu()
    x = inputs.make_qkv(2, 3, 1000, 1000, d, seed=31)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    ones = torch.ones(nblocks(1000), nblocks(1000), dtype=torch.uint8, device="cuda")
    o_b, lse_b = fa.forward_block_sparse(q, k, v, ones, causal)
    o, lse = fa.forward(q, k, v, causal=causal)
    assert torch.equal(o_b, o) and torch.equal(lse_b, lse)
    g_b = fa.backward_block_sparse(q, k, v, o, lse, do, ones, causal)
    g = fa.backward(q, k, v, o, lse, do, causal=causal)
    assert torch.equal(g_b[1], g[1]) and torch.equal(g_b[2], g[2])
    rq = g[0].detach().double().cpu().numpy()
    assert_grad_close(g_b[0], rq, "dQ")


def test_empty_mask_rows_give_zero_and_neg_inf():
    require_gpu()
    B, H, N, d = 1, 2, 700, 128
    x = inputs.make_qkv(B, H, N, N, d, seed=33)
    mask = torch.ones(nblocks(N), nblocks(N), dtype=torch.uint8)
    mask[2] = 0                                      # queries 256..383 see nothing
    mask[:, 4] = 0                                   # nobody sees keys 512..639
    o, lse = run_fwd(x, mask, False, d ** -0.5)
    o, lse = o.cpu(), lse.cpu()
    assert (o[:, :, 256:384].float() == 0).all()
    assert torch.isneginf(lse[:, :, 256:384]).all()
    o_ref, lse_ref = A.forward_block_sparse(x["q"], x["k"], x["v"], d ** -0.5, mask.numpy(), False)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    o_g, lse_g = fa.forward_block_sparse(q, k, v, cuda(mask))
    dq, dk, dv = fa.backward_block_sparse(q, k, v, o_g, lse_g, do, cuda(mask))
    fa.fa_sync_status()
    assert (dq[:, :, 256:384].float() == 0).all()
    assert (dk[:, :, 512:640].float() == 0).all() and (dv[:, :, 512:640].float() == 0).all()
    rq, rk, rv = A.backward_block_sparse(x["q"], x["k"], x["v"], x["do"], d ** -0.5, mask.numpy(), False)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_all_zero_mask():
    require_gpu()
    x = inputs.make_qkv(1, 2, 300, 300, 64, seed=34)
    mask = torch.zeros(nblocks(300), nblocks(300), dtype=torch.uint8)
    o, lse = run_fwd(x, mask, False, 0.125)
    assert (o.float() == 0).all() and torch.isneginf(lse).all()


BWD_CASES = [
    (1, 2, 1000, 1000, 128, False, 11, False),
    (1, 2, 1000, 1000, 128, True, 12, False),
    (2, 2, 700, 500, 64, False, 13, False),
    (2, 3, 640, 640, 128, True, 14, True),
    (1, 2, 900, 900, 64, True, 15, False),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("_c" if c[5] else "") + ("_ph" if c[7] else ""))
def test_block_sparse_backward_matches_oracle(case):
    require_gpu()
    B, H, nq, nkv, d, causal, seed, _ = case
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=950 + seed)
    mask = _mask(case)
    q, k, v, do = (cuda(x[n]) for n in ("q", "k", "v", "do"))
    m = cuda(mask)
    o, lse = fa.forward_block_sparse(q, k, v, m, causal, scale=scale)
    dq, dk, dv = fa.backward_block_sparse(q, k, v, o, lse, do, m, causal, scale=scale)
    fa.fa_sync_status()
    rq, rk, rv = A.backward_block_sparse(x["q"], x["k"], x["v"], x["do"], scale, mask.numpy(), causal)
    assert_grad_close(dq, rq, "dQ")
    assert_grad_close(dk, rk, "dK")
    assert_grad_close(dv, rv, "dV")


def test_block_sparse_long_sequence_sampled_rows():
    """1 x 16 x 16384 x 128, causal, under the benchmark's block pattern (band, global first
    block, 5% random), launched as the benchmark launches it; the oracle checks sampled rows of
    sampled heads."""
    require_gpu()
    B, H, N, d = 1, 16, 16384, 128
    scale = d ** -0.5
    x = inputs.make_qkv(B, H, N, N, d, seed=1003, with_do=False)
    mask = inputs.make_block_mask(nblocks(N), nblocks(N), 1005)
    o, lse = run_fwd(x, mask, True, scale)
    o, lse = o.cpu(), lse.cpu()
    g = np.random.default_rng(12)
    for h in (0, 7, 15):
        rows = np.sort(g.choice(N, size=40, replace=False))
        rows[0], rows[-1] = 0, N - 1
        o_ref, lse_ref = A.forward_block_sparse_rows(x["q"][0, h, rows], rows, x["k"][0, h], x["v"][0, h],
                                                     scale, mask.numpy(), True)
        assert_o_close(o[0, h, rows], o_ref)
        assert_lse_close(lse[0, h, rows], lse_ref)
