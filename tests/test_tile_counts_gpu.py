"""Tile skipping, counted: the diagnostic counters (fa_debug_counters) report how many S tile
products the forward kernels computed and how many (key tile, query step) pairs the backward
visited; they must equal the tiles the mask needs, no more and no fewer ("Causal masks":
T(T+1)/2 of the T^2 tiles for causal; the same skipping for windows and block masks)."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs

pytestmark = pytest.mark.gpu
T = 128


def cdiv(a, b):
    return -(-a // b)


def counted(fn):
    c = torch.zeros(2, dtype=torch.int64, device="cuda")
    fa.fa_debug_counters(c)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        fa.fa_debug_counters(None)
    fa.fa_sync_status()
    return int(c[0]), int(c[1])


def fwd_tiles(nq, nkv, causal=False, window=None, mask=None):
    """S products one head needs: per query tile, the key tiles holding a key some row sees."""
    total = 0
    for qt in range(cdiv(nq, T)):
        r0, r1 = qt * T, min(nq, qt * T + T) - 1
        if mask is not None:
            total += sum(1 for kt in range(cdiv(nkv, T)) if mask[qt, kt] and (not causal or kt <= qt))
            continue
        lo, hi = 0, nkv - 1
        if causal:
            hi = min(hi, r1)
        if window is not None:
            left, right = window
            if left >= 0:
                lo = max(lo, r0 - left)
            if right >= 0:
                hi = min(hi, r1 + right)
        total += (hi // T - lo // T + 1) if hi >= lo else 0
    return total


def bwd_steps(nq, nkv, d, causal=False, window=None, mask=None):
    """(key tile, query step) pairs one head's backward visits; a step is 64 queries at d = 128."""
    bm = 64 if d == 128 else 128
    nsteps = cdiv(nq, bm)
    total = 0
    for kt in range(cdiv(nkv, T)):
        k0 = kt * T
        if mask is not None:
            for qb in range(cdiv(nq, T)):
                if mask[qb, kt] and (not causal or qb >= kt):
                    total += min(T // bm, cdiv(nq - qb * T, bm))
            continue
        start, end = 0, nsteps
        if causal:
            start = k0 // bm
        if window is not None:
            left, right = window
            if right >= 0:
                start = max(0, k0 - right) // bm
            if left >= 0:
                end = min(nsteps, (k0 + T - 1 + left) // bm + 1)
        total += max(0, end - start)
    return total


FWD = [  # (B, H, N_q, N_kv, d, causal)
    (2, 3, 1000, 1000, 128, True),       # short heads: the persistent kernel
    (1, 2, 2000, 2000, 64, True),
    (1, 2, 700, 1500, 128, False),
    (2, 2, 1000, 300, 64, False),
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: "x".join(map(str, c[:5])) + ("_c" if c[5] else ""))
def test_forward_computes_exactly_the_needed_tiles(case):
    B, H, nq, nkv, d, causal = case
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=5, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    s_count, _ = counted(lambda: fa.forward(q, k, v, causal=causal))
    assert s_count == B * H * fwd_tiles(nq, nkv, causal)


@pytest.mark.parametrize("window", [(300, 0), (100, 200), (-1, 50)])
def test_window_forward_and_backward_visit_exactly_the_band(window):
    B, H, N, d = 1, 2, 3000, 128
    x = inputs.make_qkv(B, H, N, N, d, seed=6)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    (s_count, _) = counted(lambda: fa.forward_window(q, k, v, *window))
    assert s_count == B * H * fwd_tiles(N, N, window=window)
    o, lse = fa.forward_window(q, k, v, *window)
    (_, steps) = counted(lambda: fa.backward_window(q, k, v, o, lse, do, *window))
    assert steps == B * H * bwd_steps(N, N, d, window=window)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_block_sparse_visits_exactly_the_set_blocks(causal, d):
    B, H, N = 2, 2, 1500
    x = inputs.make_qkv(B, H, N, N, d, seed=7)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    mask = inputs.make_block_mask(cdiv(N, T), cdiv(N, T), 8, band=0, n_global=1, p_random=0.3)
    m = mask.cuda()
    (s_count, _) = counted(lambda: fa.forward_block_sparse(q, k, v, m, causal))
    assert s_count == B * H * fwd_tiles(N, N, causal, mask=mask.numpy())
    o, lse = fa.forward_block_sparse(q, k, v, m, causal)
    (_, steps) = counted(lambda: fa.backward_block_sparse(q, k, v, o, lse, do, m, causal))
    assert steps == B * H * bwd_steps(N, N, d, causal, mask=mask.numpy())


@pytest.mark.parametrize("case", [(2, 3, 1000, 1000, 128, True), (1, 2, 700, 500, 64, False),
                                  (1, 2, 1300, 1300, 64, True)],
                         ids=lambda c: "x".join(map(str, c[:5])) + ("_c" if c[5] else ""))
def test_backward_visits_exactly_the_needed_pairs(case):
    B, H, nq, nkv, d, causal = case
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=9)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal)
    (_, steps) = counted(lambda: fa.backward(q, k, v, o, lse, do, causal=causal))
    assert steps == B * H * bwd_steps(nq, nkv, d, causal)


def test_fp8_forward_causal_tile_count():
    B, H, N = 1, 2, 2000
    x = inputs.make_qkv_fp8(B, H, N, N, 128, seed=10)
    q8, k8, v8 = (x[n].cuda() for n in ("q8", "k8", "v8"))
    (s_count, _) = counted(lambda: fa.forward_fp8(q8, k8, v8, x["descale_q"], x["descale_k"],
                                                  x["descale_v"], causal=True))
    assert s_count == B * H * fwd_tiles(N, N, True)


def test_counting_stops_when_unset():
    c = torch.zeros(2, dtype=torch.int64, device="cuda")
    x = inputs.make_qkv(1, 1, 300, 300, 64, seed=11, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    fa.fa_debug_counters(c)
    fa.forward(q, k, v)
    fa.fa_debug_counters(None)
    torch.cuda.synchronize()
    first = c.cpu().numpy().copy()
    assert first[0] == fwd_tiles(300, 300)
    fa.forward(q, k, v)
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy(), first)
