"""Split-KV decode over a paged KV cache: each row against the fp64 oracle's plain definition on
that row's first seqlens_k[b] keys, equality with the contiguous-cache decode, and invalid block
tables or lengths reported rather than faulted on.

The cache is built from contiguous per-row K/V: the blocks a row needs are scattered over a
larger pool in a seeded random order, every other cache row (including the tails of partly used
blocks) is set to NaN, and unused table entries are -1, so a read of anything but the row's own
keys shows up in the output."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_lse_close, assert_o_close, cuda, poisoned, require_gpu

pytestmark = pytest.mark.gpu


def build_paged(k, v, lens, block_size, spare_blocks, seed):
    """k, v [B, H, N, d] (CPU) -> k_cache, v_cache [num_blocks, block_size, H, d], block_table
    [B, max_blocks] int32 with -1 in unused entries."""
    B, H, N, d = k.shape
    need = [-(-L // block_size) for L in lens]
    max_blocks = max(1, -(-N // block_size))
    num_blocks = sum(need) + spare_blocks
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(num_blocks, generator=g)
    kc = torch.full((num_blocks, block_size, H, d), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((num_blocks, block_size, H, d), float("nan"), dtype=torch.bfloat16)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    nxt = 0
    for b, L in enumerate(lens):
        for j in range(need[b]):
            phys = int(order[nxt])
            nxt += 1
            table[b, j] = phys
            lo, hi = j * block_size, min(L, (j + 1) * block_size)
            kc[phys, : hi - lo] = k[b, :, lo:hi].transpose(0, 1)
            vc[phys, : hi - lo] = v[b, :, lo:hi].transpose(0, 1)
    return kc, vc, table


def run_paged(q, kc, vc, table, lens, max_seqlen, scale, n_splits):
    B, H, _, d = q.shape
    need = fa.fa_decode_workspace_size(B, H, max_seqlen, d, n_splits)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((B, H, 1), torch.float32)
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    fa.fa_decode_paged(q, kc, vc, o, lse, table, seqlens, max_seqlen, scale, n_splits, ws)
    fa.fa_sync_status()
    return o, lse


def check_rows(o, lse, x, lens, scale):
    for b, L in enumerate(lens):
        if L == 0:
            assert (o[b].float() == 0).all().item()
            assert torch.isneginf(lse[b]).all().item()
            continue
        o_ref, lse_ref = A.decode(x["q"][b:b + 1], x["k"][b:b + 1, :, :L], x["v"][b:b + 1, :, :L], scale)
        assert_o_close(o[b:b + 1], o_ref)
        assert_lse_close(lse[b:b + 1], lse_ref)


# (lens per batch row, H, d, block_size, n_splits)
CASES = [
    ([1000, 37, 513], 4, 128, 64, 7),
    ([4096, 4096], 2, 128, 256, 0),             # full blocks, automatic split count
    ([300, 0, 64, 129], 3, 64, 128, 5),         # a row with no keys, partly used blocks
    ([1, 2, 3, 70], 2, 128, 64, 64),            # more splits than keys in every row
    ([2500], 8, 64, 512, 16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}rows_d{c[2]}_bs{c[3]}_s{c[4]}")
def test_paged_decode_matches_oracle(case):
    require_gpu()
    lens, H, d, bs, n_splits = case
    B, N = len(lens), max(lens)
    x = inputs.make_qkv(B, H, 1, N, d, seed=400 + N + bs, with_do=False)
    kc, vc, table = build_paged(x["k"], x["v"], lens, bs, spare_blocks=3, seed=N)
    scale = d ** -0.5
    o, lse = run_paged(cuda(x["q"]), cuda(kc), cuda(vc), cuda(table), lens, N, scale, n_splits)
    check_rows(o, lse, x, lens, scale)


def test_paged_equals_contiguous_decode_when_lengths_match():
    """Same keys, same chunking: the paged path must reproduce the contiguous one bit for bit."""
    require_gpu()
    B, H, N, d, n_splits = 3, 4, 2048, 128, 8
    x = inputs.make_qkv(B, H, 1, N, d, seed=17, with_do=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, N, d, n_splits), dtype=torch.uint8, device="cuda")
    o_c = poisoned(q.shape, torch.bfloat16)
    lse_c = poisoned((B, H, 1), torch.float32)
    fa.fa_decode_splitkv(q, k, v, o_c, lse_c, d ** -0.5, n_splits, ws)
    kc, vc, table = build_paged(x["k"], x["v"], [N] * B, 128, spare_blocks=5, seed=3)
    o_p, lse_p = run_paged(q, cuda(kc), cuda(vc), cuda(table), [N] * B, N, d ** -0.5, n_splits)
    assert torch.equal(o_p, o_c)
    assert torch.equal(lse_p, lse_c)


def test_paged_decode_workload_sampled_rows():
    """A serving-sized batch: 32 rows of mixed lengths up to 8192 keys over 256-key blocks; the
    oracle checks a sample of rows, every row must be finite."""
    require_gpu()
    B, H, d, bs = 32, 8, 128, 256
    rng = np.random.default_rng(11)
    lens = [int(L) for L in rng.integers(1, 8193, size=B)]
    N = max(lens)
    x = inputs.make_qkv(B, H, 1, N, d, seed=12, with_do=False)
    kc, vc, table = build_paged(x["k"], x["v"], lens, bs, spare_blocks=16, seed=13)
    scale = d ** -0.5
    o, lse = run_paged(cuda(x["q"]), cuda(kc), cuda(vc), cuda(table), lens, N, scale, 0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rows = [0, 7, 19, 31]
    sub = {n: x[n][rows] for n in ("q", "k", "v")}
    check_rows(o[rows], lse[rows], sub, [lens[r] for r in rows], scale)


@pytest.mark.parametrize("bad", ["block_id", "seqlen"])
def test_paged_bad_table_or_length_is_reported(bad):
    require_gpu()
    B, H, N, d, bs = 2, 2, 512, 64, 128
    x = inputs.make_qkv(B, H, 1, N, d, seed=5, with_do=False)
    kc, vc, table = build_paged(x["k"], x["v"], [N, N], bs, spare_blocks=0, seed=1)
    lens = [N, N]
    if bad == "block_id":
        table[1, 2] = kc.shape[0]            # one past the pool
    else:
        lens = [N, N + 1]                    # longer than max_seqlen_k
    with pytest.raises(fa.FaError) as e:
        run_paged(cuda(x["q"]), cuda(kc), cuda(vc), cuda(table), lens, N, d ** -0.5, 4)
    assert e.value.status == 1
    fa.fa_sync_status()                      # the recorded state was cleared
