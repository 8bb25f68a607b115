"""Split-KV decode parity: the CUDA path (through the C ABI) against the fp64 oracle's full-row
definition, split invariance, empty chunks and the full-size decode workload (sampled heads)."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_lse_close, assert_o_close, cuda, poisoned, require_gpu

pytestmark = pytest.mark.gpu


def run_decode(q, k, v, scale, n_splits):
    B, H, _, d = q.shape
    need = fa.fa_decode_workspace_size(B, H, k.shape[2], d, n_splits)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((B, H, 1), torch.float32)
    fa.fa_decode_splitkv(q, k, v, o, lse, scale, n_splits, ws)
    fa.fa_sync_status()
    return o, lse


# (B, H, N_kv, d, n_splits)
CASES = [
    (1, 1, 512, 128, 8),
    (2, 3, 1000, 128, 7),
    (2, 2, 37, 64, 64),        # more splits than keys: most chunks are empty
    (1, 4, 4096, 64, 0),       # automatic split count
    (3, 2, 100, 128, 1),
    (2, 2, 65, 128, 2),
    (4, 4, 2048, 128, 16),
    (1, 2, 3000, 64, 5),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_decode_matches_oracle(case):
    require_gpu()
    B, H, n_kv, d, n_splits = case
    x = inputs.make_qkv(B, H, 1, n_kv, d, seed=21 + n_kv, with_do=False)
    scale = d ** -0.5
    o, lse = run_decode(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), scale, n_splits)
    o_ref, lse_ref = A.decode(x["q"], x["k"], x["v"], scale)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def test_decode_split_invariance():
    require_gpu()
    x = inputs.make_qkv(2, 4, 1, 4096, 128, seed=5, with_do=False)
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    o_ref, lse_ref = A.decode(x["q"], x["k"], x["v"], 128 ** -0.5)
    outs = [run_decode(q, k, v, 128 ** -0.5, s) for s in (1, 2, 64)]
    for o, lse in outs:
        assert_o_close(o, o_ref)
        assert_lse_close(lse, lse_ref)
    # the split count changes only rounding
    assert (outs[0][0].float() - outs[2][0].float()).abs().max().item() <= 1e-2


def test_decode_empty_cache():
    require_gpu()
    q = cuda(torch.randn(2, 3, 1, 128).to(torch.bfloat16))
    k = torch.empty(2, 3, 0, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = run_decode(q, k, k, 0.1, 4)
    assert (o.float() == 0).all() and torch.isneginf(lse).all()


def test_decode_full_workload_sampled_heads():
    """The decode workload at full size (34 GB of K/V, drawn on the device from the seed), the
    launch configuration the benchmark times; the oracle checks a sample of (b, h) rows."""
    require_gpu()
    w = inputs.DECODE
    x = inputs.make_workload(w, with_do=False, device="cuda")
    o, lse = run_decode(x["q"], x["k"], x["v"], w.scale, w.n_splits)
    o, lse = o.cpu(), lse.cpu()
    for bh in (0, 1, 777, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        q = x["q"][b:b + 1, h:h + 1].cpu()
        k = x["k"][b:b + 1, h:h + 1].cpu()
        v = x["v"][b:b + 1, h:h + 1].cpu()
        o_ref, lse_ref = A.decode(q, k, v, w.scale)
        assert_o_close(o[b, h], o_ref[0, 0])
        assert_lse_close(lse[b, h], lse_ref[0, 0])
        # the method's own split/merge in fp64 agrees with the full row
        m, l, ot = A.decode_partials(q[0, 0], k[0, 0], v[0, 0], w.scale, w.n_splits)
        om, lm = A.decode_merge(m, l, ot)
        assert np.abs(om - o_ref[0, 0, 0]).max() < 1e-12 and abs(lm - lse_ref[0, 0, 0]) < 1e-12
    del x
    torch.cuda.empty_cache()
