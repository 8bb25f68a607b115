"""Variable-length (packed, cu_seqlens) forward: each sequence against the fp64 oracle's plain
definition on that sequence alone; equivalence with the fixed-length kernel; invalid boundaries
are reported, not faulted on."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_lse_close, assert_o_close, poisoned, require_gpu

pytestmark = pytest.mark.gpu


def pack(lq, lk, H, d, seed):
    """Per-sequence seeded draws, packed token-major [total, H, d]; returns CPU tensors."""
    qs, ks, vs, per = [], [], [], []
    for s, (nq, nk) in enumerate(zip(lq, lk)):
        x = inputs.make_qkv(1, H, nq, nk, d, seed + s, with_do=False)
        per.append(x)
        qs.append(x["q"][0].transpose(0, 1))       # [nq, H, d]
        ks.append(x["k"][0].transpose(0, 1))
        vs.append(x["v"][0].transpose(0, 1))
    cu_q = torch.tensor([0] + list(np.cumsum(lq)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(lk)), dtype=torch.int32)
    return torch.cat(qs).contiguous(), torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), cu_q, cu_k, per


def run_varlen(q, k, v, cu_q, cu_k, lq, lk, causal, scale):
    H = q.shape[1]
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((H, q.shape[0]), torch.float32)
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, lse, cu_q.cuda(), cu_k.cuda(), max(lq),
                     max(lk), scale, causal)
    fa.fa_sync_status()
    return o.cpu(), lse.cpu()


CASES = [
    ([100, 1, 300, 128, 129, 513], None, 2, 128, False),
    ([100, 1, 300, 128, 129, 513], None, 2, 128, True),
    ([64, 257, 5, 1000], None, 3, 64, True),
    ([37, 200, 400], [90, 15, 700], 2, 128, False),          # different q and k lengths
    ([50, 0, 80], [60, 0, 80], 2, 64, False),                # an empty sequence
    ([40, 70], [0, 33], 1, 128, False),                      # a sequence with no keys
    # long packed sequences, as in the bench's varlen workload: many tiles, ragged last pairs
    ([3000, 17, 4100], None, 2, 128, True),
    ([2500, 700], None, 2, 64, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{len(c[0])}seq_d{c[3]}_{'c' if c[4] else 'nc'}")
def test_varlen_forward_matches_oracle_per_sequence(case):
    require_gpu()
    lq, lk, H, d, causal = case
    lk = lq if lk is None else lk
    scale = d ** -0.5
    q, k, v, cu_q, cu_k, per = pack(lq, lk, H, d, seed=300 + sum(lq))
    o, lse = run_varlen(q, k, v, cu_q, cu_k, lq, lk, causal, scale)
    for s, x in enumerate(per):
        a, b = int(cu_q[s]), int(cu_q[s + 1])
        if b == a:
            continue
        o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], scale, causal)
        assert_o_close(o[a:b].transpose(0, 1), o_ref[0])
        assert_lse_close(lse[:, a:b], lse_ref[0])


def test_varlen_equals_fixed_length_when_all_lengths_match():
    require_gpu()
    B, H, N, d = 3, 4, 384, 128
    x = inputs.make_qkv(B, H, N, N, d, seed=9, with_do=False)
    o_fix, lse_fix = fa.forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=True)
    pk = lambda t: t.transpose(1, 2).reshape(B * N, H, d).contiguous().cuda()
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32).cuda()
    o_var, lse_var = fa.forward_varlen(pk(x["q"]), pk(x["k"]), pk(x["v"]), cu, cu, N, N, causal=True)
    fa.fa_sync_status()
    assert torch.equal(o_var, pk(o_fix.cpu()))
    assert torch.equal(lse_var.reshape(H, B, N).permute(1, 0, 2).cpu(), lse_fix.cpu())


def test_varlen_bad_boundaries_are_reported():
    require_gpu()
    H, d = 2, 64
    q = torch.randn(100, H, d, device="cuda").to(torch.bfloat16)
    cu_bad = torch.tensor([0, 60, 150], dtype=torch.int32, device="cuda")   # 150 > total 100
    o = torch.empty_like(q)
    lse = torch.empty(H, 100, device="cuda")
    fa.fa_fwd_varlen(q, q, q, o, lse, cu_bad, cu_bad, 90, 90, 0.125, False)
    with pytest.raises(fa.FaError) as e:
        fa.fa_sync_status()
    assert e.value.status == 1
    fa.fa_sync_status()


BWD_CASES = [
    ([100, 1, 300, 128, 129, 513], None, 2, 128, False),
    ([100, 1, 300, 128, 129, 513], None, 2, 128, True),
    ([64, 257, 5, 1000], None, 3, 64, True),
    ([37, 200, 400], [90, 15, 700], 2, 128, False),
    ([50, 0, 80], [60, 0, 80], 2, 64, False),
    ([3000, 17, 4100], None, 2, 128, True),
    ([2500, 700], None, 2, 64, False),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"{len(c[0])}seq_d{c[3]}_{'c' if c[4] else 'nc'}")
def test_varlen_backward_matches_oracle_per_sequence(case):
    require_gpu()
    from tests.gpu_common import assert_grad_close
    lq, lk, H, d, causal = case
    lk = lq if lk is None else lk
    scale = d ** -0.5
    q, k, v, cu_q, cu_k, per = pack(lq, lk, H, d, seed=700 + sum(lq))
    dos = [inputs.make_qkv(1, H, nq, 1, d, 900 + s, with_do=True)["do"] for s, nq in enumerate(lq)]
    do = torch.cat([t[0].transpose(0, 1) for t in dos]).contiguous()
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    cq, ck = cu_q.cuda(), cu_k.cuda()
    o, lse = fa.forward_varlen(qc, kc, vc, cq, ck, max(lq), max(lk), causal=causal, scale=scale)
    dq, dk, dv = fa.backward_varlen(qc, kc, vc, o, lse, doc, cq, ck, max(lq), max(lk), causal=causal,
                                    scale=scale)
    fa.fa_sync_status()
    got = {"dQ": dq.cpu().double(), "dK": dk.cpu().double(), "dV": dv.cpu().double()}
    ref = {n: torch.zeros_like(t) for n, t in got.items()}
    for s, x in enumerate(per):
        aq, bq, ak, bk = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        if bq == aq or bk == ak:
            continue            # nothing to differentiate (the reference gradients are zero)
        rq, rk, rv, _ = A.backward(x["q"], x["k"], x["v"], dos[s], scale, causal)
        ref["dQ"][aq:bq] = torch.from_numpy(rq[0]).transpose(0, 1)
        ref["dK"][ak:bk] = torch.from_numpy(rk[0]).transpose(0, 1)
        ref["dV"][ak:bk] = torch.from_numpy(rv[0]).transpose(0, 1)
    # relative to each packed tensor's largest reference magnitude (as for fixed length)
    for n in ("dQ", "dK", "dV"):
        assert_grad_close(got[n], ref[n].numpy(), n)
