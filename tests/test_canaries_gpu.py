"""Out-of-bounds writes, caught with canaries (the planned stand-in for a memory checker): every
output and workspace of every entry point sits inside a larger device buffer whose guard bands
hold a sentinel bit pattern; after the call the guards must be untouched and the output itself
fully written (it starts as the same sentinel, a NaN).  Shapes are ragged so the last tiles of
every kernel are partial."""
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs

pytestmark = pytest.mark.gpu
GUARD = 4096                                      # bytes of guard on each side


class Guarded:
    """A tensor of ``shape``/``dtype`` placed between two guard bands of one allocation."""

    def __init__(self, shape, dtype, fill_inside=True):
        self.dtype = dtype
        esz = torch.tensor([], dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.g = GUARD // esz
        self.n = n
        self.raw = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self.bits = self.raw.view(torch.int16 if esz == 2 else (torch.int32 if esz == 4 else torch.uint8))
        self.sentinel = {2: 0x7F81, 4: 0x7F800001, 1: 0xA5}[esz]    # signalling NaNs / a byte
        self.bits.fill_(self.sentinel)
        self.t = self.raw[self.g:self.g + n].view(shape)

    def check(self, name, fully_written=True):
        g = self.bits[:self.g]
        h = self.bits[self.g + self.n:]
        assert bool((g == self.sentinel).all()), f"{name}: write before the buffer"
        assert bool((h == self.sentinel).all()), f"{name}: write past the buffer"
        if fully_written and self.n:
            inside = self.bits[self.g:self.g + self.n]
            assert not bool((inside == self.sentinel).any()), f"{name}: element never written"


def qkv(B, H, nq, nkv, d, seed, with_do=True):
    x = inputs.make_qkv(B, H, nq, nkv, d, seed=seed, with_do=with_do)
    return {k: v.cuda() for k, v in x.items()}


@pytest.mark.parametrize("shape", [(2, 3, 700, 700, 128, True), (1, 2, 1300, 900, 64, False),
                                   (1, 2, 2100, 2100, 128, True), (1, 1, 77, 300, 64, False)],
                         ids=lambda s: "x".join(map(str, s[:5])) + ("_c" if s[5] else ""))
def test_forward_and_backward_stay_in_bounds(shape):
    B, H, nq, nkv, d, causal = shape
    x = qkv(B, H, nq, nkv, d, seed=21)
    o = Guarded((B, H, nq, d), torch.bfloat16)
    lse = Guarded((B, H, nq), torch.float32)
    fa.fa_fwd(x["q"], x["k"], x["v"], o.t, lse.t, d ** -0.5, causal)
    fa.fa_sync_status()
    o.check("O")
    lse.check("lse")
    need = fa.fa_bwd_workspace_size(B, H, nq, nkv, d)
    ws = Guarded((need,), torch.uint8)
    dq = Guarded((B, H, nq, d), torch.bfloat16)
    dk = Guarded((B, H, nkv, d), torch.bfloat16)
    dv = Guarded((B, H, nkv, d), torch.bfloat16)
    fa.fa_bwd(x["q"], x["k"], x["v"], o.t, lse.t, x["do"], dq.t, dk.t, dv.t, ws.t, d ** -0.5, causal)
    fa.fa_sync_status()
    for g, name in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
        g.check(name)
    ws.check("workspace", fully_written=False)


def test_window_and_block_sparse_stay_in_bounds():
    B, H, N, d = 1, 2, 1500, 128
    x = qkv(B, H, N, N, d, seed=22)
    need = fa.fa_bwd_workspace_size(B, H, N, N, d)
    mask = inputs.make_block_mask(-(-N // 128), -(-N // 128), 3, band=0, p_random=0.3).cuda()
    mask[4] = 0                                  # a query block that sees nothing
    for kind in ("window", "block_sparse"):
        o = Guarded((B, H, N, d), torch.bfloat16)
        lse = Guarded((B, H, N), torch.float32)
        if kind == "window":
            fa.fa_fwd_window(x["q"], x["k"], x["v"], o.t, lse.t, d ** -0.5, 200, 10)
        else:
            fa.fa_fwd_block_sparse(x["q"], x["k"], x["v"], o.t, lse.t, d ** -0.5, mask, True)
        fa.fa_sync_status()
        o.check(f"{kind} O")
        lse.check(f"{kind} lse")
        ws = Guarded((need,), torch.uint8)
        dq, dk, dv = (Guarded((B, H, N, d), torch.bfloat16) for _ in range(3))
        if kind == "window":
            fa.fa_bwd_window(x["q"], x["k"], x["v"], o.t, lse.t, x["do"], dq.t, dk.t, dv.t, ws.t,
                             d ** -0.5, 200, 10)
        else:
            fa.fa_bwd_block_sparse(x["q"], x["k"], x["v"], o.t, lse.t, x["do"], dq.t, dk.t, dv.t, ws.t,
                                   d ** -0.5, mask, True)
        fa.fa_sync_status()
        for g, name in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
            g.check(f"{kind} {name}")
        ws.check(f"{kind} workspace", fully_written=False)


def test_varlen_stays_in_bounds():
    H, d = 3, 128
    lens = [300, 1, 0, 777, 129]
    total = sum(lens)
    g = torch.Generator().manual_seed(23)
    q, k, v, do = (torch.randn(total, H, d, generator=g).to(torch.bfloat16).cuda() for _ in range(4))
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32, device="cuda")
    o = Guarded((total, H, d), torch.bfloat16)
    lse = Guarded((H, total), torch.float32)
    fa.fa_fwd_varlen(q, k, v, o.t, lse.t, cu, cu, max(lens), max(lens), d ** -0.5, True)
    fa.fa_sync_status()
    o.check("varlen O")
    lse.check("varlen lse")
    need = fa.fa_bwd_workspace_size(1, H, total, total, d)
    ws = Guarded((need,), torch.uint8)
    dq, dk, dv = (Guarded((total, H, d), torch.bfloat16) for _ in range(3))
    fa.fa_bwd_varlen(q, k, v, o.t, lse.t, do, dq.t, dk.t, dv.t, ws.t, cu, cu, max(lens), max(lens),
                     d ** -0.5, True)
    fa.fa_sync_status()
    for gg, name in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
        gg.check(f"varlen {name}")
    ws.check("varlen workspace", fully_written=False)


def test_decode_and_fp8_stay_in_bounds():
    B, H, N, d = 3, 4, 5000, 128
    x = qkv(B, H, 1, N, d, seed=24, with_do=False)
    n_splits = 7
    need = fa.fa_decode_workspace_size(B, H, N, d, n_splits)
    ws = Guarded((need,), torch.uint8)
    o = Guarded((B, H, 1, d), torch.bfloat16)
    lse = Guarded((B, H, 1), torch.float32)
    fa.fa_decode_splitkv(x["q"], x["k"], x["v"], o.t, lse.t, d ** -0.5, n_splits, ws.t)
    fa.fa_sync_status()
    o.check("decode O")
    lse.check("decode lse")
    ws.check("decode workspace", fully_written=False)
    x8 = inputs.make_qkv_fp8(1, 2, 900, 1100, 128, seed=25)
    o8 = Guarded((1, 2, 900, 128), torch.bfloat16)
    l8 = Guarded((1, 2, 900), torch.float32)
    fa.fa_fwd_fp8(x8["q8"].cuda(), x8["k8"].cuda(), x8["v8"].cuda(), o8.t, l8.t, 128 ** -0.5,
                  x8["descale_q"], x8["descale_k"], x8["descale_v"], False)
    fa.fa_sync_status()
    o8.check("fp8 O")
    l8.check("fp8 lse")


def test_guard_detects_a_stray_write_and_a_missed_element():
    """The checker itself: a write one element past the end, or an element left unwritten, is
    reported (planted with plain tensor writes, no kernel involved)."""
    a = Guarded((3, 5), torch.bfloat16)
    a.t.zero_()
    a.check("clean")
    a.raw[a.g + a.n] = 1.0                        # one past the end
    with pytest.raises(AssertionError):
        a.check("stray")
    b = Guarded((3, 5), torch.float32)
    b.t.zero_()
    b.bits[b.g + 7] = b.sentinel                  # one element never written
    with pytest.raises(AssertionError):
        b.check("missed")
