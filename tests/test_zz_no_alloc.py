"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot allocate device
memory (for example a plugin whose host process owns all device memory, or a serving loop that
must not call cudaMalloc).  It keeps the per-chunk decode states in a fixed array inside the
library instead of a caller workspace.  It runs the same kernels in the same order as
fa_decode_splitkv, so its results must equal that call's bit for bit, and both must match the
oracle's plain decode.

This file is collected last on purpose: the entry point shares one array across calls, and the
test must pass both alone in a fresh process and after every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_lse_close, assert_o_close, cuda, poisoned, require_gpu

SCRATCH_BYTES = 8 << 20          # FA_DECODE_NOALLOC_SCRATCH_BYTES in include/fa.h
UNSUPPORTED = 2


def _part_bytes(B, H, d, n_splits):
    return B * H * n_splits * (d + 2) * 4


def _workspace_decode(q, k, v, scale, n_splits):
    """fa_decode_splitkv with a NaN-filled workspace: a state it never writes shows as NaN."""
    B, H, _, d = q.shape
    need = fa.fa_decode_workspace_size(B, H, k.shape[2], d, n_splits)
    ws = torch.full((max(need, 16) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((B, H, 1), torch.float32)
    fa.fa_decode_splitkv(q, k, v, o, lse, scale, n_splits, ws)
    return o, lse


def _noalloc_decode(q, k, v, scale, n_splits):
    B, H, _, d = q.shape
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((B, H, 1), torch.float32)
    fa.fa_decode_splitkv_noalloc(q, k, v, o, lse, scale, n_splits)
    return o, lse


def _check_equal_and_oracle(x, n_splits, heads=None):
    q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
    d = q.shape[-1]
    scale = d ** -0.5
    o_ref, lse_ref = _workspace_decode(q, k, v, scale, n_splits)
    o, lse = _noalloc_decode(q, k, v, scale, n_splits)
    fa.fa_sync_status()                       # raises on a device-side failure
    # same kernels, same order, same inputs: identical bits
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
    # and the plain definition (all heads, or the sampled (b, h) heads of a large call)
    if heads is None:
        o_or, lse_or = A.decode(x["q"], x["k"], x["v"], scale)
        assert_o_close(o, o_or)
        assert_lse_close(lse, lse_or)
    else:
        for b, h in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            o_or, lse_or = A.decode(x["q"][sl], x["k"][sl], x["v"][sl], scale)
            assert_o_close(o[sl], o_or)
            assert_lse_close(lse[sl], lse_or)


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    require_gpu()
    # the second call uses other data, another d and the automatic split count, so a state the
    # second call failed to write would still hold the first call's values
    cases = [(4, 8, 3000, 128, 7), (2, 16, 1000, 64, 0)]
    for B, H, n_kv, d, n_splits in cases:
        x = inputs.make_qkv(B, H, 1, n_kv, d, seed=77 + n_kv, with_do=False)
        _check_equal_and_oracle(x, n_splits)


@pytest.mark.gpu
def test_noalloc_decode_at_the_largest_size_its_scratch_holds():
    """B*H*n_splits*(d+2)*4 = 8,388,600 bytes: 8 below the 8 MiB scratch (2^23 is not a multiple
    of (d+2)*4 for d = 64 or 128, so no call fills it exactly)."""
    require_gpu()
    B, H, d, n_splits, n_kv = 25, 41, 64, 31, 2000
    assert SCRATCH_BYTES - (d + 2) * 4 < _part_bytes(B, H, d, n_splits) <= SCRATCH_BYTES
    x = inputs.make_qkv(B, H, 1, n_kv, d, seed=4711, with_do=False)
    _check_equal_and_oracle(x, n_splits, heads=[(0, 0), (7, 13), (24, 40)])


def test_noalloc_rejects_calls_larger_than_its_scratch():
    """Host-side checks, no kernel launched: every case returns FA_ERR_UNSUPPORTED before the
    (fake, never dereferenced) pointers are used."""
    lib = fa.load_library()
    fake = ctypes.c_void_p(0x10000)

    def call(B, H, n_kv, d, n_splits):
        return lib.fa_decode_splitkv_noalloc(fake, fake, fake, fake, fake, B, H, n_kv, d,
                                             ctypes.c_float(0.1), n_splits, None)

    # one state more than the largest call that fits (B*H*n_splits = 31,776 at d = 64)
    assert _part_bytes(2, 16, 64, 993) > SCRATCH_BYTES
    assert _part_bytes(2, 16, 64, 993) - (64 + 2) * 4 <= SCRATCH_BYTES
    assert call(2, 16, 1 << 16, 64, 993) == UNSUPPORTED
    assert "scratch" in lib.fa_last_error_message().decode()
    # the 64x32 decode workload with its 64 splits: 68 MB of states
    assert call(64, 32, 32768, 128, 64) == UNSUPPORTED
    # automatic split count: 16,384 heads get one chunk each, 8.5 MB of states
    assert call(128, 128, 1000, 128, 0) == UNSUPPORTED
    assert "scratch" in lib.fa_last_error_message().decode()


def test_decode_rejects_more_work_items_than_an_int_holds():
    """B*H*n_splits >= 2^31 is refused on the host by all three decode calls."""
    lib = fa.load_library()
    fake = ctypes.c_void_p(0x10000)
    B, H, n_splits = 1 << 20, 1 << 10, 2                       # B*H = 2^30, items = 2^31
    st = lib.fa_decode_splitkv(fake, fake, fake, fake, fake, B, H, 4096, 128, ctypes.c_float(0.1),
                               n_splits, fake, ctypes.c_size_t(1 << 62), None)
    assert st == UNSUPPORTED
    assert "n_splits" in lib.fa_last_error_message().decode()
    assert lib.fa_decode_workspace_size(B, H, 4096, 128, n_splits) == 0
    st = lib.fa_decode_splitkv_noalloc(fake, fake, fake, fake, fake, B, H, 4096, 128,
                                       ctypes.c_float(0.1), n_splits, None)
    assert st == UNSUPPORTED
    st = lib.fa_decode_paged(fake, fake, fake, fake, fake, fake, fake, B, H, 64, 64, 1024, 4096, 128,
                             ctypes.c_float(0.1), n_splits, fake, ctypes.c_size_t(1 << 62), None)
    assert st == UNSUPPORTED
    assert np.int64(B) * H * n_splits == 1 << 31
