"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot allocate device
memory (for example a plugin whose host process owns all device memory, or a serving loop that
must not call cudaMalloc).  It keeps the per-chunk decode states in a fixed array inside the
library instead of a caller workspace, so its results must match fa_decode_splitkv's.

This file is collected last on purpose: the entry point shares one array across calls, and the
test must pass both alone in a fresh process and after every other test has run."""
import ctypes

import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from tests.gpu_common import LSE_TOL, O_TOL, cuda, poisoned, require_gpu

SCRATCH_BYTES = 8 << 20          # FA_DECODE_NOALLOC_SCRATCH_BYTES in include/fa.h
UNSUPPORTED = 2


def _reference(q, k, v, scale, n_splits):
    B, H, _, d = q.shape
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, k.shape[2], d, n_splits), dtype=torch.uint8,
                     device="cuda")
    o = poisoned(q.shape, torch.bfloat16)
    lse = poisoned((B, H, 1), torch.float32)
    fa.fa_decode_splitkv(q, k, v, o, lse, scale, n_splits, ws)
    return o, lse


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    require_gpu()
    cases = [(4, 8, 3000, 128, 7), (2, 16, 1000, 64, 0)]    # the second call uses other data
    for B, H, n_kv, d, n_splits in cases:
        x = inputs.make_qkv(B, H, 1, n_kv, d, seed=77 + n_kv, with_do=False)
        q, k, v = cuda(x["q"]), cuda(x["k"]), cuda(x["v"])
        scale = d ** -0.5
        o_ref, lse_ref = _reference(q, k, v, scale, n_splits)
        o = poisoned(q.shape, torch.bfloat16)
        lse = poisoned((B, H, 1), torch.float32)
        fa.fa_decode_splitkv_noalloc(q, k, v, o, lse, scale, n_splits)
        fa.fa_sync_status()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - o_ref.float()).abs().max().item() <= O_TOL
        assert (lse - lse_ref).abs().max().item() <= LSE_TOL


def test_noalloc_rejects_calls_larger_than_its_scratch():
    """Host-side check, no kernel launched: B*H*n_splits*(d+2)*4 above the scratch size."""
    lib = fa.load_library()
    B, H, d, n_splits = 64, 32, 128, 64                      # the 64x32 decode workload: 68 MB
    assert B * H * n_splits * (d + 2) * 4 > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    st = lib.fa_decode_splitkv_noalloc(fake, fake, fake, fake, fake, B, H, 32768, d, 0.1, n_splits, None)
    assert st == UNSUPPORTED
    assert "scratch" in lib.fa_last_error_message().decode()
