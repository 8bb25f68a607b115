"""Host-side checks of the C ABI: the library builds and loads, exports every symbol include/fa.h
declares, and rejects bad arguments with the documented codes before launching anything.
None of these calls reach a CUDA kernel, so they run without a GPU."""
import ctypes
import os
import re

import pytest

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
CSRC = os.path.join(ROOT, "exact_io_aware_08_gb300", "csrc")

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_bwd", "fa_decode_splitkv", "fa_bwd_workspace_size",
                 "fa_decode_workspace_size", "fa_sync_status", "fa_status_string",
                 "fa_last_error_message"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode() == name


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N_q=128, N_kv=128, d=64,
             scale=0.125, causal=0)
    a.update(kw)
    return lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N_q"], a["N_kv"],
                      a["d"], a["scale"], a["causal"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED), (dict(causal=1, N_kv=64), UNSUPPORTED),
    (dict(q=None), INVALID), (dict(o=None), INVALID), (dict(lse=None), INVALID),
    (dict(k=FAKE + 2), INVALID), (dict(B=0), INVALID), (dict(H=-1), INVALID),
    (dict(N_q=-5), INVALID), (dict(scale=0.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(N_q=1 << 30), UNSUPPORTED),
])
def test_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code
    assert lib.fa_last_error_message().decode() not in ("", "no error")


def test_fwd_empty_query_is_a_noop(lib):
    assert fwd(lib, N_q=0, q=None, o=None, lse=None) == 0


def test_bwd_workspace_size_and_rejection(lib):
    need = lib.fa_bwd_workspace_size(2, 3, 100, 100, 64)
    assert need >= 2 * 3 * 100 * 64 * 4 + 2 * 3 * 100 * 4
    assert lib.fa_bwd_workspace_size(1, 1, 10, 10, 96) == 0
    args = [FAKE] * 9
    # too small, misaligned and null workspaces are all FA_ERR_WORKSPACE
    for ws, nbytes in ((FAKE, need - 1), (FAKE + 16, need), (None, need)):
        st = lib.fa_bwd(*args, ws, nbytes, 2, 3, 100, 100, 64, 0.125, 0, None)
        assert st == WORKSPACE
    st = lib.fa_bwd(*args, FAKE, need, 2, 3, 100, 90, 64, 0.125, 1, None)
    assert st == UNSUPPORTED
    args[5] = None   # dO
    assert lib.fa_bwd(*args, FAKE, need, 2, 3, 100, 100, 64, 0.125, 0, None) == INVALID


def test_decode_workspace_and_rejection(lib):
    need = lib.fa_decode_workspace_size(4, 2, 1000, 128, 8)
    assert need == 4 * 2 * 8 * (128 + 2) * 4
    assert lib.fa_decode_workspace_size(4, 2, 1000, 128, 0) > 0        # automatic split count
    assert lib.fa_decode_workspace_size(4, 2, 1000, 128, 5000) == 0
    st = lib.fa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 1000, 128, 0.1, 8, FAKE,
                               need - 4, None)
    assert st == WORKSPACE
    st = lib.fa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 1000, 128, 0.1, 2000, FAKE,
                               1 << 30, None)
    assert st == UNSUPPORTED
    st = lib.fa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 1000, 80, 0.1, 8, FAKE,
                               1 << 30, None)
    assert st == UNSUPPORTED


def test_python_binding_raises_loudly_without_library(tmp_path):
    with pytest.raises(fa.FaError):
        fa.load_library(str(tmp_path / "missing.so"))


def test_library_source_never_allocates():
    """The library takes all memory from the caller: no cudaMalloc/cudaFree in its sources."""
    for fn in os.listdir(CSRC):
        text = open(os.path.join(CSRC, fn)).read()
        assert "cudaMalloc" not in text and "cudaFree" not in text, fn


def test_selftest_rejects_bad_limits(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == INVALID
    assert lib.fa_selftest_wait_timeout(20 * 1000 * 1000, None) == INVALID


def test_paged_decode_rejection(lib):
    """Host-side checks of fa_decode_paged: block size, table capacity, alignment, workspace."""
    def call(block_size=128, num_blocks=8, max_blocks=4, max_seqlen=500, d=128, ws_bytes=1 << 30,
             table=FAKE, seqlens=FAKE, n_splits=4):
        return lib.fa_decode_paged(FAKE, FAKE, FAKE, FAKE, FAKE, table, seqlens, 2, 2, max_blocks,
                                   block_size, num_blocks, max_seqlen, d, 0.1, n_splits, FAKE,
                                   ws_bytes, None)
    assert call(block_size=96) == UNSUPPORTED
    assert call(block_size=32) == UNSUPPORTED
    assert call(max_seqlen=513) == INVALID                    # 4 blocks of 128 hold 512 keys
    assert call(num_blocks=0) == INVALID
    assert call(table=None) == INVALID
    assert call(seqlens=FAKE + 2) == INVALID
    assert call(d=80) == UNSUPPORTED
    assert call(ws_bytes=2 * 2 * 4 * 130 * 4 - 4) == WORKSPACE
    assert call(num_blocks=1 << 24, block_size=256) == UNSUPPORTED   # rows past 2^31


def test_fwd_fp8_rejection(lib):
    def call(d=128, scale=0.1, dq=0.01, dk=0.01, dv=0.01, causal=0, N_kv=256, k=FAKE):
        return lib.fa_fwd_fp8(FAKE, k, FAKE, FAKE, FAKE, 1, 2, 256, N_kv, d, scale, dq, dk, dv,
                              causal, None)
    assert call(d=64) == UNSUPPORTED
    assert call(dq=0.0) == INVALID
    assert call(dv=float("nan")) == INVALID
    assert call(dk=-1.0) == INVALID
    assert call(scale=float("inf")) == INVALID
    assert call(dq=1e-30, dk=1e-30) == INVALID          # the product underflows to 0
    assert call(causal=1, N_kv=128) == UNSUPPORTED
    assert call(k=FAKE + 8) == INVALID


def test_window_entry_points_validate_like_the_plain_ones(lib):
    st = lib.fa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 96, 0.1, 10, 0, None)
    assert st == UNSUPPORTED
    st = lib.fa_fwd_window(FAKE, None, FAKE, FAKE, FAKE, 1, 2, 256, 128, 0.1, 10, 0, None)
    assert st == INVALID
    need = lib.fa_bwd_workspace_size(1, 2, 256, 256, 128)
    args = [FAKE] * 9
    st = lib.fa_bwd_window(*args, FAKE, need - 1, 1, 2, 256, 128, 0.1, 10, 0, None)
    assert st == WORKSPACE


def test_block_sparse_entry_points_validate_before_launching(lib):
    fwd = lib.fa_fwd_block_sparse
    # (q, k, v, o, lse, B, H, N_q, N_kv, d, scale, causal, mask, per_head, stream)
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 96, 0.1, 0, FAKE, 0, None) == UNSUPPORTED
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 0.1, 0, None, 0, None) == INVALID
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 0.1, 0, FAKE, 2, None) == INVALID
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 384, 128, 0.1, 1, FAKE, 0, None) == UNSUPPORTED
    # more than 1024 key blocks
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 1024 * 128 + 1, 128, 0.1, 0, FAKE, 0,
               None) == UNSUPPORTED
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, float("nan"), 0, FAKE, 0, None) == INVALID
    need = lib.fa_bwd_workspace_size(1, 2, 256, 256, 128)
    args = [FAKE] * 9
    bwd = lib.fa_bwd_block_sparse
    assert bwd(*args, FAKE, need - 1, 1, 2, 256, 256, 128, 0.1, 0, FAKE, 0, None) == WORKSPACE
    assert bwd(*args, FAKE, need, 1, 2, 256, 256, 128, 0.1, 0, None, 0, None) == INVALID
    assert bwd(*args, FAKE, need, 1, 2, 256, 256, 64, 0.1, 1, FAKE, 3, None) == INVALID
