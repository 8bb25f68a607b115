"""exact_io_aware_08_gb300 -- exact IO-aware attention (FlashAttention) for GB300 (sm_103a).

A thin ctypes binding over ``libfa.so`` (the C ABI in ``include/fa.h``).  Functions with the C
names take torch CUDA tensors and only marshal pointers, sizes and the current stream; every
step of the computation runs in the library's kernels.  There is no fallback: if the library is
missing or a call is rejected, a ``FaError`` is raised.

Convenience wrappers ``forward``, ``backward`` and ``decode`` allocate outputs with torch (the
library itself never allocates).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FaError", "load_library", "library_path",
    "fa_fwd", "fa_bwd", "fa_bwd_prep", "fa_bwd_main", "fa_bwd_finish", "fa_decode_splitkv", "fa_bwd_workspace_size", "fa_decode_splitkv_noalloc",
    "fa_decode_workspace_size", "fa_sync_status", "fa_status_string", "fa_last_error_message",
    "forward", "backward", "decode", "fa_fwd_varlen", "forward_varlen",
    "fa_bwd_varlen", "backward_varlen", "fa_decode_paged", "decode_paged", "fa_fwd_fp8", "forward_fp8",
    "fa_fwd_window", "fa_bwd_window", "forward_window", "backward_window",
    "fa_fwd_block_sparse", "fa_bwd_block_sparse", "forward_block_sparse", "backward_block_sparse",
    "BLOCK_SIZE", "fa_debug_counters",
]

BLOCK_SIZE = 128   # block-sparse attention: blocks of 128 queries x 128 keys

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa.so")
_lib = None
_lock = threading.Lock()

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_WORKSPACE",
                4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT"}


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P, _P, _I, _I, _I, _I, _I, _I,
                           _I, _F, _I, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_prep": (_I, [_P, _P, _P, _S, _I, _I, _I, _I, _I, _P]),
    "fa_bwd_main": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_finish": (_I, [_P, _P, _S, _I, _I, _I, _I, _I, _F, _P]),
    "fa_decode_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "fa_decode_splitkv_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_window": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_bwd_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_fwd_block_sparse": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P]),
    "fa_bwd_block_sparse": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _I, _I, _I, _I, _I, _F,
                                 _I, _P, _I, _P]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _F, _F, _I, _P]),
    "fa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S,
                             _P]),
    "fa_sync_status": (_I, [_P]),
    "fa_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "fa_debug_counters": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_error_message": (ctypes.c_char_p, []),
}


def load_library(path: str | None = None):
    """Load libfa.so (raises FaError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise FaError(4, f"{p} not found: build it with `python -m exact_io_aware_08_gb300.build`"
                             " (the library has no fallback implementation)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(status: int):
    if status != FA_OK:
        lib = load_library()
        raise FaError(status, lib.fa_last_error_message().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _dims(q, k):
    B, H, n_q, d = q.shape
    return B, H, n_q, k.shape[2], d


# --------------------------------------------------------------------------------------------
# C-named entry points (pointers from tensors; no allocation, no computation)
# --------------------------------------------------------------------------------------------

def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None):
    B, H, n_q, n_kv, d = _dims(q, k)
    _check(load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, n_q, n_kv,
                                 d, float(scale), int(bool(causal)), _stream(stream)))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, scale: float, causal: bool, stream=None):
    """Packed variable-length forward: q/o [total_q, H, d], k/v [total_k, H, d], lse [H, total_q],
    cu_seqlens_* int32 device tensors of n_seqs + 1 boundaries."""
    total_q, H, d = q.shape
    total_k = k.shape[0]
    n_seqs = cu_seqlens_q.numel() - 1
    _check(load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), n_seqs, H, total_q,
                                        total_k, int(max_seqlen_q), int(max_seqlen_k), d,
                                        float(scale), int(bool(causal)), _stream(stream)))


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                   causal: bool = False, scale: float | None = None, stream=None):
    """Returns (O [total_q, H, d] bf16, lse [H, total_q] fp32)."""
    import torch
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale,
                  causal, stream)
    return o, lse


def fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, ws, cu_seqlens_q, cu_seqlens_k,
                  max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool, stream=None):
    total_q, H, d = q.shape
    _check(load_library().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws),
                                        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                        cu_seqlens_q.numel() - 1, H, total_q, k.shape[0],
                                        int(max_seqlen_q), int(max_seqlen_k), d, float(scale),
                                        int(bool(causal)), _stream(stream)))


def backward_varlen(q, k, v, o, lse, do, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    causal: bool = False, scale: float | None = None, stream=None):
    """Returns (dQ, dK, dV) for packed [total, H, d] tensors."""
    import torch
    total_q, H, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    ws = torch.empty(max(fa_bwd_workspace_size(1, H, total_q, k.shape[0], d), 256), dtype=torch.uint8,
                     device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, ws, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, scale, causal, stream)
    return dq, dk, dv


def fa_bwd_workspace_size(B: int, H: int, n_q: int, n_kv: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, n_q, n_kv, d))


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, scale: float, causal: bool, stream=None):
    B, H, n_q, n_kv, d = _dims(q, k)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                                 _ptr(dk), _ptr(dv), _ptr(ws), ws_bytes, B, H, n_q, n_kv, d,
                                 float(scale), int(bool(causal)), _stream(stream)))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def fa_bwd_prep(o, do, ws, n_kv: int, stream=None):
    B, H, n_q, d = o.shape
    _check(load_library().fa_bwd_prep(_ptr(o), _ptr(do), _ptr(ws), _nbytes(ws), B, H, n_q, n_kv, d,
                                      _stream(stream)))


def fa_bwd_main(q, k, v, lse, do, dk, dv, ws, scale: float, causal: bool, stream=None):
    B, H, n_q, n_kv, d = _dims(q, k)
    _check(load_library().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(do), _ptr(dk),
                                      _ptr(dv), _ptr(ws), _nbytes(ws), B, H, n_q, n_kv, d,
                                      float(scale), int(bool(causal)), _stream(stream)))


def fa_bwd_finish(dq, ws, n_kv: int, scale: float, stream=None):
    B, H, n_q, d = dq.shape
    _check(load_library().fa_bwd_finish(_ptr(dq), _ptr(ws), _nbytes(ws), B, H, n_q, n_kv, d,
                                        float(scale), _stream(stream)))


def fa_decode_workspace_size(B: int, H: int, n_kv: int, d: int, n_splits: int) -> int:
    return int(load_library().fa_decode_workspace_size(B, H, n_kv, d, n_splits))


def fa_decode_splitkv(q, k, v, o, lse, scale: float, n_splits: int, ws, stream=None):
    B, H, _, d = q.shape
    n_kv = k.shape[2]
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().fa_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, n_kv,
                                            d, float(scale), int(n_splits), _ptr(ws), ws_bytes,
                                            _stream(stream)))


def fa_decode_splitkv_noalloc(q, k, v, o, lse, scale: float, n_splits: int, stream=None):
    """Split-KV decode without a workspace: the library keeps the per-chunk states in a fixed
    device array of FA_DECODE_NOALLOC_SCRATCH_BYTES (see include/fa.h for the limit and the
    rule that overlapping calls race on it)."""
    B, H, _, d = q.shape
    _check(load_library().fa_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                                    k.shape[2], d, float(scale), int(n_splits),
                                                    _stream(stream)))


def fa_fwd_window(q, k, v, o, lse, scale: float, window_left: int, window_right: int, stream=None):
    B, H, N, d = q.shape
    _check(load_library().fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                        float(scale), int(window_left), int(window_right),
                                        _stream(stream)))


def fa_bwd_window(q, k, v, o, lse, do, dq, dk, dv, ws, scale: float, window_left: int,
                  window_right: int, stream=None):
    B, H, N, d = q.shape
    _check(load_library().fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws), B, H,
                                        N, d, float(scale), int(window_left), int(window_right),
                                        _stream(stream)))


def _mask_args(block_mask, B, H):
    """(pointer, per_head) of a uint8 device block mask: [nqb, nkb] shared or [B, H, nqb, nkb]."""
    per_head = 1 if block_mask.dim() == 4 else 0
    if per_head and tuple(block_mask.shape[:2]) != (B, H):
        raise FaError(1, f"per-head block mask must be [B, H, nqb, nkb], got {tuple(block_mask.shape)}")
    if not block_mask.is_contiguous():
        raise FaError(1, "block mask must be contiguous")
    return _ptr(block_mask), per_head


def fa_fwd_block_sparse(q, k, v, o, lse, scale: float, block_mask, causal: bool = False, stream=None):
    """block_mask: uint8 on the device, [ceil(N_q/128), ceil(N_kv/128)] or per head
    [B, H, ceil(N_q/128), ceil(N_kv/128)]; nonzero = block computed."""
    B, H, n_q, d = q.shape
    n_kv = k.shape[2]
    mp, per_head = _mask_args(block_mask, B, H)
    _check(load_library().fa_fwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                              n_q, n_kv, d, float(scale), int(bool(causal)), mp,
                                              per_head, _stream(stream)))


def fa_bwd_block_sparse(q, k, v, o, lse, do, dq, dk, dv, ws, scale: float, block_mask,
                        causal: bool = False, stream=None):
    B, H, n_q, d = q.shape
    n_kv = k.shape[2]
    mp, per_head = _mask_args(block_mask, B, H)
    _check(load_library().fa_bwd_block_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), _nbytes(ws), B,
                                              H, n_q, n_kv, d, float(scale), int(bool(causal)), mp,
                                              per_head, _stream(stream)))


def fa_fwd_fp8(q8, k8, v8, o, lse, scale: float, descale_q: float, descale_k: float,
               descale_v: float, causal: bool = False, stream=None):
    """q8, k8, v8: e4m3 codes (uint8 or float8_e4m3fn tensors) [B,H,N,d]; o bf16, lse fp32."""
    B, H, n_q, d = q8.shape
    n_kv = k8.shape[2]
    _check(load_library().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(o), _ptr(lse), B, H, n_q,
                                     n_kv, d, float(scale), float(descale_q), float(descale_k),
                                     float(descale_v), int(bool(causal)), _stream(stream)))


def fa_decode_paged(q, k_cache, v_cache, o, lse, block_table, seqlens_k, max_seqlen_k: int,
                    scale: float, n_splits: int, ws, stream=None):
    """q [B,H,1,d]; k/v cache [num_blocks, block_size, H, d]; block_table [B, max_blocks] int32;
    seqlens_k [B] int32 (both on the device)."""
    B, H, _, d = q.shape
    num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load_library().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                          _ptr(block_table), _ptr(seqlens_k), B, H,
                                          block_table.shape[1], block_size, num_blocks,
                                          int(max_seqlen_k), d, float(scale), int(n_splits),
                                          _ptr(ws), ws_bytes, _stream(stream)))


def fa_debug_counters(counters):
    """Point the diagnostic tile counters at ``counters`` (a uint64/int64 device tensor of >= 2
    entries), or turn them off with None (see include/fa.h)."""
    _check(load_library().fa_debug_counters(None if counters is None else _ptr(counters)))


def fa_sync_status(stream=None):
    _check(load_library().fa_sync_status(_stream(stream)))


def fa_selftest_wait_timeout(limit_us: int, stream=None):
    """Enqueue the diagnostic bounded wait (see include/fa.h); check it with fa_sync_status()."""
    _check(load_library().fa_selftest_wait_timeout(int(limit_us), _stream(stream)))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


def fa_last_error_message() -> str:
    return load_library().fa_last_error_message().decode()


# --------------------------------------------------------------------------------------------
# Convenience wrappers: torch allocates the outputs, the library computes them
# --------------------------------------------------------------------------------------------

def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Returns (O bf16 [B,H,N_q,d], lse fp32 [B,H,N_q])."""
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, stream=None,
             workspace=None):
    """Returns (dQ, dK, dV) in bf16."""
    import torch
    B, H, n_q, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    need = fa_bwd_workspace_size(B, H, n_q, k.shape[2], d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, scale, causal, stream)
    return dq, dk, dv


def decode(q, k, v, n_splits: int = 0, scale: float | None = None, stream=None, workspace=None):
    """Single-query split-KV decode: q [B,H,1,d], k/v [B,H,N_kv,d] -> (O [B,H,1,d], lse [B,H,1])."""
    import torch
    B, H, _, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    need = fa_decode_workspace_size(B, H, k.shape[2], d, n_splits)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    fa_decode_splitkv(q, k, v, o, lse, scale, n_splits, workspace, stream)
    return o, lse


def decode_paged(q, k_cache, v_cache, block_table, seqlens_k, max_seqlen_k: int, n_splits: int = 0,
                 scale: float | None = None, stream=None, workspace=None):
    """Split-KV decode over a paged cache -> (O [B,H,1,d], lse [B,H,1])."""
    import torch
    B, H, _, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    need = fa_decode_workspace_size(B, H, max_seqlen_k, d, n_splits)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    fa_decode_paged(q, k_cache, v_cache, o, lse, block_table, seqlens_k, max_seqlen_k, scale,
                    n_splits, workspace, stream)
    return o, lse


def forward_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float,
                causal: bool = False, scale: float | None = None, stream=None):
    """FP8 forward -> (O bf16 [B,H,N_q,d], lse fp32 [B,H,N_q])."""
    import torch
    B, H, n_q, d = q8.shape
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty((B, H, n_q, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q8.device)
    fa_fwd_fp8(q8, k8, v8, o, lse, scale, descale_q, descale_k, descale_v, causal, stream)
    return o, lse


def forward_window(q, k, v, window_left: int, window_right: int, scale: float | None = None,
                   stream=None):
    """Sliding-window forward: query i sees keys i - window_left .. i + window_right (a negative
    bound is unbounded) -> (O, lse)."""
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa_fwd_window(q, k, v, o, lse, scale, window_left, window_right, stream)
    return o, lse


def backward_window(q, k, v, o, lse, do, window_left: int, window_right: int,
                    scale: float | None = None, stream=None, workspace=None):
    import torch
    B, H, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    need = fa_bwd_workspace_size(B, H, N, N, d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_window(q, k, v, o, lse, do, dq, dk, dv, workspace, scale, window_left, window_right, stream)
    return dq, dk, dv


def forward_block_sparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None,
                         stream=None):
    """Block-sparse forward (blocks of 128 x 128; see fa_fwd_block_sparse) -> (O, lse)."""
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa_fwd_block_sparse(q, k, v, o, lse, scale, block_mask, causal, stream)
    return o, lse


def backward_block_sparse(q, k, v, o, lse, do, block_mask, causal: bool = False,
                          scale: float | None = None, stream=None, workspace=None):
    """Block-sparse backward -> (dQ, dK, dV) in bf16."""
    import torch
    B, H, n_q, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    need = fa_bwd_workspace_size(B, H, n_q, k.shape[2], d)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_block_sparse(q, k, v, o, lse, do, dq, dk, dv, workspace, scale, block_mask, causal, stream)
    return dq, dk, dv
