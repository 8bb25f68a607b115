"""Algorithmic work and traffic counts used for throughput and roofline figures.

Counts follow "FlashAttention and online softmax" (ML Systems lesson 4):
  * forward FLOP = 4 d * pairs per head (QK^T and PV, 2 N^2 d each; section 3 "HBM traffic",
    "The roofline view");
  * backward FLOP = 10 d * pairs per head (four matmuls plus the recomputation of S; section 3
    "Backward pass: recompute instead of store", "FLOPs");
  * pairs = N_q * N_kv, or N (N + 1) / 2 visible (query, key) pairs when causal ("Causal masks");
  * causal tiles computed = T (T + 1) / 2 of T^2 ("Causal masks");
  * standard traffic 4 N^2 + 4 N d and tiled traffic 2 N d + 2 N^2 d / B_r elements per head
    (section 3 "HBM traffic").
"""
from __future__ import annotations


def pairs(n_q: int, n_kv: int, causal: bool) -> int:
    if causal:
        assert n_q == n_kv
        return n_q * (n_q + 1) // 2
    return n_q * n_kv


def fwd_flops(B: int, H: int, n_q: int, n_kv: int, d: int, causal: bool) -> int:
    return 4 * d * pairs(n_q, n_kv, causal) * B * H


def bwd_flops(B: int, H: int, n_q: int, n_kv: int, d: int, causal: bool) -> int:
    return 10 * d * pairs(n_q, n_kv, causal) * B * H


def causal_tiles(n: int, tile: int) -> int:
    t = -(-n // tile)
    return t * (t + 1) // 2


def standard_traffic_elements(n: int, d: int) -> int:
    return 4 * n * n + 4 * n * d


def tiled_traffic_elements(n: int, d: int, b_r: int) -> float:
    return 2 * n * d + 2 * n * n * d / b_r


def decode_bytes(B: int, H: int, n_kv: int, d: int) -> int:
    """Algorithmic HBM bytes of one decode call: K and V (bf16), q and O (bf16), lse (fp32)."""
    return 2 * B * H * n_kv * d * 2 + 2 * B * H * d * 2 + 4 * B * H


def decode_partial_bytes(B: int, H: int, d: int, n_splits: int) -> int:
    """Extra bytes of the split/merge exchange: (m, l, o~) fp32 written once and read once."""
    return 2 * B * H * n_splits * (d + 2) * 4


def fwd_bytes(B: int, H: int, n_q: int, n_kv: int, d: int) -> int:
    """Compulsory HBM bytes of the forward: read Q, K, V, write O (bf16) and lse (fp32)."""
    return (2 * n_q + 2 * n_kv) * d * 2 * B * H + 4 * n_q * B * H


def bwd_bytes(B: int, H: int, n_q: int, n_kv: int, d: int) -> int:
    """Compulsory HBM bytes of the backward: read Q, K, V, O, dO, lse; write dQ, dK, dV."""
    return (3 * n_q + 2 * n_kv + 2 * n_kv + n_q) * d * 2 * B * H + 4 * n_q * B * H


def window_pairs(n: int, left: int, right: int) -> int:
    """Visible (query, key) pairs of one head under the window i - left <= j <= i + right over
    n positions (a negative bound is unbounded): sum over i of the clipped window width."""
    total = 0
    lo_w = n if left < 0 else left
    hi_w = n if right < 0 else right
    for i in range(n):
        total += min(n - 1, i + hi_w) - max(0, i - lo_w) + 1
    return total


def window_fwd_flops(B: int, H: int, n: int, d: int, left: int, right: int) -> int:
    return 4 * d * window_pairs(n, left, right) * B * H


def window_bwd_flops(B: int, H: int, n: int, d: int, left: int, right: int) -> int:
    return 10 * d * window_pairs(n, left, right) * B * H


def block_sparse_pairs(block_mask, n_q: int, n_kv: int, causal: bool, block: int = 128) -> int:
    """Visible (query, key) pairs under a 0/1 block mask ([n_qblocks, n_kblocks] for one head,
    or [..., n_qblocks, n_kblocks] summed over the leading axes), with causal (n_q == n_kv) also
    j <= i: per set block its clipped rows x columns, a diagonal block only its lower triangle."""
    import numpy as np
    m = np.asarray(block_mask).astype(bool)
    m = m.reshape(-1, m.shape[-2], m.shape[-1]).sum(axis=0)   # set count per block over heads
    total = 0
    for qb in range(m.shape[0]):
        rows = min(block, n_q - qb * block)
        for kb in range(m.shape[1]):
            if not m[qb, kb]:
                continue
            cols = min(block, n_kv - kb * block)
            if causal and kb > qb:
                continue
            if causal and kb == qb:
                per = sum(min(i + 1, cols) for i in range(rows))
            else:
                per = rows * cols
            total += int(m[qb, kb]) * per
    return total
