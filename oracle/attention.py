"""CPU fp64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this module.  The library's product path never calls it, and it shares no code with the CUDA
kernels (no headers, helpers or constants).

Pages cited (by title and section):
  [Lesson4]  "FlashAttention and online softmax", ML Systems lesson 4 (learn.mohebi.ai).
  [Scratch]  "FlashAttention from Scratch -- The Paradox of Doing More Math to Go Faster"
             (ta-paperlens).

What the oracle computes.  The pages state that the tiled method is exact: it reaches the plain
definition of attention, only reordered (Lesson4 §3 "The online softmax theorem", proof step 4;
Lesson4 §7 "Common mistakes": "It is exact").  So the oracle for the forward and backward passes
is that plain definition, with an explicit N_q x N_kv score matrix per head:

  S = tau * Q K^T (causal: S_ij = -inf for j > i)               [Lesson4 §2 table, step 1]
  three-pass safe softmax per row: m = max S, l = sum e^{S-m},
  P = e^{S-m} / l                                                [Lesson4 §2 "One query, one pass"]
  O = P V ; lse = m + ln l                                       [Lesson4 §2 "The GPU picture"]
  dV = P^T dO ; dP = dO V^T ; D_i = sum_j P_ij dP_ij ;
  dS = P o (dP - D) ; dQ = tau dS K ; dK = tau dS^T Q           [Lesson4 §3 "Backward pass"]

The online recurrence (Lesson4 §3 theorem) and the merge of two partial results (Lesson4 §3
"Merging two partial results") are also written out, step by step in the pages' notation; the
tests use them for the pages' worked examples, the decode check and the online = three-pass
theorem.  The matmuls are NumPy library calls; nothing else is blocked, fused or reordered.

Every function here is pinned by ``tests/test_oracle.py`` against values the pages print,
closed forms, invariants, independent library routines (scipy's softmax, torch's fp64 SDPA and
autograd) and finite differences.

Readings where the pages leave a step open:
  * tau is the caller's ``scale`` (one page prints QK^T/d, having lost the square root);
  * causal means query i sees keys j <= i, with N_q == N_kv (Lesson4 "Causal masks");
  * a row that sees no key has lse = -inf and O = 0, never NaN (Lesson4 §3 "Compute it stably");
  * lse is the natural logarithm;
  * block-sparse attention (Scratch "Results" names it, with no pattern) is the plain definition
    under a 0/1 mask over (query block, key block) pairs, ANDed with the causal mask if asked.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _as_f64(x) -> np.ndarray:
    """Exact upcast: bf16/fp32 torch tensors or arrays -> fp64 NumPy."""
    try:
        import torch  # local import: the oracle itself needs only NumPy
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------------
# Softmax pieces
# --------------------------------------------------------------------------------------------

def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool) -> np.ndarray:
    """S = tau Q K^T for one head, [N_q, N_kv]; causal entries j > i set to -inf.

    [Lesson4 §2 "The GPU picture", table row 1; Lesson4 "Causal masks": query i sees keys j <= i]
    """
    s = scale * (q @ k.T)
    if causal:
        n_q, n_kv = s.shape
        i = np.arange(n_q)[:, None]
        j = np.arange(n_kv)[None, :]
        s = np.where(j <= i, s, NEG_INF)
    return s


def three_pass_softmax(s: np.ndarray):
    """Row-wise safe softmax in three passes; returns (P, m, l).

    Pass 1 finds the row max m, pass 2 sums e^{s-m}, pass 3 forms the weights.
    [Lesson4 §2 "One query, one pass": "Why subtract the max" and "The problem"]
    A row with no visible score (all -inf) gets m = -inf, l = 0 and P = 0.
    """
    m = s.max(axis=-1) if s.shape[-1] > 0 else np.full(s.shape[:-1], NEG_INF)   # pass 1
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[..., None])                                           # e^{-inf} = 0
    l = e.sum(axis=-1)                                                          # pass 2
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(l[..., None] > 0, e / np.where(l > 0, l, 1.0)[..., None], 0.0)  # pass 3
    return p, m, l


def lse_from(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """lse = m + ln l, the per-row logsumexp; -inf for rows with no visible key.

    [Lesson4 §2 "The GPU picture": lse_i = m_i + log l_i]
    """
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)


# --------------------------------------------------------------------------------------------
# Forward / backward, plain definition
# --------------------------------------------------------------------------------------------

def forward_head(q, k, v, scale: float, causal: bool):
    """One head: O = softmax(tau Q K^T) V and lse.  Returns (O, lse, P)."""
    s = scores(q, k, scale, causal)
    p, m, l = three_pass_softmax(s)
    o = p @ v
    return o, lse_from(m, l), p


def forward(q, k, v, scale: float, causal: bool = False):
    """Attention forward over [B, H, N, d] inputs; returns fp64 (O [B,H,N_q,d], lse [B,H,N_q])."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, n_q, d = q.shape
    o = np.zeros((B, H, n_q, v.shape[-1]))
    lse = np.full((B, H, n_q), NEG_INF)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h], _ = forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


def backward_head(q, k, v, do, scale: float, causal: bool):
    """One head, analytic gradients of L = sum(dO o O).  Returns (dQ, dK, dV, D).

    [Lesson4 §3 "Backward pass: recompute instead of store", steps 1-4; D is formed as
    sum_j P_ij dP_ij, its definition, so that the identity D = rowsum(dO o O) stays a test.]
    """
    _, _, p = forward_head(q, k, v, scale, causal)
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=-1)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, D


def backward(q, k, v, do, scale: float, causal: bool = False):
    """Attention backward over [B, H, N, d]; returns fp64 (dQ, dK, dV, D)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, n_q, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros((B, H, n_q))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h], D[b, h] = backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv, D


def forward_rows(q_rows, row_index, k, v, scale: float, causal: bool):
    """Forward for selected query rows of one head (full-size sampling).

    ``row_index`` gives each row's position i in the sequence; with ``causal`` the row sees keys
    j <= i.  Same definition as ``forward_head``, evaluated for a subset of independent rows.
    """
    q_rows, k, v = _as_f64(q_rows), _as_f64(k), _as_f64(v)
    s = scale * (q_rows @ k.T)
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= np.asarray(row_index)[:, None], s, NEG_INF)
    p, m, l = three_pass_softmax(s)
    return p @ v, lse_from(m, l)


def backward_sampled(q, k, v, do, scale: float, causal: bool, q_rows, k_rows, block: int = 1024):
    """Gradients of one head at selected rows: dQ at query rows ``q_rows``, dK and dV at key
    rows ``k_rows`` (for full-size checks where whole N x N matrices do not fit).

    Same definition as ``backward_head``, evaluated for subsets.  Every query row's lse_i and
    D_i = sum_j P_ij dP_ij is needed; they are formed row by row (rows are independent) in
    blocks of ``block`` rows.  Then P_ij = e^{S_ij - lse_i} on the needed rows / columns
    [Lesson4 §3 "Backward pass", step 1: the lse already holds the max and the sum].
    Returns (dQ [len(q_rows), d], dK [len(k_rows), d], dV [len(k_rows), d]).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    n_q = q.shape[0]
    q_rows = np.asarray(q_rows)
    k_rows = np.asarray(k_rows)
    lse = np.empty(n_q)
    D = np.empty(n_q)
    for r0 in range(0, n_q, block):
        rows = np.arange(r0, min(n_q, r0 + block))
        s = scale * (q[rows] @ k.T)
        if causal:
            s = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None], s, NEG_INF)
        p, m, l = three_pass_softmax(s)
        lse[rows] = lse_from(m, l)
        D[rows] = (p * (do[rows] @ v.T)).sum(axis=-1)

    def probs(rows, cols):
        s = scale * (q[rows] @ k[cols].T)
        if causal:
            s = np.where(cols[None, :] <= rows[:, None], s, NEG_INF)
        return np.exp(s - lse[rows][:, None])

    all_q = np.arange(n_q)
    all_k = np.arange(k.shape[0])
    p = probs(q_rows, all_k)
    ds = p * (do[q_rows] @ v.T - D[q_rows][:, None])
    dq = scale * (ds @ k)
    pc = probs(all_q, k_rows)
    dsc = pc * (do @ v[k_rows].T - D[:, None])
    dv = pc.T @ do
    dk = scale * (dsc.T @ q)
    return dq, dk, dv


# --------------------------------------------------------------------------------------------
# Online recurrence and merge (the method's own steps, pages' notation)
# --------------------------------------------------------------------------------------------

def online_step(m_prev, l_prev, o_prev, x_blk, v_blk):
    """One block of the online softmax recurrence for one query row.

    m_j = max(m_{j-1}, max_i x_i);  l_j = e^{m_{j-1}-m_j} l_{j-1} + sum_i e^{x_i - m_j};
    o_j = e^{m_{j-1}-m_j} o_{j-1} + sum_i e^{x_i - m_j} v_i.
    [Lesson4 §3 "The online softmax theorem"; the -inf start follows proof step 2]
    Returns (m_j, l_j, o_j, factor).
    """
    x_blk = np.asarray(x_blk, dtype=np.float64)
    v_blk = np.asarray(v_blk, dtype=np.float64)
    m_new = max(m_prev, float(x_blk.max())) if x_blk.size else m_prev
    if m_new == NEG_INF:                       # nothing visible yet: state stays empty
        return m_new, l_prev, o_prev, 1.0
    factor = math.exp(m_prev - m_new) if m_prev != NEG_INF else 0.0
    w = np.exp(x_blk - m_new)
    l_new = factor * l_prev + w.sum()
    o_new = factor * np.asarray(o_prev, dtype=np.float64) + np.tensordot(w, v_blk, axes=(0, 0))
    return m_new, l_new, o_new, factor


def online_softmax(x, v, block_bounds):
    """Run the recurrence over the blocks [b0:b1) given by ``block_bounds``.

    Returns (m_T, l_T, o_T, trace) where trace lists (factor, l_j, o_j) per block.
    """
    x = np.asarray(x, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m, l = NEG_INF, 0.0
    o = np.zeros(v.shape[1:]) if v.ndim > 1 else 0.0
    trace = []
    for b0, b1 in block_bounds:
        m, l, o, f = online_step(m, l, o, x[b0:b1], v[b0:b1])
        trace.append((f, l, o))
    return m, l, o, trace


def merge(o_a, lse_a, o_b, lse_b):
    """Merge two partial results over disjoint key sets.

    lse = log(e^{lse_A} + e^{lse_B}) computed as max + log1p(e^{-|diff|});
    o = e^{lse_A - lse} o_A + e^{lse_B - lse} o_B.  An empty set has lse = -inf and weight 0;
    two empty sets give o = 0, lse = -inf.
    [Lesson4 §3 "Merging two partial results" and "Compute it stably"]
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    if lse_a == NEG_INF and lse_b == NEG_INF:
        return np.zeros_like(o_a), NEG_INF
    if lse_a == NEG_INF:
        return o_b.copy(), float(lse_b)
    if lse_b == NEG_INF:
        return o_a.copy(), float(lse_a)
    hi = max(lse_a, lse_b)
    lse = hi + math.log1p(math.exp(-abs(lse_a - lse_b)))
    return math.exp(lse_a - lse) * o_a + math.exp(lse_b - lse) * o_b, lse


# --------------------------------------------------------------------------------------------
# Split-KV decode
# --------------------------------------------------------------------------------------------

def decode_partials(q, k, v, scale: float, n_splits: int):
    """Per-chunk state of split-KV decode for one head and one query row.

    The key axis is cut into ``n_splits`` contiguous chunks of ceil(N_kv / n_splits) keys
    (the last may be shorter or empty).  Each chunk's state (m_c, l_c, o~_c) is the online
    state after that chunk alone, i.e. its max, its sum of e^{x-m_c} and its unnormalised
    weighted sum.  [Lesson4 §3 "Split-KV for decoding (flash-decoding)"; the (m, l, o~) triple
    is the theorem's state]
    Returns arrays m [n], l [n], o [n, d].
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    n_kv, d = k.shape
    chunk = -(-n_kv // n_splits) if n_kv else 0
    m = np.full(n_splits, NEG_INF)
    l = np.zeros(n_splits)
    o = np.zeros((n_splits, v.shape[-1]))
    x = scale * (k @ q.reshape(-1))
    for c in range(n_splits):
        lo, hi = c * chunk, min(n_kv, (c + 1) * chunk)
        if hi <= lo:
            continue
        mc, lc, oc, _ = online_step(NEG_INF, 0.0, np.zeros(v.shape[-1]), x[lo:hi], v[lo:hi])
        m[c], l[c], o[c] = mc, lc, oc
    return m, l, o


def decode_merge(m, l, o):
    """Merge k per-chunk states: m = max m_c, l = sum e^{m_c-m} l_c, O = sum e^{m_c-m} o~_c / l.

    Equivalent to folding the pairwise merge over the chunks (each chunk's lse is
    m_c + ln l_c and its normalised output o~_c / l_c).  Empty chunks (m_c = -inf) weigh 0.
    [Lesson4 §3 "Merging two partial results"; "Split-KV for decoding"]
    Returns (O [d], lse).
    """
    m = np.asarray(m, dtype=np.float64)
    live = np.isfinite(m)
    if not live.any():
        return np.zeros(np.asarray(o).shape[-1]), NEG_INF
    mm = m[live].max()
    w = np.where(live, np.exp(np.where(live, m, mm) - mm), 0.0)
    l_tot = (w * np.asarray(l)).sum()
    o_tot = (w[:, None] * np.asarray(o)).sum(axis=0) / l_tot
    return o_tot, mm + math.log(l_tot)


def decode(q, k, v, scale: float):
    """Decode reference by the plain definition: one query row over all keys of each head.

    q [B,H,1,d], k/v [B,H,N_kv,d] -> (O [B,H,1,d], lse [B,H,1]).
    """
    return forward(q, k, v, scale, causal=False)


# --------------------------------------------------------------------------------------------
# FP8 forward
# --------------------------------------------------------------------------------------------
# The pages name low precision (FP8) as one of FlashAttention-3's techniques and give no
# formula for it ([Lesson4] "Causal masks and FlashAttention-3"; [Scratch] "Later versions").
# Reading taken: Q, K and V arrive as 8-bit e4m3 codes with one scale per tensor, x = s_x * x8,
# and the result is exact attention of those dequantized tensors.  How the kernel rounds its
# intermediate weights is the kernel's business; its accuracy bar is set against this result.

def decode_e4m3(codes) -> np.ndarray:
    """Value of each 8-bit e4m3 code: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def forward_fp8(q8, k8, v8, scale: float, descale_q: float, descale_k: float, descale_v: float,
                causal: bool = False):
    """Attention of the dequantized tensors s_q Q8, s_k K8, s_v V8 (codes as uint8 arrays or
    tensors of shape [B, H, N, d]); returns fp64 (O, lse) as ``forward``."""
    def deq(x, s):
        try:
            import torch
            if isinstance(x, torch.Tensor):
                x = x.detach().cpu().view(torch.uint8).numpy()
        except ImportError:  # pragma: no cover
            pass
        return decode_e4m3(x) * float(s)
    return forward(deq(q8, descale_q), deq(k8, descale_k), deq(v8, descale_v), scale, causal)


# --------------------------------------------------------------------------------------------
# Sliding-window attention
# --------------------------------------------------------------------------------------------
# The pages name sliding-window masks, next to causal ones, as what long-context training uses,
# with the same tile skipping ([Lesson4] section 6 "Where it shows up", Training).  Reading
# taken: query i sees key j iff i - left <= j <= i + right, over one sequence (N_q == N_kv); a
# negative bound is unbounded on that side, so (left, right) = (-1, 0) is the causal mask and
# (-1, -1) no mask.  Everything else is the plain definition with those scores at -inf.

def window_visible(n_q: int, n_kv: int, left: int, right: int) -> np.ndarray:
    """Boolean [n_q, n_kv]: True where key j is inside query i's window."""
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    vis = np.ones((n_q, n_kv), dtype=bool)
    if left >= 0:
        vis &= j >= i - left
    if right >= 0:
        vis &= j <= i + right
    return vis


def forward_window_head(q, k, v, scale: float, left: int, right: int):
    """One head under a sliding window: returns (O, lse, P)."""
    s = scale * (q @ k.T)
    s = np.where(window_visible(q.shape[0], k.shape[0], left, right), s, NEG_INF)
    p, m, l = three_pass_softmax(s)
    return p @ v, lse_from(m, l), p


def forward_window(q, k, v, scale: float, left: int, right: int):
    """Sliding-window forward over [B, H, N, d]; fp64 (O, lse)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, n_q, d = q.shape
    o = np.zeros((B, H, n_q, v.shape[-1]))
    lse = np.full((B, H, n_q), NEG_INF)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h], _ = forward_window_head(q[b, h], k[b, h], v[b, h], scale, left, right)
    return o, lse


def backward_window(q, k, v, do, scale: float, left: int, right: int):
    """Sliding-window gradients: the backward formulas of ``backward_head`` with the window's P
    (masked scores have P = 0, so they contribute nothing)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            _, _, p = forward_window_head(q[b, h], k[b, h], v[b, h], scale, left, right)
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            D = (p * dp).sum(axis=-1)
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def forward_window_rows(q_rows, row_index, k, v, scale: float, left: int, right: int):
    """Sliding-window forward for selected query rows of one head (full-size sampling); the
    same definition as ``forward_window_head`` evaluated for a subset of independent rows."""
    q_rows, k, v = _as_f64(q_rows), _as_f64(k), _as_f64(v)
    s = scale * (q_rows @ k.T)
    i = np.asarray(row_index)[:, None]
    j = np.arange(k.shape[0])[None, :]
    vis = np.ones(s.shape, dtype=bool)
    if left >= 0:
        vis &= j >= i - left
    if right >= 0:
        vis &= j <= i + right
    p, m, l = three_pass_softmax(np.where(vis, s, NEG_INF))
    return p @ v, lse_from(m, l)


# --------------------------------------------------------------------------------------------
# Block-sparse attention
# --------------------------------------------------------------------------------------------
# [Scratch] "Results" names a block-sparse variant of the method (the same IO-aware tiling
# applied to a sparse pattern) without fixing a pattern.  Reading taken: a 0/1 mask over
# (query block, key block) pairs of a fixed block size; attention is the plain definition over
# the keys of the set blocks, and with ``causal`` also only j <= i ([Lesson4] "Causal masks");
# a row that sees no key gets O = 0 and lse = -inf, as for an empty key set.  The mask is either
# one [n_qblocks, n_kblocks] array for every head or one per head, [B, H, n_qblocks, n_kblocks].

def block_visible(block_mask, n_q: int, n_kv: int, block: int, causal: bool) -> np.ndarray:
    """Boolean [n_q, n_kv]: True where mask[i // block, j // block] is set (and j <= i if causal)."""
    bm = np.asarray(block_mask).astype(bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_kv)[None, :]
    vis = bm[i // block, j // block]
    if causal:
        vis = vis & (j <= i)
    return vis


def _mask_of_head(block_mask, b: int, h: int):
    m = np.asarray(block_mask)
    return m if m.ndim == 2 else m[b, h]


def forward_block_sparse_head(q, k, v, scale: float, block_mask, block: int, causal: bool):
    """One head under a block mask: returns (O, lse, P)."""
    s = scale * (q @ k.T)
    s = np.where(block_visible(block_mask, q.shape[0], k.shape[0], block, causal), s, NEG_INF)
    p, m, l = three_pass_softmax(s)
    return p @ v, lse_from(m, l), p


def forward_block_sparse(q, k, v, scale: float, block_mask, causal: bool = False, block: int = 128):
    """Block-sparse forward over [B, H, N, d]; fp64 (O, lse)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, n_q, _ = q.shape
    o = np.zeros((B, H, n_q, v.shape[-1]))
    lse = np.full((B, H, n_q), NEG_INF)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h], _ = forward_block_sparse_head(
                q[b, h], k[b, h], v[b, h], scale, _mask_of_head(block_mask, b, h), block, causal)
    return o, lse


def backward_block_sparse(q, k, v, do, scale: float, block_mask, causal: bool = False,
                          block: int = 128):
    """Block-sparse gradients: the backward formulas of ``backward_head`` with the masked P
    (scores outside the set blocks have P = 0 and contribute nothing)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            _, _, p = forward_block_sparse_head(q[b, h], k[b, h], v[b, h], scale,
                                                _mask_of_head(block_mask, b, h), block, causal)
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            D = (p * dp).sum(axis=-1)
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def forward_block_sparse_rows(q_rows, row_index, k, v, scale: float, block_mask, causal: bool,
                              block: int = 128):
    """Block-sparse forward for selected query rows of one head (full-size sampling): the same
    definition as ``forward_block_sparse_head`` evaluated for a subset of independent rows."""
    q_rows, k, v = _as_f64(q_rows), _as_f64(k), _as_f64(v)
    s = scale * (q_rows @ k.T)
    i = np.asarray(row_index)[:, None]
    j = np.arange(k.shape[0])[None, :]
    vis = np.asarray(block_mask).astype(bool)[i // block, j // block]
    if causal:
        vis = vis & (j <= i)
    p, m, l = three_pass_softmax(np.where(vis, s, NEG_INF))
    return p @ v, lse_from(m, l)
