"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and the benchmark.

This module holds no attention arithmetic: it only draws random tensors and names the
workload shapes.  Both sides of every parity check receive the same bytes from here.

Recipe (the same for every workload):
  * a ``torch.Generator`` seeded with ``seed``; Q, K, V and dO are drawn in that order as
    fp32 ``randn`` of shape [B, H, N, d] and rounded to bf16 (round-to-nearest-even);
  * values are i.i.d. N(0, 1);
  * the long-sequence workload additionally scales ``round(frac * N_kv)`` K rows per (b, h)
    by 8 (an exact power of two, applied after the bf16 rounding), the rows chosen by a
    seeded ``randperm`` drawn after dO.  Large keys force big jumps of the running row max.

Workloads are small-to-large versions of the shapes the attention pages discuss (a GPT-2-medium
attention layer, a long 16K sequence, single-token decode over a 32K KV cache).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N_q: int
    N_kv: int
    d: int
    causal: bool
    seed: int
    outlier_frac: float = 0.0
    n_splits: int = 0          # decode only

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def describe(self) -> str:
        kind = "decode" if self.N_q == 1 and self.n_splits else ("causal" if self.causal else "non-causal")
        return (f"{self.name}: B={self.B} H={self.H} N_q={self.N_q} N_kv={self.N_kv} d={self.d} "
                f"{kind}" + (f" splits={self.n_splits}" if self.n_splits else ""))


# The five workloads.  Seeds are 1000 + index.
TINY = Workload("tiny_1x1x128x64", 1, 1, 128, 128, 64, False, 1000)
GPT2M = Workload("gpt2m_8x16x1024x64_causal", 8, 16, 1024, 1024, 64, True, 1001)
HEADLINE = Workload("attn_4x32x4096x128", 4, 32, 4096, 4096, 128, False, 1002)
HEADLINE_CAUSAL = dataclasses.replace(HEADLINE, name="attn_4x32x4096x128_causal", causal=True)
LONG = Workload("long_1x16x16384x128_causal_outliers", 1, 16, 16384, 16384, 128, True, 1003,
                outlier_frac=0.01)
DECODE = Workload("decode_64x32x32768x128_splits64", 64, 32, 1, 32768, 128, False, 1004,
                  n_splits=64)

ALL = (TINY, GPT2M, HEADLINE, HEADLINE_CAUSAL, LONG, DECODE)


def _draw(gen: torch.Generator, shape, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def make_qkv(B: int, H: int, N_q: int, N_kv: int, d: int, seed: int, *,
             outlier_frac: float = 0.0, with_do: bool = True, device: str = "cpu"):
    """Return dict(q, k, v[, do]) of contiguous bf16 tensors [B, H, N, d].

    ``device='cuda'`` draws with a CUDA generator (different numbers from the CPU draw, same
    recipe); it is used only where a host draw would take minutes (the 34 GB decode cache).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {
        "q": _draw(gen, (B, H, N_q, d), device),
        "k": _draw(gen, (B, H, N_kv, d), device),
        "v": _draw(gen, (B, H, N_kv, d), device),
    }
    if with_do:
        out["do"] = _draw(gen, (B, H, N_q, d), device)
    if outlier_frac > 0.0 and N_kv > 0:
        n_out = int(round(outlier_frac * N_kv))
        k = out["k"]
        for b in range(B):
            for h in range(H):
                rows = torch.randperm(N_kv, generator=gen, device=device)[:n_out]
                k[b, h, rows] = k[b, h, rows] * 8  # exact in bf16: a power of two
    return out


def make_workload(w: Workload, *, with_do: bool = True, device: str = "cpu"):
    return make_qkv(w.B, w.H, w.N_q, w.N_kv, w.d, w.seed, outlier_frac=w.outlier_frac,
                    with_do=with_do, device=device)


FP8_E4M3_MAX = 448.0


def make_qkv_fp8(B: int, H: int, N_q: int, N_kv: int, d: int, seed: int, *, device: str = "cpu"):
    """FP8 inputs: the same fp32 ``randn`` draws as ``make_qkv`` (Q, K, V in that order), each
    tensor given one scale s = amax / 448 and cast to e4m3 (round-to-nearest-even) as x / s.

    Returns dict(q8, k8, v8 = uint8 code tensors [B, H, N, d]; descale_q, descale_k,
    descale_v = the scales s as Python floats).  Dequantized value = s * e4m3(code).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {}
    for name, n in (("q", N_q), ("k", N_kv), ("v", N_kv)):
        x = torch.randn((B, H, n, d), generator=gen, dtype=torch.float32, device=device)
        amax = float(x.abs().max()) if x.numel() else 1.0
        s = amax / FP8_E4M3_MAX if amax > 0 else 1.0
        out[name + "8"] = (x / s).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        out["descale_" + name] = s
    return out


def make_block_mask(n_qblocks: int, n_kblocks: int, seed: int, *, band: int = 1, n_global: int = 1,
                    p_random: float = 0.05, heads: tuple[int, int] | None = None) -> torch.Tensor:
    """Seeded 0/1 block pattern (uint8, CPU) of the kind block-sparse attention is used with: a
    band of ``band`` blocks either side of the diagonal, the first ``n_global`` key blocks for
    every query block, and each other block with probability ``p_random``.  ``heads = (B, H)``
    gives one independent pattern per head, [B, H, n_qblocks, n_kblocks]."""
    gen = torch.Generator().manual_seed(seed)
    shape = ((*heads, n_qblocks, n_kblocks) if heads else (n_qblocks, n_kblocks))
    m = torch.rand(shape, generator=gen) < p_random
    i = torch.arange(n_qblocks)[:, None]
    j = torch.arange(n_kblocks)[None, :]
    m |= (j - i).abs() <= band
    m |= j < n_global
    return m.to(torch.uint8)


def make_varlen_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> list[int]:
    """Seeded sequence lengths, uniform in [lo, hi], for a packed variable-length batch."""
    gen = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n_seqs,), generator=gen)]


def make_packed(total: int, H: int, d: int, seed: int, *, device: str, with_do: bool = True):
    """Packed token-major [total, H, d] Q, K, V (and dO): fp32 N(0,1) draws from a seeded CUDA
    generator rounded to bf16 (the recipe of ``make_qkv``, drawn on the device because benchmark
    batches are large)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    names = ("q", "k", "v", "do") if with_do else ("q", "k", "v")
    return {n: torch.randn((total, H, d), generator=gen, device=device).to(torch.bfloat16) for n in names}
