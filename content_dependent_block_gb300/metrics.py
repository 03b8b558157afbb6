"""Algorithmic work counts used by the benchmark's roofline.

FLOP convention (page "sparse-attention-triton-bench", Key finding and
Two-stage block indexer: 87.2B sparse vs 2.24T dense FLOPs at N=32768,
B=64, k=16, heads=8, d=64; 1,024 tokens per query):

  per query score against one key   : 2d (q.k) + 2d (p.v) + 5 softmax ops
  sparse forward = N*H*[(4d+5)*k*B + 2d*nb]   (fine stage + coarse scoring)
  dense  forward = N^2*H*(4d+5)

This convention reproduces the page's printed figures exactly
(87,241,523,200 -> "87.2B"; 2,241,972,928,512 -> "2.24T"; ratio 3.89%).
Only selected work is credited: padding, the hi/lo split of the coarse
contraction and any recomputation are never counted.
"""
from __future__ import annotations


def sparse_flops(n: int, heads: int, d: int, key_block: int, topk: int) -> int:
    nb = -(-n // key_block)
    kk = min(topk, nb)
    return n * heads * ((4 * d + 5) * kk * key_block + 2 * d * nb)


def sparse_flops_split(n: int, heads: int, d: int, key_block: int, topk: int):
    """(tensor-core FLOPs, softmax FP32 ops) of the dynamic forward."""
    nb = -(-n // key_block)
    kk = min(topk, nb)
    mma = n * heads * (4 * d * kk * key_block + 2 * d * nb)
    soft = n * heads * 5 * kk * key_block
    return mma, soft


def dense_flops(n: int, heads: int, d: int) -> int:
    return n * n * heads * (4 * d + 5)


def pairs_flops(pairs: int, d: int) -> int:
    """FLOPs of attention over an explicit count of (query, key) pairs."""
    return pairs * (4 * d + 5)


def local_global_pairs(n: int, w: int, s: int) -> int:
    """Active (i, j) pairs of the local-window + global-stride mask, counted
    in closed form (page "yayme/CUDA-kernel", sparsity pattern)."""
    total = 0
    globals_ = (n - 1) // s + 1 if s > 0 else 0
    for i in range(n):
        lo = max(0, i - w) if w >= 0 else 1
        hi = min(n - 1, i + w) if w >= 0 else 0
        band = hi - lo + 1 if w >= 0 else 0
        if s > 0 and w >= 0:
            # global columns inside the band are already counted
            in_band = hi // s - (lo - 1) // s if lo > 0 else hi // s + 1
            total += band + globals_ - in_band
        else:
            total += band + globals_
    return total


def sliding_pairs(n: int, W: int) -> int:
    """Active pairs of the causal sliding window i-W < j <= i."""
    full = max(0, n - W)
    ramp = min(n, W)
    return full * W + ramp * (ramp + 1) // 2


def unique_bytes(n: int, heads: int, d: int, elem: int) -> int:
    """Compulsory HBM bytes of one forward: read Q, K, V once, write O."""
    return 4 * n * heads * d * elem


def format_si(x: float, digits: int) -> str:
    """Format like the page does: 87.2B, 2.24T."""
    for div, suf in ((1e12, "T"), (1e9, "B"), (1e6, "M")):
        if x >= div:
            return f"{x / div:.{digits}g}{suf}"
    return f"{x:.{digits}g}"
