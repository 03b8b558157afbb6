"""Seeded synthetic workloads for content-dependent block-sparse attention.

This module only draws numbers and names shapes: it holds none of the
method's arithmetic (no pooling, scoring, selection or softmax).  Both the
CUDA path (through the binding) and the CPU oracle consume the exact same
bytes produced here.

Recipe (the pages name no dataset; every tensor is synthetic):
  * one ``numpy.random.Generator(PCG64(seed))`` per workload, seed 0;
  * draw order Q, K-centres, K-noise, V, each float32 standard normal;
  * "planted" workloads build K as a per-block centre c_b ~ N(0, sigma^2)^d
    shared by the block's B keys plus i.i.d. N(0, 1) noise, so that block
    scores separate (page "sparse-attention-triton-bench", Two-stage block
    indexer: blocks are scored by their mean key);
  * bf16 workloads round the float32 draws to bfloat16 with
    round-to-nearest-even; the arrays handed out are the raw bf16 bit
    patterns (uint16), so nothing downstream re-rounds.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One attention problem: [bh, n, d] tensors plus the sparsity recipe."""

    name: str
    bh: int                 # batch * heads (batch is 1 everywhere)
    n: int                  # tokens
    d: int                  # head dim
    dtype: str              # "bf16" or "fp32"
    kind: str               # "dynamic" | "local_global" | "sliding"
    key_block: int = 64     # B: tokens per key block
    topk: int = 0           # k (dynamic only)
    centre_sigma: float = 0.0   # >0: planted block centres on K
    window: int = -1        # w for local_global
    stride: int = 0         # s for local_global
    sliding: int = 0        # W for sliding
    q_group: int = 1        # queries per list row (static lists)
    seed: int = 0
    note: str = ""
    # selection options (dynamic only): causal selection, the query's own
    # block always selected, per-(batch*head) budgets (empty: topk for all)
    causal: bool = False
    local_block: bool = False
    head_topk: tuple = ()
    # skewed lists: `popular` blocks spread over the sequence that nearly
    # every query selects (keys of those blocks shifted along channel 0,
    # queries shifted the same way); 0 = none
    popular: int = 0

    @property
    def has_options(self) -> bool:
        return self.causal or self.local_block or bool(self.head_topk)

    @property
    def nb(self) -> int:
        return (self.n + self.key_block - 1) // self.key_block


# The workloads the method is exercised on.  "tiny" and "ragged" shapes are
# parity cases only; the 32k one is the throughput configuration.
WORKLOADS = {
    "dyn_n1024": Workload(
        "dyn_n1024", bh=2, n=1024, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=4, note="iid N(0,1), 16 blocks, top-4, non-causal"),
    "local_global_n4096": Workload(
        "local_global_n4096", bh=1, n=4096, d=64, dtype="fp32",
        kind="local_global", key_block=16, q_group=16, window=32, stride=512,
        note="fp32, |i-j|<=32 or j%512==0, 16x16 active-tile lists"),
    "local_global_n4100": Workload(
        "local_global_n4100", bh=1, n=4100, d=64, dtype="fp32",
        kind="local_global", key_block=16, q_group=16, window=32, stride=512,
        note="as n4096 with a ragged 4-token tail"),
    "dyn_n8192": Workload(
        "dyn_n8192", bh=8, n=8192, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=16, centre_sigma=0.5,
        note="planted centres N(0,0.5^2), 128 blocks, top-16"),
    "dyn_n32768": Workload(
        "dyn_n32768", bh=8, n=32768, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=16, centre_sigma=0.5,
        note="planted centres, 512 blocks, top-16 (1024 tokens/query)"),
    "dyn_n32768_causal": Workload(
        "dyn_n32768_causal", bh=8, n=32768, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=16, centre_sigma=0.5, causal=True, local_block=True,
        note="as dyn_n32768; causal selection (blocks b <= i/64, keys j <= i), "
             "own block always selected"),
    "dyn_n32768_budgets": Workload(
        "dyn_n32768_budgets", bh=8, n=32768, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=16, centre_sigma=0.5, head_topk=(16, 12, 8, 4, 16, 12, 8, 4),
        note="as dyn_n32768; per-head budgets 16/12/8/4 (twice)"),
    "dyn_n32768_skew": Workload(
        "dyn_n32768_skew", bh=8, n=32768, d=64, dtype="bf16", kind="dynamic",
        key_block=64, topk=16, centre_sigma=0.5, popular=8,
        note="as dyn_n32768 plus 8 popular blocks nearly every query selects: "
             "skewed lists, a popular (head, range, block) bin holds ~30x the mean"),
    "dyn_n131072": Workload(
        "dyn_n131072", bh=8, n=131072, d=128, dtype="bf16", kind="dynamic",
        key_block=64, topk=32, centre_sigma=0.5,
        note="planted centres, 2048 blocks, top-32"),
    "sliding_n131072": Workload(
        "sliding_n131072", bh=8, n=131072, d=128, dtype="bf16",
        kind="sliding", key_block=64, q_group=128, sliding=4096,
        centre_sigma=0.5,
        note="same tensors as dyn_n131072; causal window W=4096 over "
             "64-token key blocks listed per 128-query tile"),
}


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (NaN kept)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    r = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Tensors:
    """Host copies of one workload's inputs, [bh, n, d] C-contiguous.

    For bf16 workloads q/k/v are uint16 bit patterns; for fp32 they are
    float32.  ``dtype`` says which.
    """

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dtype: str
    meta: dict = field(default_factory=dict)

    def as_f32(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        return bf16_bits_to_f32(a) if self.dtype == "bf16" else a


def generate(w: Workload, *, bh: Optional[int] = None, n: Optional[int] = None,
             seed: Optional[int] = None) -> Tensors:
    """Draw the workload's Q, K, V (optionally at an overridden bh / n).

    Draw order is Q, K-centres, K-noise, V from one PCG64 stream.
    """
    bh = w.bh if bh is None else bh
    n = w.n if n is None else n
    seed = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (bh, n, w.d)
    q = rng.standard_normal(shape, dtype=np.float32)
    nb = (n + w.key_block - 1) // w.key_block
    centres = None
    if w.centre_sigma > 0:
        centres = rng.standard_normal((bh, nb, w.d), dtype=np.float32)
        centres *= np.float32(w.centre_sigma)
    k = rng.standard_normal(shape, dtype=np.float32)
    if centres is not None:
        # every token of block b gets c_b added (ragged last block included)
        tok_block = np.arange(n) // w.key_block
        k += centres[:, tok_block, :]
    v = rng.standard_normal(shape, dtype=np.float32)
    if w.popular > 0:
        # no extra draws: the other workloads' streams stay as they are
        q[:, :, 0] += np.float32(3.0)
        pop = np.linspace(0, nb - 1, w.popular).round().astype(np.int64)
        for b in pop:
            k[:, b * w.key_block:(b + 1) * w.key_block, 0] += np.float32(6.0)
    if w.dtype == "bf16":
        return Tensors(bf16_bits_rne(q), bf16_bits_rne(k), bf16_bits_rne(v),
                       "bf16", {"seed": seed})
    return Tensors(q, k, v, "fp32", {"seed": seed})


def sample_rows(bh: int, n: int, count_per_head: int, seed: int = 1,
                extra: tuple = ()) -> np.ndarray:
    """Deterministic sample of flat row ids (bh*n + i) for sampled parity.

    Always includes the first and last query of every head (edges) plus
    ``extra`` explicit query positions, then evenly spread seeded picks.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = []
    for h in range(bh):
        picks = set([0, n - 1] + [int(e) for e in extra if 0 <= e < n])
        if count_per_head > len(picks):
            picks.update(int(x) for x in
                         rng.choice(n, size=min(n, count_per_head), replace=False))
        rows.extend(h * n + i for i in sorted(picks))
    return np.asarray(rows, dtype=np.int64)
