"""fp64 CPU oracle for content-dependent block-sparse attention (forward).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  The
product path never imports this package, and this package never imports the
product (``content_dependent_block_gb300``): the two share no code.

The arithmetic lives in ``bsa_oracle.c`` (plain C, double precision, OpenMP
over rows); this file only marshals numpy arrays.  ``build()`` compiles the C
file with gcc into ``oracle/_build/liboracle.so`` (also done lazily on first
use).  Every function cites the page passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

BF16, FP32 = 0, 1
MASK_LOCAL_GLOBAL, MASK_SLIDING, MASK_CAUSAL = 1, 2, 3

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2 -fopenmp, no fast-math) if needed."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or
             os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        dbl = ctypes.c_double
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_pool.argtypes = [vp, i32, i64, i64, i64, i64, vp]
        lib.orc_scores.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, i64, vp]
        lib.orc_topk.argtypes = [vp, i64, i64, i64, vp, vp]
        lib.orc_select.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, i32, i32, vp]
        lib.orc_fine.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, vp, i64,
                                 vp, i64, i32, dbl, vp, vp, vp]
        lib.orc_fine_backward.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, i64, i32,
                                          dbl, vp, vp, vp]
        lib.orc_mask.argtypes = [i32, i64, i64, i64, i64, i64]
        lib.orc_mask.restype = ctypes.c_int
        lib.orc_masked.argtypes = [vp, vp, vp, i32, i64, i64, i64, i32, i64,
                                   i64, i64, vp, i64, dbl, vp, vp, vp]
        lib.orc_active_tiles.argtypes = [i64, i64, i64, i32, i64, i64, i64,
                                         i64, i64, vp]
        lib.orc_active_tiles.restype = ctypes.c_int64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return FP32
    raise TypeError(f"oracle inputs are bf16 bit patterns (uint16) or float32, got {x.dtype}")


def _check3(*arrs):
    shape = arrs[0].shape
    for a in arrs:
        if a.ndim != 3 or a.shape != shape or not a.flags.c_contiguous:
            raise ValueError("Q/K/V must be C-contiguous [bh, n, d] arrays of one shape")
        if a.dtype != arrs[0].dtype:
            raise ValueError("Q/K/V must share one dtype")
    return shape


def num_threads() -> int:
    return int(_load().orc_num_threads())


def pool(k: np.ndarray, key_block: int) -> np.ndarray:
    """Block means Kbar [bh, nb, d] (page "sparse-attention-triton-bench",
    Two-stage block indexer, Stage 1)."""
    bh, n, d = _check3(k)
    nb = -(-n // key_block)
    out = np.empty((bh, nb, d), dtype=np.float64)
    _load().orc_pool(_ptr(k), _dtype_code(k), bh, n, d, key_block, _ptr(out))
    return out


def all_rows(bh: int, n: int) -> np.ndarray:
    return np.arange(bh * n, dtype=np.int64)


def scores(q: np.ndarray, kbar: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Unscaled coarse scores S[r, b] = q_i . Kbar_b for rows r (flat bh*n+i)."""
    bh, n, d = _check3(q)
    nb = kbar.shape[1]
    kbar = np.ascontiguousarray(kbar, dtype=np.float64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, nb), dtype=np.float64)
    _load().orc_scores(_ptr(q), _dtype_code(q), bh, n, d, _ptr(kbar), nb,
                       _ptr(rows), rows.size, _ptr(out))
    return out


def topk(s: np.ndarray, k: int):
    """Top-k blocks per row: ascending block ids [rows, k] (-1 padded) and the
    k-th best score per row (page "sparse-attention-triton-bench", Stage 2)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    nrows, nb = s.shape
    idx = np.empty((nrows, k), dtype=np.int32)
    kth = np.empty(nrows, dtype=np.float64)
    _load().orc_topk(_ptr(s), nrows, nb, k, _ptr(idx), _ptr(kth))
    return idx, kth


def select(s: np.ndarray, rows: np.ndarray, n: int, key_block: int, k: int, *,
           head_k: Optional[np.ndarray] = None, causal: bool = False,
           local: bool = False) -> np.ndarray:
    """Selection with options: per-(batch*head) budgets ``head_k`` (int, in
    [0, k]; page "sparse-attention-triton-bench", What's next), causal
    eligibility b <= i // key_block (page "Block-Sparse & Linear Attention
    Kernels", section 1, causal pattern) and the always-include-local-block
    variant.  ``s`` holds the scores of ``rows`` (flat bh*n + i).  Returns
    ascending ids [len(rows), k], -1 padded."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    nrows, nb = s.shape
    if nrows != rows.size:
        raise ValueError("one score row per requested query row")
    hk = None if head_k is None else np.ascontiguousarray(head_k, dtype=np.int32)
    idx = np.empty((nrows, k), dtype=np.int32)
    _load().orc_select(_ptr(s), _ptr(rows), nrows, nb, n, key_block, k,
                       None if hk is None else _ptr(hk), int(causal), int(local), _ptr(idx))
    return idx


def fine(q, k, v, key_block: int, idx: np.ndarray, rows: np.ndarray,
         scale: Optional[float] = None, causal: bool = False):
    """Softmax attention of each row over the tokens of its listed blocks
    (only keys j <= i with ``causal``).

    ``idx`` is [len(rows), kmax] int32 (entries < 0 ignored).  Returns
    (O [rows, d] float64, lse [rows], psum [rows]).
    """
    bh, n, d = _check3(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if idx.shape[0] != rows.size:
        raise ValueError("idx needs one row per requested query row")
    kk = idx.shape[1]
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    psum = np.empty(rows.size, dtype=np.float64)
    _load().orc_fine(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), bh, n, d,
                     key_block, _ptr(idx), kk, _ptr(rows), rows.size, int(causal),
                     ctypes.c_double(scale), _ptr(o), _ptr(lse), _ptr(psum))
    return o, lse, psum


def fine_backward(q, k, v, do, key_block: int, idx: np.ndarray,
                  scale: Optional[float] = None, causal: bool = False):
    """Gradients (dQ, dK, dV) [bh, n, d] float64 of the fine stage with the
    selection fixed (page "sparse-attention-triton-bench", What's next:
    backward pass).  ``idx`` holds the lists of every row, [bh*n, kmax]."""
    bh, n, d = _check3(q, k, v, do)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(bh * n, -1)
    out = [np.empty((bh, n, d), dtype=np.float64) for _ in range(3)]
    _load().orc_fine_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _dtype_code(q), bh, n, d,
                              key_block, _ptr(idx), idx.shape[1], int(causal),
                              ctypes.c_double(scale), *(_ptr(a) for a in out))
    return tuple(out)


def mask(kind: int, i: int, j: int, w: int = -1, s: int = 0, W: int = 0) -> bool:
    return bool(_load().orc_mask(kind, w, s, W, i, j))


def masked(q, k, v, kind: int, rows: np.ndarray, *, w: int = -1, s: int = 0,
           W: int = 0, scale: Optional[float] = None):
    """Dense attention over {j : mask(i, j)} (static patterns, plain
    definition).  Returns (O [rows, d], lse, psum)."""
    bh, n, d = _check3(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    psum = np.empty(rows.size, dtype=np.float64)
    _load().orc_masked(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), bh, n, d,
                       kind, w, s, W, _ptr(rows), rows.size,
                       ctypes.c_double(scale), _ptr(o), _ptr(lse), _ptr(psum))
    return o, lse, psum


def active_tiles(n: int, tq: int, tk: int, kind: int, *, w: int = -1,
                 s: int = 0, W: int = 0, row_begin: int = 0,
                 row_end: Optional[int] = None):
    """Brute-force tile activity [rows, ceil(n/tk)] (uint8) and the number of
    active (i, j) pairs inside the evaluated tile rows."""
    nqt = -(-n // tq)
    nkt = -(-n // tk)
    row_end = nqt if row_end is None else row_end
    act = np.zeros((row_end - row_begin, nkt), dtype=np.uint8)
    pairs = _load().orc_active_tiles(n, tq, tk, kind, w, s, W, row_begin,
                                     row_end, _ptr(act))
    return act, int(pairs)


def forward(q, k, v, key_block: int, topk_k: int, rows: np.ndarray,
            scale: Optional[float] = None, *, head_k: Optional[np.ndarray] = None,
            causal: bool = False, local: bool = False):
    """The whole dynamic path for the requested rows, step by step:
    pool -> scores -> top-k (or the selection with options) -> fine.
    Returns a dict of every intermediate (``kth`` only without options)."""
    kbar = pool(k, key_block)
    s = scores(q, kbar, rows)
    if head_k is None and not causal and not local:
        idx, kth = topk(s, topk_k)
    else:
        idx = select(s, rows, q.shape[1], key_block, topk_k, head_k=head_k,
                     causal=causal, local=local)
        kth = None
    o, lse, psum = fine(q, k, v, key_block, idx, rows, scale, causal=causal)
    return {"kbar": kbar, "scores": s, "idx": idx, "kth": kth, "o": o,
            "lse": lse, "psum": psum}
