"""Thin ctypes binding over libbsa.so (include/bsa.h).

Argument marshalling only: every step of the method runs in the library's
CUDA kernels.  Device tensors come from PyTorch (it provides device memory,
streams and events); work is enqueued on PyTorch's current stream.  If
libbsa.so has not been built, every call raises ``BsaError`` -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from . import _build

BF16, FP32 = 0, 1
MASK_NONE, MASK_LOCAL_GLOBAL, MASK_SLIDING, MASK_CAUSAL = 0, 1, 2, 3

STATUS = {0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_UNSUPPORTED",
          3: "BSA_ERR_BAD_INDEX", 4: "BSA_ERR_WORKSPACE", 5: "BSA_ERR_CUDA",
          6: "BSA_ERR_TIMEOUT", 7: "BSA_ERR_ALIGNMENT"}

# Every symbol include/bsa.h declares.
EXPORTS = (
    "bsa_pool_blocks", "bsa_coarse_topk_workspace_size", "bsa_coarse_topk",
    "bsa_coarse_topk_ex", "bsa_fine_attention_workspace_size", "bsa_fine_attention",
    "bsa_fine_attention_lse", "bsa_fine_backward_workspace_size", "bsa_fine_backward",
    "bsa_fine_backward_lse",
    "bsa_forward_workspace_size", "bsa_forward", "bsa_forward_ex", "bsa_forward_lse",
    "bsa_forward_noalloc",
    "bsa_forward_launches", "bsa_forward_graph_create", "bsa_graph_launch", "bsa_graph_destroy",
    "bsa_static_max_blocks",
    "bsa_static_blocks", "bsa_get_device_status", "bsa_selftest_wait_timeout", "bsa_status_string",
    "bsa_last_error", "bsa_version",
)


class BsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("bh", ctypes.c_int64), ("n", ctypes.c_int64),
                ("d", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class Mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("stride", ctypes.c_int32), ("sliding", ctypes.c_int32)]


class ListDesc(ctypes.Structure):
    _fields_ = [("q_group", ctypes.c_int32), ("key_block", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("per_head", ctypes.c_int32)]


class Select(ctypes.Structure):
    """bsa_select: per-head budgets (device int32 [bh] or NULL), causal
    selection, always-include-local-block."""
    _fields_ = [("head_topk", ctypes.c_void_p), ("causal", ctypes.c_int32),
                ("local_block", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libbsa.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise BsaError(5, f"{path} is missing: build it with content_dependent_block_gb300._build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_size_t, ctypes.c_float)
    sig = {
        "bsa_pool_blocks": ([Shape, vp, i32, vp, vp], i32),
        "bsa_coarse_topk_workspace_size": ([Shape, i32, i32], sz),
        "bsa_coarse_topk": ([Shape, vp, vp, i32, i32, vp, vp, sz, vp], i32),
        "bsa_coarse_topk_ex": ([Shape, vp, vp, i32, i32, ctypes.POINTER(Select), vp, vp, sz, vp],
                               i32),
        "bsa_fine_attention_workspace_size": ([Shape, ListDesc, Mask], sz),
        "bsa_fine_attention": ([Shape, vp, vp, vp, vp, ListDesc, Mask, f32, vp, vp, sz, vp], i32),
        "bsa_fine_attention_lse": ([Shape, vp, vp, vp, vp, ListDesc, Mask, f32, vp, vp, vp, sz, vp],
                                   i32),
        "bsa_fine_backward_workspace_size": ([Shape, ListDesc], sz),
        "bsa_fine_backward": ([Shape, vp, vp, vp, vp, vp, vp, ListDesc, Mask, f32, vp, vp, vp, vp, sz,
                               vp], i32),
        "bsa_fine_backward_lse": ([Shape, vp, vp, vp, vp, vp, vp, ListDesc, Mask, f32, vp, vp, vp, vp,
                                   vp, sz, vp], i32),
        "bsa_forward_workspace_size": ([Shape, i32, i32], sz),
        "bsa_forward": ([Shape, vp, vp, vp, i32, i32, f32, vp, vp, vp, sz, vp], i32),
        "bsa_forward_ex": ([Shape, vp, vp, vp, i32, i32, ctypes.POINTER(Select), f32, vp, vp, vp,
                            sz, vp], i32),
        "bsa_forward_lse": ([Shape, vp, vp, vp, i32, i32, ctypes.POINTER(Select), f32, vp, vp, vp,
                             vp, sz, vp], i32),
        "bsa_forward_noalloc": ([Shape, vp, vp, vp, i32, i32, f32, vp, vp, vp], i32),
        "bsa_forward_graph_create": ([Shape, vp, vp, vp, i32, i32, ctypes.POINTER(Select), f32, vp,
                                      vp, vp, sz, ctypes.POINTER(vp)], i32),
        "bsa_graph_launch": ([vp, vp], i32),
        "bsa_graph_destroy": ([vp], i32),
        "bsa_forward_launches": ([Shape, i32, i32], i32),
        "bsa_static_max_blocks": ([i64, i32, i32, Mask], i32),
        "bsa_static_blocks": ([i64, i32, i32, Mask, vp, i32, vp, vp], i32),
        "bsa_get_device_status": ([vp, vp], i32),
        "bsa_selftest_wait_timeout": ([i32, ctypes.c_uint64, vp], i32),
        "bsa_status_string": ([i32], ctypes.c_char_p),
        "bsa_last_error": ([], ctypes.c_char_p),
        "bsa_version": ([], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(code: int):
    if code != 0:
        raise BsaError(code, lib().bsa_last_error().decode())


def _torch():
    import torch
    return torch


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _shape(t) -> Shape:
    torch = _torch()
    if t.dim() != 3 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("tensors must be contiguous CUDA [bh, n, d]")
    if t.dtype == torch.bfloat16:
        dt = BF16
    elif t.dtype == torch.float32:
        dt = FP32
    else:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return Shape(t.shape[0], t.shape[1], t.shape[2], dt)


def _workspace(nbytes: int, device):
    if nbytes == 0:
        return None
    return _torch().empty(nbytes, dtype=_torch().uint8, device=device)


def mask_struct(kind: int = MASK_NONE, window: int = -1, stride: int = 0, sliding: int = 0) -> Mask:
    return Mask(kind, window, stride, sliding)


def pool_blocks(k, key_block: int):
    """Block means Kbar [bh, ceil(n/B), d] fp32 of bf16 keys."""
    s = _shape(k)
    nb = -(-s.n // key_block)
    kbar = _torch().empty((s.bh, nb, s.d), dtype=_torch().float32, device=k.device)
    _check(lib().bsa_pool_blocks(s, _ptr(k), key_block, _ptr(kbar), _stream()))
    return kbar


def _select(head_topk, causal: bool, local_block: bool):
    """A Select for the options, or None when there are none."""
    if head_topk is None and not causal and not local_block:
        return None
    if head_topk is not None and (head_topk.dtype != _torch().int32 or not head_topk.is_cuda
                                  or not head_topk.is_contiguous()):
        raise TypeError("head_topk must be a contiguous int32 CUDA tensor [bh]")
    return Select(None if head_topk is None else head_topk.data_ptr(), int(bool(causal)),
                  int(bool(local_block)))


def coarse_topk(q, kbar, key_block: int, topk: int, *, head_topk=None, causal: bool = False,
                local_block: bool = False):
    """Top-k block ids [bh, n, topk] int32 (ascending, -1 padded); with the
    selection options of bsa_coarse_topk_ex when any is given."""
    s = _shape(q)
    idx = _torch().empty((s.bh, s.n, topk), dtype=_torch().int32, device=q.device)
    ws_n = lib().bsa_coarse_topk_workspace_size(s, key_block, topk)
    ws = _workspace(ws_n, q.device)
    sel = _select(head_topk, causal, local_block)
    _check(lib().bsa_coarse_topk_ex(s, _ptr(q), _ptr(kbar), key_block, topk,
                                    None if sel is None else ctypes.byref(sel), _ptr(idx),
                                    _ptr(ws), ws_n, _stream()))
    return idx


def fine_attention(q, k, v, block_list=None, *, key_block: int, q_group: int = 1,
                   per_head: bool = True, mask: Optional[Mask] = None, scale: float = 0.0,
                   out=None):
    """Softmax attention of each query over its listed blocks' tokens.

    ``block_list``: int32 device tensor [bh or 1, ceil(n/q_group), max_blocks]
    (or 2-D [rows, max_blocks] when shared by all heads), None = all blocks.
    """
    s = _shape(q)
    mask = mask or mask_struct()
    if block_list is not None:
        if block_list.dtype != _torch().int32 or not block_list.is_contiguous():
            raise TypeError("block_list must be a contiguous int32 tensor")
        ld = ListDesc(q_group, key_block, block_list.shape[-1], 1 if per_head else 0)
    else:
        ld = ListDesc(1, key_block, 0, 0)
    out = _torch().empty_like(q) if out is None else out
    ws_n = lib().bsa_fine_attention_workspace_size(s, ld, mask)
    ws = _workspace(ws_n, q.device)
    _check(lib().bsa_fine_attention(s, _ptr(q), _ptr(k), _ptr(v), _ptr(block_list), ld, mask,
                                    float(scale), _ptr(out), _ptr(ws), ws_n, _stream()))
    return out


def fine_attention_lse(q, k, v, block_list, *, key_block: int, causal: bool = False,
                       scale: float = 0.0, out=None):
    """(O, lse): fine attention over the per-query lists ``block_list``
    [bh, n, k] and each query's log2-sum-exp (fp32 [bh, n]) for
    fine_backward(..., lse=lse); see bsa_fine_attention_lse in bsa.h."""
    torch = _torch()
    s = _shape(q)
    if block_list.dtype != torch.int32 or not block_list.is_contiguous():
        raise TypeError("block_list must be a contiguous int32 tensor")
    ld = ListDesc(1, key_block, block_list.shape[-1], 1)
    m = mask_struct(MASK_CAUSAL if causal else MASK_NONE)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    ws_n = lib().bsa_fine_attention_workspace_size(s, ld, m)
    ws = _workspace(ws_n, q.device)
    _check(lib().bsa_fine_attention_lse(s, _ptr(q), _ptr(k), _ptr(v), _ptr(block_list), ld, m,
                                        float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws_n,
                                        _stream()))
    return out, lse


def fine_backward(q, k, v, out, dout, block_list, *, key_block: int, causal: bool = False,
                  scale: float = 0.0, lse=None):
    """Gradients (dq, dk, dv), fp32 [bh, n, d], of the fine stage over the
    per-query lists ``block_list`` [bh, n, k] (held fixed); with ``lse``
    (from fine_attention_lse on the same inputs) the softmax statistics are
    not recomputed.  See bsa_fine_backward / bsa_fine_backward_lse in bsa.h."""
    torch = _torch()
    s = _shape(q)
    if block_list.dtype != torch.int32 or not block_list.is_contiguous():
        raise TypeError("block_list must be a contiguous int32 tensor")
    ld = ListDesc(1, key_block, block_list.shape[-1], 1)
    m = mask_struct(MASK_CAUSAL if causal else MASK_NONE)
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=q.device) for _ in range(3))
    ws_n = lib().bsa_fine_backward_workspace_size(s, ld)
    ws = _workspace(ws_n, q.device)
    if lse is None:
        _check(lib().bsa_fine_backward(s, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                       _ptr(block_list), ld, m, float(scale), _ptr(dq), _ptr(dk),
                                       _ptr(dv), _ptr(ws), ws_n, _stream()))
    else:
        if lse.dtype != torch.float32 or not lse.is_contiguous():
            raise TypeError("lse must be a contiguous float32 tensor [bh, n]")
        _check(lib().bsa_fine_backward_lse(s, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                           _ptr(block_list), ld, m, float(scale), _ptr(lse),
                                           _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws_n,
                                           _stream()))
    return dq, dk, dv


class Forward:
    """Reusable forward: owns the output, selection and workspace buffers for
    one shape so repeated calls allocate nothing.  With ``graph=True`` the
    forward is captured once as a CUDA graph (bsa_forward_graph_create) for
    the q, k, v buffers of the first call and replayed with one launch; a
    call with other buffers captures again."""

    def __init__(self, bh: int, n: int, d: int, key_block: int, topk: int, device="cuda",
                 scale: float = 0.0, *, head_topk=None, causal: bool = False,
                 local_block: bool = False, graph: bool = False):
        torch = _torch()
        self.shape = Shape(bh, n, d, BF16)
        self.key_block, self.topk, self.scale = key_block, topk, scale
        self.head_topk = head_topk            # kept alive: the library reads it on every call
        self.sel = _select(head_topk, causal, local_block)
        self.use_graph = graph
        self._graph = None                    # (handle, (q, k, v) pointers, keep_idx)
        self.ws_bytes = lib().bsa_forward_workspace_size(self.shape, key_block, topk)
        self.ws = _workspace(self.ws_bytes, device)
        self.out = torch.empty((bh, n, d), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((bh, n, topk), dtype=torch.int32, device=device)

    @property
    def launches(self) -> int:
        """Kernel launches one call enqueues."""
        return int(lib().bsa_forward_launches(self.shape, self.key_block, self.topk))

    def __call__(self, q, k, v, keep_idx: bool = True):
        s = _shape(q)
        if (s.bh, s.n, s.d) != (self.shape.bh, self.shape.n, self.shape.d):
            raise ValueError("shape differs from the one this Forward was built for")
        sel = None if self.sel is None else ctypes.byref(self.sel)
        if not self.use_graph:
            _check(lib().bsa_forward_ex(self.shape, _ptr(q), _ptr(k), _ptr(v), self.key_block,
                                        self.topk, sel, float(self.scale), _ptr(self.out),
                                        _ptr(self.idx if keep_idx else None), _ptr(self.ws),
                                        self.ws_bytes, _stream()))
            return self.out
        key = ((q.data_ptr(), k.data_ptr(), v.data_ptr()), keep_idx)
        if self._graph is None or self._graph[1] != key:
            self.close()
            h = ctypes.c_void_p()
            _check(lib().bsa_forward_graph_create(
                self.shape, _ptr(q), _ptr(k), _ptr(v), self.key_block, self.topk, sel,
                float(self.scale), _ptr(self.out), _ptr(self.idx if keep_idx else None),
                _ptr(self.ws), self.ws_bytes, ctypes.byref(h)))
            self._graph = (h, key)
        _check(lib().bsa_graph_launch(self._graph[0], _stream()))
        return self.out

    def close(self):
        """Release the captured graph, if any."""
        if self._graph is not None:
            lib().bsa_graph_destroy(self._graph[0])
            self._graph = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward(q, k, v, key_block: int, topk: int, scale: float = 0.0, *, head_topk=None,
            causal: bool = False, local_block: bool = False) -> Tuple[object, object]:
    """Whole dynamic forward (with the selection options of bsa_forward_ex);
    returns (out, idx)."""
    s = _shape(q)
    f = Forward(s.bh, s.n, s.d, key_block, topk, device=q.device, scale=scale,
                head_topk=head_topk, causal=causal, local_block=local_block)
    out = f(q, k, v, keep_idx=True)
    return out, f.idx


def forward_lse(q, k, v, key_block: int, topk: int, scale: float = 0.0, *, head_topk=None,
                causal: bool = False, local_block: bool = False):
    """Whole dynamic forward that also keeps each query's log2-sum-exp for
    fine_backward(..., lse=lse); returns (out, idx, lse).  See
    bsa_forward_lse in bsa.h."""
    torch = _torch()
    s = _shape(q)
    out = torch.empty_like(q)
    idx = torch.empty((s.bh, s.n, topk), dtype=torch.int32, device=q.device)
    lse = torch.empty((s.bh, s.n), dtype=torch.float32, device=q.device)
    sel = _select(head_topk, causal, local_block)
    ws_n = lib().bsa_forward_workspace_size(s, key_block, topk)
    ws = _workspace(ws_n, q.device)
    _check(lib().bsa_forward_lse(s, _ptr(q), _ptr(k), _ptr(v), key_block, topk,
                                 None if sel is None else ctypes.byref(sel), float(scale),
                                 _ptr(out), _ptr(idx), _ptr(lse), _ptr(ws), ws_n, _stream()))
    return out, idx, lse


def forward_noalloc(q, k, v, key_block: int, topk: int, scale: float = 0.0, out=None, idx=None):
    """Whole dynamic forward using the library's static scratch (no workspace
    allocation); returns (out, idx).  See bsa_forward_noalloc in bsa.h."""
    torch = _torch()
    s = _shape(q)
    out = torch.empty_like(q) if out is None else out
    idx = torch.empty((s.bh, s.n, topk), dtype=torch.int32, device=q.device) if idx is None else idx
    _check(lib().bsa_forward_noalloc(s, _ptr(q), _ptr(k), _ptr(v), key_block, topk, float(scale),
                                     _ptr(out), _ptr(idx), _stream()))
    return out, idx


def static_blocks(n: int, q_group: int, key_block: int, mask: Mask):
    """Host-built static list: (list [rows, max_blocks] int32, counts, active_pairs)."""
    L = lib()
    mb = L.bsa_static_max_blocks(n, q_group, key_block, mask)
    if mb < 0:
        raise BsaError(-mb, L.bsa_last_error().decode() or "bad static-list arguments")
    rows = -(-n // q_group)
    lst = np.empty((rows, max(mb, 1)), dtype=np.int32)
    counts = np.empty(rows, dtype=np.int32)
    pairs = ctypes.c_int64(0)
    _check(L.bsa_static_blocks(n, q_group, key_block, mask,
                               lst.ctypes.data_as(ctypes.c_void_p), lst.shape[1],
                               counts.ctypes.data_as(ctypes.c_void_p), ctypes.byref(pairs)))
    return lst, counts, int(pairs.value)


def device_status() -> int:
    """Read and clear the device status word (synchronises the stream)."""
    v = ctypes.c_int32(0)
    _check(lib().bsa_get_device_status(ctypes.byref(v), _stream()))
    return int(v.value)


def selftest_wait_timeout(kind: int, limit_ns: int) -> None:
    """Enqueue the bounded-wait self-test (bsa_selftest_wait_timeout): a wait
    nothing completes gives up after about limit_ns and records
    BSA_ERR_TIMEOUT; read it with device_status()."""
    _check(lib().bsa_selftest_wait_timeout(int(kind), int(limit_ns), _stream()))
