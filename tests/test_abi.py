"""The C-ABI library: it builds, loads, exports every declared symbol and
rejects bad arguments on the host (no GPU needed: validation runs before any
CUDA call)."""
import ctypes
import os
import re

import pytest

from content_dependent_block_gb300 import _build, bsa

HEADER = os.path.join(_build.INCLUDE, "bsa.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return bsa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(bsa.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.bsa_version() >= 100
    assert L.bsa_status_string(0) == b"ok"
    assert L.bsa_status_string(3) == b"block index out of range"
    assert L.bsa_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x10000)          # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x10008)


def _shape(bh=1, n=128, d=64, dtype=bsa.BF16):
    return bsa.Shape(bh, n, d, dtype)


@pytest.mark.parametrize("shape,code", [
    (_shape(d=96), 2), (_shape(n=0), 1), (_shape(bh=0), 1), (_shape(dtype=7), 1),
    (_shape(bh=70000), 2), (_shape(dtype=bsa.FP32), 2),
])
def test_forward_rejects_bad_shapes(L, shape, code):
    r = L.bsa_forward(shape, FAKE, FAKE, FAKE, 64, 4, 0.0, FAKE, None, FAKE, 1 << 30, None)
    assert r == code, L.bsa_last_error()


@pytest.mark.parametrize("kb,topk,code", [(48, 4, 2), (64, 0, 2), (64, 33, 2), (256, 4, 2)])
def test_forward_rejects_bad_block_or_k(L, kb, topk, code):
    r = L.bsa_forward(_shape(), FAKE, FAKE, FAKE, kb, topk, 0.0, FAKE, None, FAKE, 1 << 30, None)
    assert r == code


def test_forward_rejects_null_misaligned_and_small_workspace(L):
    s = _shape()
    assert L.bsa_forward(s, None, FAKE, FAKE, 64, 4, 0.0, FAKE, None, FAKE, 1 << 30, None) == 1
    assert L.bsa_forward(s, FAKE, MISALIGNED, FAKE, 64, 4, 0.0, FAKE, None, FAKE, 1 << 30, None) == 7
    need = L.bsa_forward_workspace_size(s, 64, 4)
    assert need > 0
    assert L.bsa_forward(s, FAKE, FAKE, FAKE, 64, 4, 0.0, FAKE, None, FAKE, need - 1, None) == 4
    assert L.bsa_forward(s, FAKE, FAKE, FAKE, 64, 4, 0.0, FAKE, None, None, need, None) == 4
    assert L.bsa_forward(s, FAKE, FAKE, FAKE, 64, 4, 0.0, FAKE, None, ctypes.c_void_p(0x10010),
                         need, None) == 7
    assert b"workspace" in L.bsa_last_error() or b"aligned" in L.bsa_last_error()


def test_fine_attention_rejects_bad_mask_and_list(L):
    s = _shape(dtype=bsa.FP32)
    ld = bsa.ListDesc(16, 16, 4, 0)
    assert L.bsa_fine_attention(s, FAKE, FAKE, FAKE, FAKE, ld, bsa.mask_struct(5), 0.0, FAKE,
                                None, 0, None) == 1
    assert L.bsa_fine_attention(s, FAKE, FAKE, FAKE, FAKE, ld, bsa.mask_struct(2, sliding=0), 0.0,
                                FAKE, None, 0, None) == 1
    assert L.bsa_fine_attention(s, FAKE, FAKE, FAKE, FAKE, bsa.ListDesc(0, 16, 4, 0),
                                bsa.mask_struct(), 0.0, FAKE, None, 0, None) == 1
    assert L.bsa_fine_attention(s, FAKE, FAKE, FAKE, FAKE, bsa.ListDesc(16, 24, 4, 0),
                                bsa.mask_struct(), 0.0, FAKE, None, 0, None) == 2


def test_pool_and_coarse_reject_fp32(L):
    s = _shape(dtype=bsa.FP32)
    assert L.bsa_pool_blocks(s, FAKE, 64, FAKE, None) == 2
    assert L.bsa_coarse_topk(s, FAKE, FAKE, 64, 4, FAKE, None, 0, None) == 2
    assert L.bsa_coarse_topk_ex(s, FAKE, FAKE, 64, 4, None, FAKE, None, 0, None) == 2


def test_graph_handles_are_checked(L):
    assert L.bsa_forward_graph_create(_shape(), FAKE, FAKE, FAKE, 64, 4, None, 0.0, FAKE, None,
                                      FAKE, 1 << 30, None) == 1
    assert L.bsa_graph_launch(None, None) == 1
    assert L.bsa_graph_destroy(None) == 0


def test_select_options_are_checked(L):
    s = _shape()
    bad = bsa.Select(0x10002, 1, 0)                   # head_topk not 4-byte aligned
    need = L.bsa_coarse_topk_workspace_size(s, 64, 4)
    assert L.bsa_coarse_topk_ex(s, FAKE, FAKE, 64, 4, ctypes.byref(bad), FAKE, FAKE, need,
                                None) == 7
    need = L.bsa_forward_workspace_size(s, 64, 4)
    assert L.bsa_forward_ex(s, FAKE, FAKE, FAKE, 64, 4, ctypes.byref(bad), 0.0, FAKE, None, FAKE,
                            need, None) == 7
    assert L.bsa_forward_ex(s, FAKE, FAKE, FAKE, 64, 33, None, 0.0, FAKE, None, FAKE, need,
                            None) == 2
    # the workspace does not depend on the options
    assert L.bsa_forward_workspace_size(s, 64, 4) == need


def test_backward_rejects_bad_arguments(L):
    s = _shape(n=256)
    ld = bsa.ListDesc(1, 64, 4, 1)
    need = L.bsa_fine_backward_workspace_size(s, ld)
    assert need > 0
    none = bsa.mask_struct()
    args = lambda **kw: [kw.get("shape", s), FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("lst", FAKE),
                         kw.get("ld", ld), kw.get("mask", none), 0.0, kw.get("dq", FAKE), FAKE,
                         FAKE, kw.get("ws", FAKE), kw.get("wsn", need), None]
    assert L.bsa_fine_backward(*args(shape=_shape(n=256, dtype=bsa.FP32))) == 2
    assert L.bsa_fine_backward(*args(shape=_shape(n=256, d=96))) == 2
    assert L.bsa_fine_backward(*args(ld=bsa.ListDesc(128, 64, 4, 0))) == 2      # static lists
    assert L.bsa_fine_backward(*args(mask=bsa.mask_struct(bsa.MASK_SLIDING, sliding=8))) == 2
    assert L.bsa_fine_backward(*args(lst=None)) == 1
    assert L.bsa_fine_backward(*args(dq=MISALIGNED)) == 7
    assert L.bsa_fine_backward(*args(wsn=need - 1)) == 4
    assert L.bsa_fine_backward(*args(shape=_shape(n=256, d=128), ld=bsa.ListDesc(1, 128, 4, 1))) == 2
    assert L.bsa_fine_backward_workspace_size(s, bsa.ListDesc(128, 64, 4, 0)) == 0


def test_saved_statistics_entry_points_reject_bad_arguments(L):
    s = _shape(n=256)
    ld = bsa.ListDesc(1, 64, 4, 1)
    none = bsa.mask_struct()
    need = L.bsa_fine_attention_workspace_size(s, ld, none)
    odd = ctypes.c_void_p(0x10002)                 # not 4-byte aligned
    fa = lambda lse, ld_=ld: L.bsa_fine_attention_lse(s, FAKE, FAKE, FAKE, FAKE, ld_, none, 0.0,
                                                      FAKE, lse, FAKE, need, None)
    assert fa(None) == 1
    assert fa(odd) == 7
    assert fa(FAKE, bsa.ListDesc(1, 32, 4, 1)) == 2            # not the block-major path
    assert fa(FAKE, bsa.ListDesc(128, 64, 4, 0)) == 2          # static tile lists
    nbw = L.bsa_fine_backward_workspace_size(s, ld)
    fb = lambda lse: L.bsa_fine_backward_lse(s, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ld, none, 0.0,
                                             lse, FAKE, FAKE, FAKE, FAKE, nbw, None)
    assert fb(None) == 1
    assert fb(odd) == 7
    nf = L.bsa_forward_workspace_size(s, 64, 4)
    fw = lambda kb, lse: L.bsa_forward_lse(s, FAKE, FAKE, FAKE, kb, 4, None, 0.0, FAKE, None, lse,
                                           FAKE, nf, None)
    assert fw(64, None) == 1
    assert fw(64, odd) == 7
    assert fw(32, FAKE) == 2                                  # not the block-major path


def test_static_path_workspace_is_optional_and_sized(L):
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=256)
    s = _shape(bh=2, n=1000, d=128)
    tiles, nb = -(-1000 // 128), -(-1000 // 64)
    need = L.bsa_fine_attention_workspace_size(s, bsa.ListDesc(128, 64, 9, 0), m)
    assert need >= 2 * nb * 4 + 2 * tiles * 4
    # fp32 and other tile heights take the query-major kernel: no workspace
    assert L.bsa_fine_attention_workspace_size(_shape(dtype=bsa.FP32), bsa.ListDesc(128, 64, 9, 0), m) == 0
    assert L.bsa_fine_attention_workspace_size(s, bsa.ListDesc(16, 64, 9, 0), m) == 0


def test_static_blocks_rejects_bad_arguments(L):
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=0)
    assert L.bsa_static_max_blocks(100, 16, 16, m) < 0
    lst = (ctypes.c_int32 * 64)()
    m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, 32, 512)
    # too few slots per row
    assert L.bsa_static_blocks(4096, 16, 16, m, ctypes.cast(lst, ctypes.c_void_p), 2, None, None) == 1
    assert L.bsa_static_blocks(4096, 16, 16, m, None, 16, None, None) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(bsa, "_lib", None)
    monkeypatch.setattr(bsa, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(bsa.BsaError):
        bsa.lib()


@pytest.mark.parametrize("kind,limit", [(2, 1_000_000), (-1, 1_000_000), (0, 999), (1, 2_000_000_001)])
def test_wait_selftest_rejects_bad_arguments(L, kind, limit):
    assert L.bsa_selftest_wait_timeout(kind, limit, None) == 1
    assert b"kind" in L.bsa_last_error() or b"limit" in L.bsa_last_error()


def test_forward_launch_counts(L):
    """A small problem runs as one fused launch; the 32k-token one as pool,
    scores + top-k, the three inversion kernels and the fine kernel."""
    assert L.bsa_forward_launches(_shape(bh=2, n=1024), 64, 4) == 1
    assert L.bsa_forward_launches(_shape(bh=8, n=8192), 64, 16) == 6
    assert L.bsa_forward_launches(_shape(bh=8, n=32768), 64, 16) == 6
