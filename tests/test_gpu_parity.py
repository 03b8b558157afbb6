"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Small workloads are compared on every row; the long-context ones (n = 32k
and 131k) on seeded row samples the oracle computes one by one, through the
same reusable ``Forward`` object the benchmark times.
"""
import numpy as np
import pytest

import oracle
import workloads
from content_dependent_block_gb300 import _build, bsa
from tests import parity

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    bsa.lib()
    assert bsa.device_status() == 0


_cache = {}


def tensors(name, **kw):
    key = (name, tuple(sorted(kw.items())))
    if key not in _cache:
        _cache.clear()
        w = W[name]
        t = workloads.generate(w, **kw)
        dev = tuple(parity.to_device(getattr(t, x), t.dtype) for x in "qkv")
        _cache[key] = (w, t, dev)
    return _cache[key]


def rows_for(w, bh, n, full_limit=70000, per_head=48):
    if bh * n <= full_limit:
        return oracle.all_rows(bh, n)
    return workloads.sample_rows(bh, n, per_head, extra=(w.key_block - 1, w.key_block, n // 2))


DYN = ["dyn_n1024", "dyn_n8192", "dyn_n32768", "dyn_n131072"]


@pytest.mark.parametrize("name", DYN)
def test_pool_matches_oracle(name):
    w, t, (q, k, v) = tensors(name)
    kbar = bsa.pool_blocks(k, w.key_block)
    ref = oracle.pool(t.k, w.key_block)
    got = kbar.cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("name", DYN)
def test_coarse_topk_matches_oracle_within_tie_band(name):
    w, t, (q, k, v) = tensors(name)
    kbar = bsa.pool_blocks(k, w.key_block)
    idx = bsa.coarse_topk(q, kbar, w.key_block, w.topk)
    rows = rows_for(w, w.bh, w.n)
    res_kbar = oracle.pool(t.k, w.key_block)
    s = oracle.scores(t.q, res_kbar, rows)
    oidx, kth = oracle.topk(s, w.topk)
    gidx = idx.cpu().numpy().reshape(-1, w.topk)[rows]
    differing = parity.check_selection(gidx, oidx, s, kth, w.nb)
    assert differing <= max(2, rows.size // 200), f"{differing} rows differ (all within band)"
    assert bsa.device_status() == 0


@pytest.mark.parametrize("name", DYN)
def test_fine_stage_on_oracle_indices(name):
    w, t, (q, k, v) = tensors(name)
    rows = rows_for(w, w.bh, w.n)
    s = oracle.scores(t.q, oracle.pool(t.k, w.key_block), rows)
    oidx, _ = oracle.topk(s, w.topk)
    # the list is the GPU's own selection except on the compared rows, which
    # carry the oracle's selection
    kbar = bsa.pool_blocks(k, w.key_block)
    lst = bsa.coarse_topk(q, kbar, w.key_block, w.topk).reshape(-1, w.topk)
    import torch
    lst[torch.from_numpy(rows).cuda()] = torch.from_numpy(oidx).cuda()
    out = bsa.fine_attention(q, k, v, lst.reshape(w.bh, w.n, w.topk), key_block=w.key_block)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, w.key_block, oidx, rows)
    got = parity.from_device(out).reshape(-1, w.d)[rows]
    parity.assert_close(got, o_ref, "bf16", f"{name} fine stage")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("name", DYN)
def test_forward_matches_oracle(name):
    w, t, (q, k, v) = tensors(name)
    f = bsa.Forward(w.bh, w.n, w.d, w.key_block, w.topk)
    out = f(q, k, v)
    rows = rows_for(w, w.bh, w.n)
    s = oracle.scores(t.q, oracle.pool(t.k, w.key_block), rows)
    oidx, kth = oracle.topk(s, w.topk)
    gidx = f.idx.cpu().numpy().reshape(-1, w.topk)[rows]
    parity.check_selection(gidx, oidx, s, kth, w.nb)
    # the oracle recomputes the fine stage on the GPU's (validated) selection
    o_ref, _, psum = oracle.fine(t.q, t.k, t.v, w.key_block, gidx, rows)
    np.testing.assert_allclose(psum, 1.0, atol=1e-12)
    got = parity.from_device(out).reshape(-1, w.d)[rows]
    parity.assert_close(got, o_ref, "bf16", f"{name} forward")
    assert bsa.device_status() == 0


def test_forward_skewed_lists():
    """Planted popular blocks that nearly every query selects: a popular
    (head, range, block) bin holds ~30x the mean number of pairs; the work
    items split it and the persistent CTAs share it."""
    w, t, (q, k, v) = tensors("dyn_n32768_skew", bh=2, n=8192)
    f = bsa.Forward(2, 8192, w.d, w.key_block, w.topk)
    out = f(q, k, v)
    rows = oracle.all_rows(2, 8192)
    s = oracle.scores(t.q, oracle.pool(t.k, w.key_block), rows)
    oidx, kth = oracle.topk(s, w.topk)
    gidx = f.idx.cpu().numpy().reshape(-1, w.topk)
    parity.check_selection(gidx, oidx, s, kth, 8192 // w.key_block)
    pop = np.linspace(0, 8192 // w.key_block - 1, w.popular).round().astype(int)
    assert np.isin(gidx, pop).sum(1).mean() > 6          # the lists really are skewed
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, w.key_block, gidx, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, w.d), o_ref, "bf16", "skewed lists")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("name", ["local_global_n4096", "local_global_n4100"])
def test_static_local_global_fp32(name):
    w, t, (q, k, v) = tensors(name)
    m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, w.window, w.stride)
    lst, counts, pairs = bsa.static_blocks(w.n, w.q_group, w.key_block, m)
    import torch
    dl = torch.from_numpy(lst).cuda()
    out = bsa.fine_attention(q, k, v, dl, key_block=w.key_block, q_group=w.q_group,
                             per_head=False, mask=m)
    rows = oracle.all_rows(w.bh, w.n)
    o_ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_LOCAL_GLOBAL, rows, w=w.window, s=w.stride)
    parity.assert_close(parity.from_device(out).reshape(-1, w.d), o_ref, "fp32", name)
    assert bsa.device_status() == 0


def test_static_sliding_n131072_sampled():
    w, t, (q, k, v) = tensors("dyn_n131072")       # same tensors, as the workload says
    sw = W["sliding_n131072"]
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=sw.sliding)
    lst, _, _ = bsa.static_blocks(sw.n, sw.q_group, sw.key_block, m)
    import torch
    out = bsa.fine_attention(q, k, v, torch.from_numpy(lst).cuda(), key_block=sw.key_block,
                             q_group=sw.q_group, per_head=False, mask=m)
    rows = workloads.sample_rows(sw.bh, sw.n, 24, extra=(1, 63, 64, 4095, 4096, 4097))
    o_ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_SLIDING, rows, W=sw.sliding)
    got = parity.from_device(out).reshape(-1, sw.d)[rows]
    parity.assert_close(got, o_ref, "bf16", "sliding n131072")
    assert bsa.device_status() == 0


# ------------------------------------------------------------ edge cases
def _small(bh, n, d, seed, dtype="bf16", sigma=0.0, kb=64):
    w = workloads.Workload("edge", bh=bh, n=n, d=d, dtype=dtype, kind="dynamic", key_block=kb,
                           topk=4, centre_sigma=sigma, seed=seed)
    t = workloads.generate(w)
    return t, tuple(parity.to_device(getattr(t, x), dtype) for x in "qkv")


EDGE_SHAPES = [
    (1, 1000, 64, 64, 4),      # ragged last block (40 tokens)
    (2, 300, 128, 32, 5),      # d=128, ragged, odd k
    (1, 40, 64, 64, 2),        # n < B: one partial block, k > nb
    (1, 1, 64, 16, 1),         # a single token
    (3, 256, 64, 64, 8),       # k*B >= n: dense attention
    (1, 4100, 64, 16, 32),     # many blocks, k = 32
    (2, 700, 128, 64, 6),      # d=128, ragged
]


@pytest.mark.parametrize("bh,n,d,kb,topk", EDGE_SHAPES)
@pytest.mark.parametrize("staged", [False, True], ids=["forward", "staged"])
def test_forward_edge_shapes(bh, n, d, kb, topk, staged):
    """bsa_forward (small problems: the single fused launch) and, staged,
    the same method as three calls -- pool, scores + top-k, fine attention
    over the selection (tensor-core scoring, block-major fine stage for
    64-key blocks)."""
    t, (q, k, v) = _small(bh, n, d, seed=n + d, sigma=0.5, kb=kb)
    if staged:
        idx = bsa.coarse_topk(q, bsa.pool_blocks(k, kb), kb, topk)
        out = bsa.fine_attention(q, k, v, idx, key_block=kb)
    else:
        out, idx = bsa.forward(q, k, v, kb, topk)
    rows = oracle.all_rows(bh, n)
    nb = -(-n // kb)
    s = oracle.scores(t.q, oracle.pool(t.k, kb), rows)
    oidx, kth = oracle.topk(s, topk)
    gidx = idx.cpu().numpy().reshape(-1, topk)
    parity.check_selection(gidx, oidx, s, kth, nb)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, kb, gidx, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, d), o_ref, "bf16", "edge forward")
    if topk * kb >= n:
        dense, _, _ = oracle.masked(t.q, t.k, t.v, 0, rows)
        parity.assert_close(parity.from_device(out).reshape(-1, d), dense, "bf16", "dense limit")
    assert bsa.device_status() == 0


def test_fine_empty_rows_give_zeros_and_bad_index_is_reported():
    import torch
    t, (q, k, v) = _small(1, 512, 64, seed=5)
    nb = 8
    lst = np.tile(np.array([[0, 3, 5, -1]], np.int32), (512, 1))
    lst[10] = -1                       # empty row -> zeros
    lst[11] = [1, 2, 99, -1]           # out-of-range id -> skipped + reported
    out = bsa.fine_attention(q, k, v, torch.from_numpy(lst).cuda().reshape(1, 512, 4), key_block=64)
    assert bsa.device_status() == 3   # BSA_ERR_BAD_INDEX
    got = parity.from_device(out).reshape(-1, 64)
    assert (parity.out_f64(got[10]) == 0).all()
    ref_list = lst.copy()
    ref_list[11] = [1, 2, -1, -1]
    rows = oracle.all_rows(1, 512)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, 64, ref_list, rows)
    keep = np.ones(512, bool)
    keep[10] = False
    parity.assert_close(got[keep], o_ref[keep], "bf16", "listed rows")
    assert nb == 8


@pytest.mark.parametrize("bh,n,d,k", [(16, 8192, 64, 16), (4, 8192, 128, 12)])
def test_fine_padded_lists_across_query_ranges(bh, n, d, k):
    """Caller lists with padding (a quarter of the slots -1, every 97th row
    empty) through the block-major fine stage, at sizes with several query
    ranges per head and more ranges than the partial-state ring holds (the
    ring is reused): the merge takes each query's valid slots from the
    inversion's slot masks."""
    import torch
    t, (q, kk, v) = _small(bh, n, d, seed=11 + d, sigma=0.5)
    nb = -(-n // 64)
    rng = np.random.Generator(np.random.PCG64(7 + d))
    lst = rng.random((bh * n, nb)).argsort(axis=1)[:, :k].astype(np.int32)
    lst[rng.random((bh * n, k)) < 0.25] = -1
    lst[::97] = -1
    out = bsa.fine_attention(q, kk, v, torch.from_numpy(lst).cuda().reshape(bh, n, k), key_block=64)
    assert bsa.device_status() == 0
    rows = workloads.sample_rows(bh, n, 40, extra=(63, 64, 97 * 3, n // 2))
    got = parity.from_device(out).reshape(-1, d)[rows]
    empty = (lst[rows] < 0).all(axis=1)
    assert empty.any() and (~empty).any()
    assert (parity.out_f64(got[empty]) == 0).all()
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, 64, lst[rows][~empty], rows[~empty])
    parity.assert_close(got[~empty], o_ref, "bf16", "padded lists")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_fine_explicit_scale_and_dtype(dtype):
    import torch
    t, (q, k, v) = _small(2, 640, 64, seed=9, dtype=dtype)
    rng = np.random.default_rng(0)
    lst = np.stack([np.sort(rng.choice(10, 3, replace=False)) for _ in range(2 * 640)]).astype(np.int32)
    out = bsa.fine_attention(q, k, v, torch.from_numpy(lst).cuda().reshape(2, 640, 3),
                             key_block=64, scale=0.3)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, 64, lst, oracle.all_rows(2, 640), scale=0.3)
    parity.assert_close(parity.from_device(out).reshape(-1, 64), o_ref, dtype, "scaled fine")


def test_dense_list_null_is_full_attention():
    t, (q, k, v) = _small(1, 200, 64, seed=3, dtype="fp32")
    out = bsa.fine_attention(q, k, v, None, key_block=32)
    rows = oracle.all_rows(1, 200)
    dense, _, _ = oracle.masked(t.q, t.k, t.v, 0, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, 64), dense, "fp32", "null list")


# ------------------------------------- static lists on the tensor cores
# bf16, 64-key blocks, one list row per 128-query tile: the query-tile-major
# tcgen05 kernel (exact two-pass softmax), against the plain masked definition.
# Windows and strides that cut 32-key chunks at odd places: stride 1 (every
# key), a window of 0 (the diagonal only), a stride that divides no block.
@pytest.mark.parametrize("n,d,per_head,w,s", [(4096, 64, False, 32, 512), (4100, 64, True, 32, 512),
                                              (1000, 128, False, 32, 512), (2000, 64, False, 70, 100),
                                              (900, 128, False, -1, 1), (1500, 64, True, 0, 37)])
def test_static_tc_local_global_bf16(n, d, per_head, w, s):
    import torch
    t, (q, k, v) = _small(2, n, d, seed=n + 7)
    m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, w, s)
    lst, _, _ = bsa.static_blocks(n, 128, 64, m)
    dl = torch.from_numpy(np.ascontiguousarray(np.stack([lst, lst]) if per_head else lst)).cuda()
    out = bsa.fine_attention(q, k, v, dl, key_block=64, q_group=128, per_head=per_head, mask=m)
    rows = oracle.all_rows(2, n)
    ref, _, psum = oracle.masked(t.q, t.k, t.v, oracle.MASK_LOCAL_GLOBAL, rows, w=w, s=s)
    np.testing.assert_allclose(psum, 1.0, atol=1e-12)
    parity.assert_close(parity.from_device(out).reshape(-1, d), ref, "bf16",
                        f"tensor-core local+global n={n} d={d} w={w} s={s}")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("n,d,win", [(1000, 128, 300), (4100, 64, 4096), (777, 64, 1)])
def test_static_tc_sliding_bf16(n, d, win):
    import torch
    t, (q, k, v) = _small(1, n, d, seed=win)
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=win)
    lst, _, _ = bsa.static_blocks(n, 128, 64, m)
    out = bsa.fine_attention(q, k, v, torch.from_numpy(lst).cuda(), key_block=64, q_group=128,
                             per_head=False, mask=m)
    rows = oracle.all_rows(1, n)
    ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_SLIDING, rows, W=win)
    parity.assert_close(parity.from_device(out).reshape(-1, d), ref, "bf16",
                        f"tensor-core sliding n={n} W={win}")
    assert bsa.device_status() == 0


def test_static_tc_bound_fallback_bf16():
    """Rows whose score bound |q| max|k| overshoots the true maximum by far
    (a large query component on a channel where every key is zero) are
    redone by the exact two-pass launch; the other tiles keep the one-pass
    result."""
    import torch
    n, d, W = 1000, 64, 300
    w = workloads.Workload("fb", bh=2, n=n, d=d, dtype="bf16", kind="dynamic", key_block=64,
                           topk=4, seed=17)
    t = workloads.generate(w)
    qf = workloads.bf16_bits_to_f32(t.q).copy()
    kf = workloads.bf16_bits_to_f32(t.k).copy()
    qf[0, 128:384, 0] = 400.0          # two tiles of head 0: bound ~ 400 x 8 / 8 x log2 e above
    kf[:, :, 0] = 0.0
    t.q[...] = workloads.bf16_bits_rne(qf)
    t.k[...] = workloads.bf16_bits_rne(kf)
    q, k, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=W)
    lst, _, _ = bsa.static_blocks(n, 128, 64, m)
    out = bsa.fine_attention(q, k, v, torch.from_numpy(lst).cuda(), key_block=64, q_group=128,
                             per_head=False, mask=m)
    rows = oracle.all_rows(2, n)
    ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_SLIDING, rows, W=W)
    parity.assert_close(parity.from_device(out).reshape(-1, d), ref, "bf16", "bound fallback")
    assert bsa.device_status() == 0


def test_static_tc_without_workspace_runs_two_passes_bf16():
    import ctypes
    import torch
    n, d = 1100, 128
    t, (q, k, v) = _small(1, n, d, seed=23)
    m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, 40, 300)
    lst, _, _ = bsa.static_blocks(n, 128, 64, m)
    dl = torch.from_numpy(lst).cuda()
    out = torch.empty_like(q)
    L = bsa.lib()
    ld = bsa.ListDesc(128, 64, lst.shape[1], 0)
    assert L.bsa_fine_attention_workspace_size(bsa._shape(q), ld, m) > 0
    bsa._check(L.bsa_fine_attention(bsa._shape(q), bsa._ptr(q), bsa._ptr(k), bsa._ptr(v),
                                    bsa._ptr(dl), ld, m, 0.0, bsa._ptr(out), None, 0,
                                    bsa._stream()))
    one = bsa.fine_attention(q, k, v, dl, key_block=64, q_group=128, per_head=False, mask=m)
    rows = oracle.all_rows(1, n)
    ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_LOCAL_GLOBAL, rows, w=40, s=300)
    parity.assert_close(parity.from_device(out).reshape(-1, d), ref, "bf16", "two passes")
    parity.assert_close(parity.from_device(one).reshape(-1, d), ref, "bf16", "one pass")
    assert bsa.device_status() == 0


def test_static_tc_null_list_is_dense_bf16():
    t, (q, k, v) = _small(2, 700, 64, seed=11)
    out = bsa.fine_attention(q, k, v, None, key_block=64)
    rows = oracle.all_rows(2, 700)
    dense, _, _ = oracle.masked(t.q, t.k, t.v, 0, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, 64), dense, "bf16", "dense bf16")
    assert bsa.device_status() == 0
