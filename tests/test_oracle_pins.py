"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

None of these re-types the oracle's own loops: each check reaches the same
quantity by another route (a closed form, a library routine such as torch's
scaled-dot-product attention in float64, brute-force enumeration, an
invariant or a figure printed on the pages).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from content_dependent_block_gb300 import metrics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, dtype="fp32"):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(shape, dtype=np.float32)
    return workloads.bf16_bits_rne(x) if dtype == "bf16" else x


def _f64(a):
    return (workloads.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


def _sdpa(q, k, v, mask=None, scale=None):
    """torch's own attention in float64 (a library routine, not the oracle)."""
    tq, tk, tv = (torch.from_numpy(_f64(x)) for x in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=m, scale=scale).numpy()


# ---------------------------------------------------------------- pooling
def test_pool_block_of_one_is_identity():
    k = _rand((2, 37, 64), 1, "bf16")
    kbar = oracle.pool(k, 1)
    np.testing.assert_array_equal(kbar, _f64(k))


def test_pool_constant_blocks_return_the_constant():
    bh, n, d, B = 2, 100, 64, 16
    rng = np.random.default_rng(3)
    nb = -(-n // B)
    c = rng.standard_normal((bh, nb, d)).astype(np.float32)
    k = np.ascontiguousarray(c[:, np.arange(n) // B, :])
    np.testing.assert_array_equal(oracle.pool(k, B), c.astype(np.float64))


def test_pool_ramp_closed_form_including_ragged_tail():
    # K[j, c] = j + c: the mean of tokens j0..j1-1 is (j0 + j1 - 1)/2 + c
    n, d, B = 150, 64, 64          # blocks of 64, 64, 22 (ragged)
    j = np.arange(n, dtype=np.float32)[None, :, None]
    c = np.arange(d, dtype=np.float32)[None, None, :]
    k = np.ascontiguousarray(j + c)
    kbar = oracle.pool(k, B)
    for b in range(3):
        j0, j1 = b * B, min(n, (b + 1) * B)
        expect = (j0 + j1 - 1) / 2.0 + np.arange(d)
        np.testing.assert_array_equal(kbar[0, b], expect)


# -------------------------------------------------------- coarse scores
def test_scores_equal_block_mean_of_token_scores():
    # linearity: q . mean_j(k_j) == mean_j(q . k_j); right side via a dense
    # float64 matmul of the token scores, then a block average
    bh, n, d, B = 2, 200, 64, 32
    q, k = _rand((bh, n, d), 5, "bf16"), _rand((bh, n, d), 6, "bf16")
    rows = oracle.all_rows(bh, n)
    s = oracle.scores(q, oracle.pool(k, B), rows).reshape(bh, n, -1)
    tok = np.einsum("hid,hjd->hij", _f64(q), _f64(k))
    nb = -(-n // B)
    for b in range(nb):
        ref = tok[:, :, b * B:min(n, (b + 1) * B)].mean(axis=2)
        np.testing.assert_allclose(s[:, :, b], ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ top-k
def test_topk_matches_best_subset_by_enumeration():
    rng = np.random.default_rng(7)
    nb, k = 9, 3
    s = rng.standard_normal((40, nb))
    idx, kth = oracle.topk(s, k)
    for r in range(s.shape[0]):
        best = max(itertools.combinations(range(nb), k),
                   key=lambda c: sum(s[r, list(c)]))
        assert tuple(idx[r]) == tuple(sorted(best))
        assert kth[r] == min(s[r, list(best)])


def test_topk_ties_go_to_lower_block_index():
    s = np.array([[1.0, 2.0, 2.0, 2.0, 0.0, 2.0],
                  [5.0, 5.0, 5.0, 5.0, 5.0, 5.0],
                  [0.0, 3.0, 1.0, 3.0, 1.0, 1.0]])
    idx, _ = oracle.topk(s, 2)
    assert idx.tolist() == [[1, 2], [0, 1], [1, 3]]
    idx, _ = oracle.topk(s, 3)
    assert idx.tolist() == [[1, 2, 3], [0, 1, 2], [1, 2, 3]]


def test_topk_duplicate_key_blocks_resolve_to_lower_index():
    # blocks 2 and 5 hold identical keys: their means tie exactly, so a query
    # pointed at them must keep block 2 when only one more slot is left
    bh, n, d, B = 1, 8 * 16, 64, 16
    k = _rand((bh, n, d), 11, "bf16")
    k[:, 5 * B:6 * B] = k[:, 2 * B:3 * B]
    q = np.ascontiguousarray(k[:, 2 * B:2 * B + 1].repeat(n, axis=1))
    kbar = oracle.pool(k, B)
    s = oracle.scores(q, kbar, np.array([0]))
    assert s[0, 2] == s[0, 5]
    order = np.argsort(-s[0], kind="stable")
    kk = int(np.where(order == 2)[0][0]) + 1     # cut right after block 2
    idx, _ = oracle.topk(s, kk)
    assert 2 in idx[0] and 5 not in idx[0]


def test_topk_k_at_least_nb_selects_everything():
    s = np.random.default_rng(1).standard_normal((3, 5))
    idx, _ = oracle.topk(s, 7)
    assert idx.tolist() == [[0, 1, 2, 3, 4, -1, -1]] * 3


def test_planted_dominant_block_is_always_selected():
    bh, n, d, B, k = 1, 1024, 64, 64, 4
    t = workloads.generate(workloads.WORKLOADS["dyn_n1024"], bh=1)
    q = t.q.copy()
    kk = t.k.copy()
    planted = 9
    # every key of block 9 is 4x the first query: that block's mean dominates
    kk[0, planted * B:(planted + 1) * B] = workloads.bf16_bits_rne(
        4.0 * workloads.bf16_bits_to_f32(q[0, 0:1]))
    res = oracle.forward(q, kk, t.v, B, k, np.array([0]))
    assert planted in res["idx"][0]


# ------------------------------------------------------- fine attention
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_fine_with_all_blocks_is_dense_attention(dtype):
    # k*B >= N: every block is selected, so the result is exact dense attention
    bh, n, d, B = 2, 96, 64, 16
    q, k, v = (_rand((bh, n, d), s, dtype) for s in (21, 22, 23))
    rows = oracle.all_rows(bh, n)
    res = oracle.forward(q, k, v, B, 64, rows)       # k clamps to nb = 6
    assert (res["idx"][:, :6] == np.arange(6)).all()
    ref = _sdpa(q, k, v).reshape(bh * n, d)
    np.testing.assert_allclose(res["o"], ref, rtol=0, atol=1e-12)


def test_fine_matches_masked_library_attention_on_random_lists():
    bh, n, d, B, kk = 2, 160, 64, 16, 3
    q, k, v = (_rand((bh, n, d), s, "bf16") for s in (31, 32, 33))
    nb = n // B
    rng = np.random.default_rng(4)
    rows = oracle.all_rows(bh, n)
    idx = np.stack([np.sort(rng.choice(nb, kk, replace=False)) for _ in rows]).astype(np.int32)
    o, lse, psum = oracle.fine(q, k, v, B, idx, rows)
    mask = np.zeros((bh, n, n), dtype=bool)
    for r, row in enumerate(rows):
        h, i = divmod(int(row), n)
        for b in idx[r]:
            mask[h, i, b * B:(b + 1) * B] = True
    ref = _sdpa(q, k, v, mask=mask).reshape(bh * n, d)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(psum, 1.0, rtol=0, atol=1e-12)


def test_fine_single_token_returns_its_value():
    q, k, v = (_rand((1, 10, 64), s, "bf16") for s in (1, 2, 3))
    rows = np.arange(10)
    idx = np.array([[7]] * 10, dtype=np.int32)          # B=1: one token, j=7
    o, lse, _ = oracle.fine(q, k, v, 1, idx, rows)
    np.testing.assert_array_equal(o, np.repeat(_f64(v)[0, 7:8], 10, axis=0))
    s = _f64(q)[0] @ _f64(k)[0, 7] / 8.0
    np.testing.assert_allclose(lse, s, rtol=0, atol=1e-12)


def test_fine_two_tokens_is_a_logistic_mix():
    q, k, v = (_rand((1, 4, 64), s) for s in (8, 9, 10))
    o, lse, _ = oracle.fine(q, k, v, 2, np.array([[1]], np.int32), np.array([0]),
                            scale=0.3)
    s2, s3 = 0.3 * (_f64(q)[0, 0] @ _f64(k)[0, 2]), 0.3 * (_f64(q)[0, 0] @ _f64(k)[0, 3])
    w2 = 1.0 / (1.0 + math.exp(s3 - s2))
    ref = w2 * _f64(v)[0, 2] + (1.0 - w2) * _f64(v)[0, 3]
    np.testing.assert_allclose(o[0], ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], np.logaddexp(s2, s3), rtol=0, atol=1e-13)


def test_fine_output_is_a_convex_combination_and_rows_sum_to_one():
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w)
    rows = workloads.sample_rows(w.bh, w.n, 64)
    res = oracle.forward(t.q, t.k, t.v, w.key_block, w.topk, rows)
    np.testing.assert_allclose(res["psum"], 1.0, rtol=0, atol=1e-12)
    v = t.as_f32("v").astype(np.float64)
    for r, row in enumerate(rows):
        h, i = divmod(int(row), w.n)
        sel = np.concatenate([np.arange(b * 64, b * 64 + 64) for b in res["idx"][r]])
        assert (res["o"][r] <= v[h, sel].max(axis=0) + 1e-12).all()
        assert (res["o"][r] >= v[h, sel].min(axis=0) - 1e-12).all()


def test_permuting_key_blocks_permutes_indices_and_keeps_output():
    bh, n, d, B, kk = 1, 256, 64, 32, 3
    q, k, v = (_rand((bh, n, d), s, "bf16") for s in (41, 42, 43))
    nb = n // B
    perm = np.random.default_rng(5).permutation(nb)       # new block p <- old perm[p]
    tok = np.concatenate([np.arange(b * B, (b + 1) * B) for b in perm])
    k2, v2 = np.ascontiguousarray(k[:, tok]), np.ascontiguousarray(v[:, tok])
    rows = oracle.all_rows(bh, n)
    a = oracle.forward(q, k, v, B, kk, rows)
    b = oracle.forward(q, k2, v2, B, kk, rows)
    inv = np.argsort(perm)                                 # old block -> new block
    mapped = np.sort(inv[a["idx"]], axis=1)
    # identical sets unless the k-th score ties, which random bf16 data avoids
    assert (mapped == b["idx"]).all()
    np.testing.assert_allclose(a["o"], b["o"], rtol=0, atol=1e-12)


def test_scale_only_changes_fine_stage_not_selection():
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w)
    rows = workloads.sample_rows(w.bh, w.n, 16)
    a = oracle.forward(t.q, t.k, t.v, 64, 4, rows, scale=0.125)
    b = oracle.forward(t.q, t.k, t.v, 64, 4, rows, scale=1.0)
    assert (a["idx"] == b["idx"]).all()
    assert np.abs(a["o"] - b["o"]).max() > 1e-3


# ---------------------------------------------------------- static masks
def test_local_global_mask_pair_count_closed_form():
    for n, w, s in [(40, 2, 8), (64, 0, 16), (97, 5, 7), (33, -1, 4), (50, 3, 0)]:
        _, pairs = oracle.active_tiles(n, 1, 1, oracle.MASK_LOCAL_GLOBAL, w=w, s=s)
        assert pairs == metrics.local_global_pairs(n, w, s)


def test_local_global_mask_small_enumeration():
    # |i-j| <= 2 or j % 8 == 0 on N=12, written out by hand for two rows
    row0 = [j for j in range(12) if oracle.mask(oracle.MASK_LOCAL_GLOBAL, 0, j, w=2, s=8)]
    row11 = [j for j in range(12) if oracle.mask(oracle.MASK_LOCAL_GLOBAL, 11, j, w=2, s=8)]
    assert row0 == [0, 1, 2, 8]
    assert row11 == [0, 8, 9, 10, 11]


def test_sliding_mask_pair_count_and_rows():
    for n, W in [(10, 3), (64, 64), (100, 1), (70, 200)]:
        _, pairs = oracle.active_tiles(n, 1, 1, oracle.MASK_SLIDING, W=W)
        assert pairs == metrics.sliding_pairs(n, W)
    assert [j for j in range(10) if oracle.mask(oracle.MASK_SLIDING, 5, j, W=3)] == [3, 4, 5]
    assert [j for j in range(10) if oracle.mask(oracle.MASK_SLIDING, 0, j, W=3)] == [0]


def _tile_active_closed_form(I, J, tq, tk, n, w, s):
    i0, i1 = I * tq, min(n, (I + 1) * tq) - 1
    j0, j1 = J * tk, min(n, (J + 1) * tk) - 1
    # band: the interval distance between [i0,i1] and [j0,j1] is at most w
    gap = max(0, j0 - i1, i0 - j1)
    band = w >= 0 and gap <= w
    stride = s > 0 and (j1 // s) * s >= j0
    return band or stride


@pytest.mark.parametrize("n", [4096, 4100])
def test_local_global_active_tiles_and_counts(n):
    w, s, t = 32, 512, 16
    act, pairs = oracle.active_tiles(n, t, t, oracle.MASK_LOCAL_GLOBAL, w=w, s=s)
    for I in range(act.shape[0]):
        for J in range(act.shape[1]):
            assert act[I, J] == _tile_active_closed_form(I, J, t, t, n, w, s)
    assert pairs == metrics.local_global_pairs(n, w, s)
    per_row = act.sum(axis=1)
    if n == 4096:
        assert act.sum() == 3284 and pairs == 297464
        assert per_row.min() == 10 and per_row.max() == 13
    else:
        assert act.sum() == 3551 and pairs == 301820
        assert per_row.min() == 11 and per_row.max() == 14


def test_sliding_window_covering_everything_is_causal_dense():
    bh, n, d = 2, 80, 64
    q, k, v = (_rand((bh, n, d), s, "bf16") for s in (51, 52, 53))
    rows = oracle.all_rows(bh, n)
    o, _, psum = oracle.masked(q, k, v, oracle.MASK_SLIDING, rows, W=n)
    tq, tk, tv = (torch.from_numpy(_f64(x)) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(o, ref.numpy().reshape(-1, d), rtol=0, atol=1e-12)
    np.testing.assert_allclose(psum, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("w,s", [(1000, 0), (-1, 1), (3, 1)])
def test_local_global_degenerate_cases_are_dense(w, s):
    bh, n, d = 1, 64, 64
    q, k, v = (_rand((bh, n, d), x) for x in (61, 62, 63))
    o, _, _ = oracle.masked(q, k, v, oracle.MASK_LOCAL_GLOBAL, oracle.all_rows(bh, n), w=w, s=s)
    np.testing.assert_allclose(o, _sdpa(q, k, v).reshape(-1, d), rtol=0, atol=1e-12)


def test_masked_matches_library_attention_with_explicit_mask():
    bh, n, d, w, s = 1, 120, 64, 4, 32
    q, k, v = (_rand((bh, n, d), x) for x in (71, 72, 73))
    o, _, _ = oracle.masked(q, k, v, oracle.MASK_LOCAL_GLOBAL, oracle.all_rows(bh, n), w=w, s=s)
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    mask = (np.abs(i - j) <= w) | (j % s == 0)
    np.testing.assert_allclose(o, _sdpa(q, k, v, mask=mask[None]).reshape(-1, d), rtol=0, atol=1e-12)


def test_sliding_equals_fine_over_block_list_plus_token_mask_at_block_ends():
    # for the last query of a block with W a multiple of B, the window is
    # exactly W/B whole blocks: the static pattern reduces to a block list
    bh, n, d, B, W = 1, 512, 64, 64, 192
    q, k, v = (_rand((bh, n, d), x, "bf16") for x in (81, 82, 83))
    rows = np.array([B * b + B - 1 for b in range(3, 8)])
    o1, _, _ = oracle.masked(q, k, v, oracle.MASK_SLIDING, rows, W=W)
    idx = np.array([[b - 2, b - 1, b] for b in range(3, 8)], dtype=np.int32)
    o2, _, _ = oracle.fine(q, k, v, B, idx, rows)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


# ------------------------------------------------------ printed figures
def _golden():
    out = {}
    with open(os.path.join(GOLDEN, "pages_figures.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, val, *_ = [x.strip() for x in line.split("|")]
            out[key] = val
    return out


def test_flop_count_reproduces_the_printed_figures():
    g = _golden()
    sp = metrics.sparse_flops(32768, 8, 64, 64, 16)
    de = metrics.dense_flops(32768, 8, 64)
    assert sp == 87_241_523_200 and de == 2_241_972_928_512
    assert metrics.format_si(sp, 3) == g["sparse_flops_n32768"]
    assert metrics.format_si(de, 3) == g["dense_flops_n32768"]
    assert f"{100 * sp / de:.1f}%" == g["sparse_percent_of_dense_n32768"]
    assert f"{16 * 64:,}" == g["tokens_per_query_n32768_b64_k16"]


def test_sliding_window_figures():
    g = _golden()
    n, W = 131072, 4096
    assert f"{n // W}x" == g["sliding_reduction_s131072_w4096"]
    assert f"{n * n // 2**30} billion" == g["dense_pairs_per_head_s131072"]
    # the exact causal-window pair count (ramp included) sits within the
    # printed 32x of S^2, never below it
    assert 32 <= n * n / metrics.sliding_pairs(n, W) < 33
