"""Host-built static block lists against the oracle's brute-force tile scan."""
import numpy as np
import pytest

import oracle
from content_dependent_block_gb300 import _build, bsa, metrics


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()


def _oracle_lists(n, tq, tk, kind, w=-1, s=0, W=0, row_begin=0, row_end=None):
    act, pairs = oracle.active_tiles(n, tq, tk, kind, w=w, s=s, W=W,
                                     row_begin=row_begin, row_end=row_end)
    return act, pairs


def _as_sets(lst, counts):
    return [tuple(lst[r, :counts[r]]) for r in range(lst.shape[0])]


CASES = [
    # n, q_group, key_block, kind, w, s, W
    (4096, 16, 16, oracle.MASK_LOCAL_GLOBAL, 32, 512, 0),
    (4100, 16, 16, oracle.MASK_LOCAL_GLOBAL, 32, 512, 0),
    (1000, 64, 32, oracle.MASK_LOCAL_GLOBAL, 5, 97, 0),
    (777, 16, 64, oracle.MASK_LOCAL_GLOBAL, -1, 100, 0),
    (777, 32, 16, oracle.MASK_LOCAL_GLOBAL, 40, 0, 0),
    (1500, 128, 64, oracle.MASK_SLIDING, -1, 0, 256),
    (1500, 64, 64, oracle.MASK_SLIDING, -1, 0, 100),
    (300, 16, 16, oracle.MASK_SLIDING, -1, 0, 1),
    (1000, 128, 64, oracle.MASK_CAUSAL, -1, 0, 0),
    (333, 16, 32, oracle.MASK_CAUSAL, -1, 0, 0),
]


@pytest.mark.parametrize("n,tq,tk,kind,w,s,W", CASES)
def test_static_lists_match_brute_force(n, tq, tk, kind, w, s, W):
    m = bsa.mask_struct(kind, w, s, W)
    lst, counts, pairs = bsa.static_blocks(n, tq, tk, m)
    act, opairs = _oracle_lists(n, tq, tk, kind, w, s, W)
    for r in range(act.shape[0]):
        expect = tuple(np.nonzero(act[r])[0])
        got = tuple(lst[r, :counts[r]])
        assert got == expect, f"row {r}"
        assert (lst[r, counts[r]:] == -1).all()
    assert pairs == opairs
    assert lst.shape[1] == counts.max()


def test_local_global_n4096_counts():
    m = bsa.mask_struct(bsa.MASK_LOCAL_GLOBAL, 32, 512)
    for n, tiles, pairs, lo, hi in [(4096, 3284, 297464, 10, 13), (4100, 3551, 301820, 11, 14)]:
        lst, counts, p = bsa.static_blocks(n, 16, 16, m)
        assert counts.sum() == tiles and p == pairs
        assert counts.min() == lo and counts.max() == hi
        assert p == metrics.local_global_pairs(n, 32, 512)


def test_sliding_n131072_sampled_rows():
    n, tq, tk, W = 131072, 128, 64, 4096
    m = bsa.mask_struct(bsa.MASK_SLIDING, sliding=W)
    lst, counts, pairs = bsa.static_blocks(n, tq, tk, m)
    assert pairs == metrics.sliding_pairs(n, W)
    assert counts.max() == 66 and counts.min() == 2
    for r in [0, 1, 31, 32, 33, 500, 1023]:
        act, _ = _oracle_lists(n, tq, tk, oracle.MASK_SLIDING, W=W, row_begin=r, row_end=r + 1)
        assert tuple(lst[r, :counts[r]]) == tuple(np.nonzero(act[0])[0])


def test_none_mask_lists_every_block():
    lst, counts, pairs = bsa.static_blocks(200, 64, 32, bsa.mask_struct())
    assert (counts == 7).all() and pairs == 200 * 200
    assert (lst == np.arange(7)).all()
