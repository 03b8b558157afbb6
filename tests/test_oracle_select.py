"""Pins of the oracle's selection options and causal fine step (CPU only).

The options: per-head budgets (page "sparse-attention-triton-bench", What's
next: top_k chosen per head on the per-head stage-1 scores), causal dynamic
selection (page "Block-Sparse & Linear Attention Kernels", section 1, the
causal pattern, applied to the block choice and to the keys), and the
always-include-local-block variant.  Each is pinned against something other
than the oracle itself:
  - the selected set is checked against a characterisation that fixes it
    uniquely (size, eligibility, the forced block, and every selected
    by-score block beating every unselected eligible block under the
    (score desc, id asc) order), on scores with many ties;
  - special cases reduce to torch's scaled_dot_product_attention in
    float64: a causal budget covering every block is causal attention, a
    budget of one forced local block is block-diagonal attention, a full
    budget without options is dense attention.
"""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")


def _qkv(bh, n, d, seed):
    rng = np.random.default_rng(seed)
    return [workloads.bf16_bits_rne(rng.standard_normal((bh, n, d)).astype(np.float32))
            for _ in range(3)]


def _f64(x):
    return torch.from_numpy(workloads.bf16_bits_to_f32(x).astype(np.float64))


def _sdpa(q, k, v, mask=None, causal=False):
    """Library attention in float64; mask[i, j] True = attend."""
    Q, K, V = _f64(q), _f64(k), _f64(v)
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=m, is_causal=causal).numpy()


def _check_selection(sel, srow, i, kr, B, causal, local):
    """The selection of one row is the unique set with these properties."""
    nb = srow.size
    own = i // B
    elig = set(range(own + 1)) if causal else set(range(nb))
    got = [int(b) for b in sel if b >= 0]
    assert list(sel[:len(got)]) == sorted(got) and all(b == -1 for b in sel[len(got):])
    T = set(got)
    assert len(T) == len(got)                          # no repeats
    assert T <= elig
    assert len(T) == min(kr, len(elig))
    forced = {own} if (local and kr >= 1) else set()
    assert forced <= T
    for b in T - forced:
        for c in elig - T:
            assert srow[b] > srow[c] or (srow[b] == srow[c] and b < c), (b, c)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("local", [False, True])
def test_select_characterisation_with_ties(causal, local):
    rng = np.random.default_rng(11 + 2 * causal + local)
    bh, n, B, k = 3, 70, 8, 5                          # nb = 9, ragged last block
    nb = -(-n // B)
    rows = np.arange(bh * n, dtype=np.int64)
    s = rng.integers(-2, 3, size=(rows.size, nb)).astype(np.float64)   # many ties
    head_k = np.array([0, 3, k], dtype=np.int32)
    idx = oracle.select(s, rows, n, B, k, head_k=head_k, causal=causal, local=local)
    for r in range(rows.size):
        h, i = divmod(int(rows[r]), n)
        _check_selection(idx[r], s[r], i, int(head_k[h]), B, causal, local)


def test_select_without_options_is_topk():
    rng = np.random.default_rng(5)
    s = rng.integers(-3, 4, size=(40, 12)).astype(np.float64)
    rows = np.arange(40, dtype=np.int64)
    for k in (1, 4, 12, 15):
        a = oracle.select(s, rows, 40, 4, k)
        b, _ = oracle.topk(s, k)
        np.testing.assert_array_equal(a, b)


def test_causal_full_budget_is_causal_attention():
    q, k, v = _qkv(2, 200, 64, seed=1)
    nb = -(-200 // 16)
    rows = oracle.all_rows(2, 200)
    res = oracle.forward(q, k, v, 16, nb, rows, causal=True)
    ref = _sdpa(q, k, v, causal=True).reshape(-1, 64)
    np.testing.assert_allclose(res["o"], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["psum"], 1.0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_local_single_block_is_block_diagonal(causal):
    n, B = 150, 32
    q, k, v = _qkv(1, n, 64, seed=2 + causal)
    rows = oracle.all_rows(1, n)
    res = oracle.forward(q, k, v, B, 1, rows, causal=causal, local=True)
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    mask = (i // B) == (j // B)
    if causal:
        mask &= j <= i
    assert (res["idx"][:, 0] == np.arange(n) // B).all()
    np.testing.assert_allclose(res["o"], _sdpa(q, k, v, mask=mask).reshape(-1, 64),
                               rtol=0, atol=1e-12)


def test_per_head_budgets_full_and_zero():
    n, B = 128, 16
    nb = n // B
    q, k, v = _qkv(2, n, 64, seed=7)
    rows = oracle.all_rows(2, n)
    res = oracle.forward(q, k, v, B, nb, rows, head_k=np.array([nb, 0], dtype=np.int32))
    dense = _sdpa(q[:1], k[:1], v[:1]).reshape(-1, 64)
    np.testing.assert_allclose(res["o"][:n], dense, rtol=0, atol=1e-12)
    assert (res["idx"][n:] == -1).all()
    assert (res["o"][n:] == 0).all() and np.isneginf(res["lse"][n:]).all()


def test_mask_kind_causal_is_causal_attention():
    q, k, v = _qkv(1, 90, 64, seed=9)
    rows = oracle.all_rows(1, 90)
    o, _, psum = oracle.masked(q, k, v, oracle.MASK_CAUSAL, rows)
    np.testing.assert_allclose(o, _sdpa(q, k, v, causal=True).reshape(-1, 64), rtol=0, atol=1e-12)
    assert oracle.mask(oracle.MASK_CAUSAL, 5, 5) and not oracle.mask(oracle.MASK_CAUSAL, 5, 6)


# ------------------------------------------------------------ backward pass
def _random_lists(bh, n, B, k, seed, causal):
    rng = np.random.default_rng(seed)
    nb = -(-n // B)
    idx = np.full((bh * n, k), -1, np.int32)
    for r in range(bh * n):
        i = r % n
        last = i // B if causal else nb - 1
        m = rng.integers(0, min(k, last + 1) + 1)           # some rows get no block
        idx[r, :m] = np.sort(rng.choice(last + 1, size=m, replace=False))
    return idx


@pytest.mark.parametrize("causal", [False, True])
def test_backward_equals_autograd_of_masked_attention(causal):
    """The fine stage with its lists fixed is masked softmax attention; torch
    autograd of that (float64) gives the gradients."""
    bh, n, d, B, k = 2, 150, 64, 16, 4                     # ragged last block (6 tokens)
    q, kk, v = _qkv(bh, n, d, seed=40 + causal)
    do = _qkv(bh, n, d, seed=50 + causal)[0]
    idx = _random_lists(bh, n, B, k, seed=3, causal=causal)
    dq, dk, dv = oracle.fine_backward(q, kk, v, do, B, idx, causal=causal)
    mask = np.zeros((bh, n, n), dtype=bool)
    for r in range(bh * n):
        h, i = divmod(r, n)
        for b in idx[r]:
            if b >= 0:
                j = np.arange(b * B, min(n, (b + 1) * B))
                mask[h, i, j[(j <= i) if causal else slice(None)]] = True
    Q, K, V = (_f64(x).requires_grad_() for x in (q, kk, v))
    s = (Q @ K.transpose(-1, -2)) / np.sqrt(d)
    s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)           # rows with no key: zero
    (p @ V).backward(_f64(do))
    for got, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-11)
    assert (dq.reshape(-1, d)[(idx < 0).all(1)] == 0).all()  # empty rows: no gradient


def test_budgets_outside_the_list_width_are_clamped():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((2 * 50, 7))
    rows = np.arange(100, dtype=np.int64)
    got = oracle.select(s, rows, 50, 8, 4, head_k=np.array([-2, 9], dtype=np.int32))
    assert (got[:50] == -1).all()                                   # clamped to 0
    np.testing.assert_array_equal(got[50:], oracle.topk(s[50:], 4)[0])   # clamped to k
