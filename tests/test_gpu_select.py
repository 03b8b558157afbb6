"""CUDA path vs the oracle for the selection options: per-head budgets (page
"sparse-attention-triton-bench", What's next), causal dynamic selection
(page "Block-Sparse & Linear Attention Kernels", section 1, causal pattern,
at both stages) and the always-include-local-block variant; plus the causal
token mask on the static tensor-core path and on per-query lists.

Selections are compared as sets: bit-exact, except that a block may differ
when its oracle score lies within the tie band of the boundary score (the
worst by-score block the oracle kept).  Outputs use the bf16 tolerances of
tests/parity.py; the oracle recomputes the fine stage on the GPU's
(validated) selection.
"""
import numpy as np
import pytest

import oracle
import workloads
from content_dependent_block_gb300 import _build, bsa
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    bsa.lib()
    assert bsa.device_status() == 0


def _inputs(bh, n, d, seed, kb=64):
    w = workloads.Workload("sel", bh=bh, n=n, d=d, dtype="bf16", kind="dynamic", key_block=kb,
                           topk=4, centre_sigma=0.5, seed=seed)
    t = workloads.generate(w)
    return t, tuple(parity.to_device(getattr(t, x), "bf16") for x in "qkv")


def _check(gidx, oidx, s, rows, n, kb, k, head_k, causal, local):
    """Every GPU row is a valid selection and equals the oracle's up to ties."""
    nb = s.shape[1]
    differing = 0
    for r in range(rows.size):
        h, i = divmod(int(rows[r]), n)
        own = i // kb
        kr = k if head_k is None else int(head_k[h])
        elig = own + 1 if causal else nb
        want = min(kr, elig)
        g = gidx[r]
        gs = g[:want]
        assert (g[want:] == -1).all(), f"row {r}: {g} (budget {kr}, eligible {elig})"
        assert (gs >= 0).all() and (gs < elig).all(), f"row {r}: ineligible id in {g}"
        assert (np.diff(gs) > 0).all(), f"row {r}: not strictly ascending: {g}"
        forced = local and kr >= 1
        if forced:
            assert own in gs, f"row {r}: own block {own} missing from {g}"
        o = oidx[r][:want]
        if np.array_equal(gs, o):
            continue
        differing += 1
        by_score = [b for b in o if not (forced and b == own)]
        kth = min(s[r, b] for b in by_score)
        band = parity.TIE_REL * max(abs(kth), parity.TIE_FLOOR)
        for b in np.setxor1d(gs, o):
            assert abs(s[r, b] - kth) <= band, (
                f"row {r}: block {b} (score {s[r, b]:.6g}) outside the tie band of {kth:.6g}")
    return differing


OPTS = [
    dict(causal=True),
    dict(local=True),
    dict(causal=True, local=True),
    dict(budgets=True),
    dict(causal=True, local=True, budgets=True),
]


def _budgets(bh, k):
    return np.array([(h * 5) % (k + 1) for h in range(bh)], dtype=np.int32)   # includes 0 and k


@pytest.mark.parametrize("opt", OPTS, ids=lambda o: "+".join(sorted(o)))
@pytest.mark.parametrize("bh,n,d,k", [(3, 4100, 64, 8), (2, 1000, 128, 5), (4, 2048, 64, 16)])
def test_forward_options_match_oracle(opt, bh, n, d, k):
    import torch
    kb = 64
    t, (q, kk, v) = _inputs(bh, n, d, seed=n + d + k)
    causal, local = opt.get("causal", False), opt.get("local", False)
    hk = _budgets(bh, k) if opt.get("budgets") else None
    out, idx = bsa.forward(q, kk, v, kb, k, causal=causal, local_block=local,
                           head_topk=None if hk is None else torch.from_numpy(hk).cuda())
    rows = oracle.all_rows(bh, n)
    s = oracle.scores(t.q, oracle.pool(t.k, kb), rows)
    oidx = oracle.select(s, rows, n, kb, k, head_k=hk, causal=causal, local=local)
    gidx = idx.cpu().numpy().reshape(-1, k)
    differing = _check(gidx, oidx, s, rows, n, kb, k, hk, causal, local)
    assert differing <= max(2, rows.size // 200)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, kb, gidx, rows, causal=causal)
    parity.assert_close(parity.from_device(out).reshape(-1, d), o_ref, "bf16", f"options {opt}")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("opt", OPTS[:3] + OPTS[4:], ids=lambda o: "+".join(sorted(o)))
def test_coarse_options_simt_path(opt):
    """Over 4096 blocks the selection runs on the CUDA cores, not the tensor
    cores; 16-token blocks also take the query-major fine kernel."""
    import torch
    bh, n, d, kb, k = 1, 70000, 64, 16, 4
    t, (q, kk, v) = _inputs(bh, n, d, seed=3, kb=kb)
    causal, local = opt.get("causal", False), opt.get("local", False)
    hk = np.array([3], dtype=np.int32) if opt.get("budgets") else None
    out, idx = bsa.forward(q, kk, v, kb, k, causal=causal, local_block=local,
                           head_topk=None if hk is None else torch.from_numpy(hk).cuda())
    rows = workloads.sample_rows(bh, n, 200, extra=(0, 15, 16, n - 1))
    s = oracle.scores(t.q, oracle.pool(t.k, kb), rows)
    oidx = oracle.select(s, rows, n, kb, k, head_k=hk, causal=causal, local=local)
    gidx = idx.cpu().numpy().reshape(-1, k)[rows]
    _check(gidx, oidx, s, rows, n, kb, k, hk, causal, local)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, kb, gidx, rows, causal=causal)
    got = parity.from_device(out).reshape(-1, d)[rows]
    parity.assert_close(got, o_ref, "bf16", f"simt options {opt}")
    assert bsa.device_status() == 0


def test_causal_full_budget_is_causal_attention():
    bh, n, d, kb = 2, 512, 64, 64
    t, (q, kk, v) = _inputs(bh, n, d, seed=21)
    out, idx = bsa.forward(q, kk, v, kb, n // kb, causal=True)
    rows = oracle.all_rows(bh, n)
    dense, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_CAUSAL, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, d), dense, "bf16", "causal dense limit")
    assert bsa.device_status() == 0


def test_out_of_range_budget_is_clamped_and_reported():
    import torch
    t, (q, kk, v) = _inputs(2, 600, 64, seed=4)
    hk = torch.tensor([9, -1], dtype=torch.int32, device="cuda")
    _, idx = bsa.forward(q, kk, v, 64, 4, head_topk=hk)
    assert bsa.device_status() == 1                    # BSA_ERR_INVALID_ARG
    g = idx.cpu().numpy()
    assert (g[0] >= 0).all() and (g[1] == -1).all()    # clamped to 4 and to 0


def test_causal_mask_on_per_query_lists_with_nothing_admitted():
    """A listed block entirely after the query admits no key: such a row
    (and only such a row) gets zeros."""
    import torch
    n, kb = 700, 64
    t, (q, kk, v) = _inputs(1, n, 64, seed=6)
    own = np.arange(n) // kb
    lst = np.full((n, 3), -1, np.int32)
    lst[:, 0] = 10                                     # the last block: keys 640..699
    mid = (own < 10) & (np.arange(n) >= 100)           # rows 100..639: own block, then 10
    lst[mid, 0] = own[mid]
    lst[mid, 1] = 10
    out = bsa.fine_attention(q, kk, v, torch.from_numpy(lst).cuda().reshape(1, n, 3), key_block=kb,
                             mask=bsa.mask_struct(bsa.MASK_CAUSAL))
    rows = oracle.all_rows(1, n)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, kb, lst, rows, causal=True)
    got = parity.from_device(out).reshape(-1, 64)
    assert (got[:100] == 0).all()
    parity.assert_close(got, o_ref, "bf16", "causal per-query lists")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("n,d", [(1000, 64), (4100, 128)])
def test_static_tc_causal(n, d):
    import torch
    t, (q, kk, v) = _inputs(2, n, d, seed=n)
    m = bsa.mask_struct(bsa.MASK_CAUSAL)
    lst, _, _ = bsa.static_blocks(n, 128, 64, m)
    out = bsa.fine_attention(q, kk, v, torch.from_numpy(lst).cuda(), key_block=64, q_group=128,
                             per_head=False, mask=m)
    rows = oracle.all_rows(2, n) if n <= 1000 else workloads.sample_rows(2, n, 300, extra=(0, 127, 128, n - 1))
    ref, _, _ = oracle.masked(t.q, t.k, t.v, oracle.MASK_CAUSAL, rows)
    got = parity.from_device(out).reshape(-1, d)[rows]
    parity.assert_close(got, ref, "bf16", f"static causal n={n} d={d}")
    assert bsa.device_status() == 0


@pytest.mark.parametrize("opt", [dict(), dict(causal=True, local=True, budgets=True)],
                         ids=["plain", "options"])
def test_graph_replay_matches_direct_calls(opt):
    """The captured forward reads its input buffers at every replay."""
    import torch
    bh, n, d, k = 2, 3000, 64, 8
    t, (q, kk, v) = _inputs(bh, n, d, seed=31)
    hk = torch.from_numpy(_budgets(bh, k)).cuda() if opt.get("budgets") else None
    kw = dict(head_topk=hk, causal=opt.get("causal", False), local_block=opt.get("local", False))
    direct = bsa.Forward(bh, n, d, 64, k, **kw)
    graph = bsa.Forward(bh, n, d, 64, k, graph=True, **kw)
    for step in range(3):
        if step:
            q.copy_(q.roll(1, dims=1))                  # new inputs, same buffers
            v.mul_(-1)
        o1 = direct(q, kk, v).clone()
        i1 = direct.idx.clone()
        o2 = graph(q, kk, v)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(i1, graph.idx), f"step {step}"
    graph.close()
    assert bsa.device_status() == 0
