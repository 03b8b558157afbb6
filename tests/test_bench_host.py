"""Host-side logic of bench.py and the workloads (CPU): the work a selection
admits, the scores the causal selection needs, and the skewed workload."""
import numpy as np
import pytest

import bench
import oracle
import workloads

torch = pytest.importorskip("torch")


def _brute_pairs(idx, n, kb, causal):
    total = 0
    for r, row in enumerate(idx.reshape(-1, idx.shape[-1])):
        i = r % n
        for b in row:
            if b < 0:
                continue
            for j in range(b * kb, min(n, (b + 1) * kb)):
                total += (not causal) or j <= i
    return total


@pytest.mark.parametrize("causal", [False, True])
def test_admitted_pairs_counts_keys_by_brute_force(causal):
    w = workloads.Workload("t", bh=2, n=150, d=64, dtype="bf16", kind="dynamic", key_block=32,
                           topk=3, causal=causal)
    rng = np.random.default_rng(0)
    idx = np.full((2, 150, 3), -1, np.int32)
    for h in range(2):
        for i in range(150):
            last = i // 32 if causal else w.nb - 1
            m = rng.integers(0, min(3, last + 1) + 1)
            idx[h, i, :m] = np.sort(rng.choice(last + 1, size=m, replace=False))
    want = _brute_pairs(idx, 150, 32, causal)
    assert bench.admitted_pairs(torch.from_numpy(idx), w) == want
    rows = np.arange(2 * 150, dtype=np.int64)
    assert bench.admitted_pairs(idx.reshape(-1, 3), w, rows) == want


def test_eligible_scores_closed_form():
    w = workloads.Workload("t", bh=3, n=200, d=64, dtype="bf16", kind="dynamic", key_block=64,
                           topk=4, causal=True)
    assert bench.eligible_scores(w) == 3 * sum(i // 64 + 1 for i in range(200))
    w2 = workloads.Workload("t", bh=3, n=200, d=64, dtype="bf16", kind="dynamic", key_block=64,
                            topk=4)
    assert bench.eligible_scores(w2) == 3 * 200 * 4


def test_oracle_step_flops_match_the_forward_formula_without_options():
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w)
    rows = workloads.sample_rows(w.bh, w.n, 8, seed=2)
    fl = bench.oracle_step(oracle, w, t, rows)
    per_row = bench.metrics.sparse_flops(w.n, w.bh, w.d, w.key_block, w.topk) / (w.n * w.bh)
    assert fl == pytest.approx(rows.size * per_row)


def test_skewed_workload_plants_popular_blocks_without_changing_other_draws():
    base = workloads.generate(workloads.WORKLOADS["dyn_n32768"], bh=1, n=4096)
    skew = workloads.generate(workloads.WORKLOADS["dyn_n32768_skew"], bh=1, n=4096)
    qb = workloads.bf16_bits_to_f32(base.q)
    qs = workloads.bf16_bits_to_f32(skew.q)
    np.testing.assert_array_equal(base.v, skew.v)               # same stream
    np.testing.assert_array_equal(base.q[..., 1:], skew.q[..., 1:])
    assert np.abs(qs[..., 0] - qb[..., 0] - 3.0).max() < 0.07   # bf16 rounding of the shift
    kb_ = workloads.bf16_bits_to_f32(base.k)[0, :, 0]
    ks = workloads.bf16_bits_to_f32(skew.k)[0, :, 0]
    shifted = np.unique(np.nonzero(np.abs(ks - kb_) > 1.0)[0] // 64)
    assert shifted.size == 8 and shifted[0] == 0 and shifted[-1] == 4096 // 64 - 1


def test_static_oracle_sample_counts_admitted_pairs():
    w = workloads.Workload("s", bh=2, n=1024, d=64, dtype="bf16", kind="sliding", key_block=64,
                           q_group=128, sliding=300)
    t = workloads.generate(w)
    tf, rows, secs, cores, desc = bench.static_oracle_sample(w, t, 0.2)
    assert tf > 0 and rows > 0 and secs > 0 and cores >= 1 and "fp64" in desc
