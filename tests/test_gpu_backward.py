"""Backward pass of the fine stage vs the fp64 oracle (lists fixed): the
tensor-core kernel for 64-key blocks, the CUDA-core kernels for other sizes.

The GPU takes D_i = dO_i . O_i from the bf16 forward output, the oracle the
exact sum_j p_ij dP_ij; the bf16 rounding of O (2^-9 relative) bounds the
difference, so the gradients (fp32) are held to the bf16 output tolerances
of tests/parity.py, scaled by the largest reference gradient:
  relative L2 error <= 5e-3,  max-abs error <= 2e-2 * max |reference|.
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


def _inputs(bh, n, d, seed, kb):
    w = workloads.Workload("bwd", bh=bh, n=n, d=d, dtype="bf16", kind="dynamic", key_block=kb,
                           topk=4, centre_sigma=0.5, seed=seed)
    t = workloads.generate(w)
    do = workloads.bf16_bits_rne(np.random.default_rng(seed + 1).standard_normal(
        (bh, n, d)).astype(np.float32))
    return t, do


def _grad_close(got, ref, what):
    err = got.astype(np.float64) - ref
    scale = max(np.abs(ref).max(), 1e-6)
    rel_l2 = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    max_abs = np.abs(err).max()
    assert rel_l2 <= 5e-3 and max_abs <= 2e-2 * scale, (
        f"{what}: rel-L2 {rel_l2:.3e}, max-abs {max_abs:.3e} (max |ref| {scale:.3e})")


def _random_lists(bh, n, kb, k, seed, causal):
    rng = np.random.default_rng(seed)
    nb = -(-n // kb)
    idx = np.full((bh * n, k), -1, np.int32)
    for r in range(bh * n):
        last = (r % n) // kb if causal else nb - 1
        m = rng.integers(0, min(k, last + 1) + 1)            # some rows list nothing
        idx[r, :m] = np.sort(rng.choice(last + 1, size=m, replace=False))
    return idx


@pytest.mark.parametrize("bh,n,d,kb,k,causal,lists", [
    (2, 1000, 64, 64, 8, False, "selected"),     # ragged last block (40 tokens)
    (2, 1000, 64, 64, 8, True, "selected"),
    (1, 700, 128, 64, 4, True, "selected"),
    (2, 513, 64, 32, 6, False, "random"),        # empty rows, one-token last block
    (1, 300, 128, 32, 16, True, "random"),
    # 64-key blocks run on the tensor cores: random lists with empty rows, a
    # one-token last block, the causal mask, d 128, more than one 128-row tile
    # per block
    (2, 513, 64, 64, 6, False, "random"),
    (1, 300, 128, 64, 5, True, "random"),
    (2, 4100, 64, 64, 16, True, "selected"),
])
def test_backward_matches_oracle(bh, n, d, kb, k, causal, lists):
    import torch
    t, do = _inputs(bh, n, d, seed=n + d + k, kb=kb)
    q, kk, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    dout = parity.to_device(do, "bf16")
    if lists == "selected":
        out, idx = bsa.forward(q, kk, v, kb, k, causal=causal)
        lst = idx.contiguous()
        idx_np = idx.cpu().numpy().reshape(-1, k)
    else:
        idx_np = _random_lists(bh, n, kb, k, seed=7, causal=causal)
        lst = torch.from_numpy(idx_np).cuda().reshape(bh, n, k)
        out = bsa.fine_attention(q, kk, v, lst, key_block=kb,
                                 mask=bsa.mask_struct(bsa.MASK_CAUSAL if causal else bsa.MASK_NONE))
    dq, dk, dv = bsa.fine_backward(q, kk, v, out, dout, lst, key_block=kb, causal=causal)
    rq, rk, rv = oracle.fine_backward(t.q, t.k, t.v, do, kb, idx_np, causal=causal)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _grad_close(got.cpu().numpy(), ref, f"{name} bh={bh} n={n} d={d} kb={kb} k={k} causal={causal}")
    if lists == "random":
        empty = (idx_np < 0).all(1)
        assert (dq.cpu().numpy().reshape(-1, d)[empty] == 0).all()
    assert bsa.device_status() == 0


def test_backward_bad_index_is_reported():
    import torch
    t, do = _inputs(1, 256, 64, seed=5, kb=64)
    q, kk, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    lst = torch.tensor([[0, 2, -1]] * 256, dtype=torch.int32, device="cuda").reshape(1, 256, 3)
    out = bsa.fine_attention(q, kk, v, lst, key_block=64)
    lst[0, 5, 2] = 99
    bsa.fine_backward(q, kk, v, out, parity.to_device(do, "bf16"), lst, key_block=64)
    assert bsa.device_status() == 3                           # BSA_ERR_BAD_INDEX


@pytest.mark.parametrize("bh,n,d,k,causal", [
    (2, 513, 64, 6, False),       # random lists with empty rows, a one-token last block
    (1, 700, 128, 5, True),
    (2, 4100, 64, 16, True),
])
def test_saved_lse_forward_and_backward(bh, n, d, k, causal):
    """bsa_fine_attention_lse: the same O as bsa_fine_attention and each row's
    log2-sum-exp equal to the oracle's (its natural-log lse / ln 2; -inf for
    an empty row); bsa_fine_backward_lse with that lse: the oracle's
    gradients without the statistics pass."""
    import torch
    kb = 64
    t, do = _inputs(bh, n, d, seed=n + d + k + 3, kb=kb)
    q, kk, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    dout = parity.to_device(do, "bf16")
    idx_np = _random_lists(bh, n, kb, k, seed=11, causal=causal)
    lst = torch.from_numpy(idx_np).cuda().reshape(bh, n, k)
    mask = bsa.mask_struct(bsa.MASK_CAUSAL if causal else bsa.MASK_NONE)
    out = bsa.fine_attention(q, kk, v, lst, key_block=kb, mask=mask)
    out2, lse = bsa.fine_attention_lse(q, kk, v, lst, key_block=kb, causal=causal)
    assert torch.equal(out, out2)
    rows = oracle.all_rows(bh, n)
    _, ref_lse, _ = oracle.fine(t.q, t.k, t.v, kb, idx_np, rows, causal=causal)
    got = lse.cpu().numpy().reshape(-1).astype(np.float64)
    ref2 = ref_lse / np.log(2.0)
    empty = ~np.isfinite(ref2)
    assert empty.any() and (got[empty] == -np.inf).all()
    assert np.abs(got[~empty] - ref2[~empty]).max() <= 1e-3 * max(1.0, np.abs(ref2[~empty]).max())
    dq, dk, dv = bsa.fine_backward(q, kk, v, out, dout, lst, key_block=kb, causal=causal, lse=lse)
    rq, rk, rv = oracle.fine_backward(t.q, t.k, t.v, do, kb, idx_np, causal=causal)
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _grad_close(g.cpu().numpy(), ref, f"{name} (saved lse) bh={bh} n={n} d={d} k={k}")
    assert bsa.device_status() == 0


def test_saved_lse_outside_the_block_major_path_is_unsupported():
    import torch
    t, _ = _inputs(1, 256, 64, seed=2, kb=32)
    q, kk, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    lst = torch.zeros((1, 256, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(bsa.BsaError):
        bsa.fine_attention_lse(q, kk, v, lst, key_block=32)


@pytest.mark.parametrize("bh,n,d,k,causal", [
    (1, 1000, 64, 4, False),      # small enough for the one-launch forward without statistics
    (2, 4100, 64, 16, True),
    (1, 2100, 128, 8, False),
])
def test_training_step_forward_lse_then_backward(bh, n, d, k, causal):
    """bsa_forward_lse: a selection the oracle's check accepts, the output
    and the rows' log2-sum-exp of the oracle over that selection;
    bsa_fine_backward_lse over it then matches the oracle's gradients."""
    kb = 64
    t, do = _inputs(bh, n, d, seed=n + 5 * d + k, kb=kb)
    q, kk, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    dout = parity.to_device(do, "bf16")
    out, idx, lse = bsa.forward_lse(q, kk, v, kb, k, causal=causal)
    idx_np = idx.cpu().numpy().reshape(-1, k)
    rows = oracle.all_rows(bh, n)
    if not causal:
        s = oracle.scores(t.q, oracle.pool(t.k, kb), rows)
        oidx, kth = oracle.topk(s, k)
        parity.check_selection(idx_np, oidx, s, kth, -(-n // kb))
    o_ref, ref_lse, _ = oracle.fine(t.q, t.k, t.v, kb, idx_np, rows, causal=causal)
    parity.assert_close(parity.from_device(out).reshape(-1, d), o_ref, "bf16", "forward_lse output")
    ref2 = ref_lse / np.log(2.0)
    got = lse.cpu().numpy().reshape(-1).astype(np.float64)
    assert np.isfinite(ref2).all()
    assert np.abs(got - ref2).max() <= 1e-3 * max(1.0, np.abs(ref2).max())
    dq, dk, dv = bsa.fine_backward(q, kk, v, out, dout, idx, key_block=kb, causal=causal, lse=lse)
    rq, rk, rv = oracle.fine_backward(t.q, t.k, t.v, do, kb, idx_np, causal=causal)
    for name, g, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _grad_close(g.cpu().numpy(), ref, f"{name} (training step) bh={bh} n={n} d={d} k={k}")
    assert bsa.device_status() == 0
