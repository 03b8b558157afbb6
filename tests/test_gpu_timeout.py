"""The failure path of the bounded waits, on the GPU, without a fault.

Every hand-off of the tensor-core kernels waits on an mbarrier or on a
counter in global memory, and each wait gives up after a time limit,
records BSA_ERR_TIMEOUT in the device status word and lets the kernel
return.  bsa_selftest_wait_timeout runs those same wait functions on a
barrier no thread arrives on and a counter no thread raises, with a short
limit; these tests check that the wait runs out in about that time, the
status word says so, and the context stays usable: a forward right after it
matches the oracle with a clean status.
"""
import time

import pytest

import oracle
import workloads
from content_dependent_block_gb300 import bsa
from tests import parity

pytestmark = pytest.mark.gpu

TIMEOUT = 6


@pytest.fixture(scope="module")
def torch():
    import torch
    bsa.lib()
    return torch


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "counter"])
@pytest.mark.parametrize("limit_ms", [1, 20])
def test_wait_runs_out_and_reports(torch, kind, limit_ms):
    assert bsa.device_status() in (0, TIMEOUT)      # start from a clear word
    assert bsa.device_status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bsa.selftest_wait_timeout(kind, limit_ms * 1_000_000)
    torch.cuda.synchronize()                        # the kernel came back
    dt = time.perf_counter() - t0
    assert bsa.device_status() == TIMEOUT
    assert bsa.device_status() == 0                 # reading cleared it
    # it waited at least the limit, and gave up within a bounded time after it
    assert dt >= limit_ms * 1e-3 * 0.9
    assert dt < limit_ms * 1e-3 + 1.0


def test_forward_after_a_timeout_is_clean(torch):
    bsa.device_status()
    bsa.selftest_wait_timeout(0, 1_000_000)
    torch.cuda.synchronize()
    assert bsa.device_status() == TIMEOUT
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w)
    q, k, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    out, idx = bsa.forward(q, k, v, w.key_block, w.topk)
    torch.cuda.synchronize()
    assert bsa.device_status() == 0
    rows = oracle.all_rows(w.bh, w.n)
    s = oracle.scores(t.q, oracle.pool(t.k, w.key_block), rows)
    oidx, kth = oracle.topk(s, w.topk)
    gidx = idx.cpu().numpy().reshape(-1, w.topk)
    parity.check_selection(gidx, oidx, s, kth, w.nb)
    o_ref, _, _ = oracle.fine(t.q, t.k, t.v, w.key_block, gidx, rows)
    parity.assert_close(parity.from_device(out).reshape(-1, w.d), o_ref, "bf16",
                        "forward after a timeout")


def test_a_pending_timeout_makes_kernels_skip_work(torch):
    """While the word holds BSA_ERR_TIMEOUT, kernels return early (their
    results are invalid anyway); once it is read, work runs again."""
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w)
    q, k, v = (parity.to_device(getattr(t, x), "bf16") for x in "qkv")
    bsa.device_status()
    bsa.selftest_wait_timeout(1, 1_000_000)
    # a second self-test while the word is set gives up at once
    t0 = time.perf_counter()
    bsa.selftest_wait_timeout(1, 500_000_000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 0.4
    assert bsa.device_status() == TIMEOUT
    out, _ = bsa.forward(q, k, v, w.key_block, w.topk)
    torch.cuda.synchronize()
    assert bsa.device_status() == 0
    assert torch.isfinite(out.float()).all()
