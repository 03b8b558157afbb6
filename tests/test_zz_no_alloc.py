"""bsa_forward_noalloc: the forward for callers that cannot allocate device
memory at call time (its scratch is a static array inside the library).

Called through the C ABI and compared with bsa_forward (caller workspace) on
two consecutive calls with different inputs, so that leftovers of the first
call in the shared static scratch would show up in the second; the device's
free memory is the same before and after the second call.  Kept in a file of
its own that is collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from content_dependent_block_gb300 import _build, bsa
from tests import parity

pytestmark = pytest.mark.gpu


def _inputs(seed):
    w = workloads.WORKLOADS["dyn_n1024"]
    t = workloads.generate(w, seed=seed)
    return w, tuple(parity.to_device(getattr(t, x), "bf16") for x in "qkv")


def test_noalloc_matches_workspace_forward_on_two_calls():
    import torch
    _build.build()
    L = bsa.lib()
    for seed in (0, 1):
        w, (q, k, v) = _inputs(seed)
        ref_out, ref_idx = bsa.forward(q, k, v, w.key_block, w.topk)
        shape = bsa.Shape(w.bh, w.n, w.d, bsa.BF16)
        out = torch.full_like(q, float("nan"))
        idx = torch.full((w.bh, w.n, w.topk), -7, dtype=torch.int32, device=q.device)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = L.bsa_forward_noalloc(shape, bsa._ptr(q), bsa._ptr(k), bsa._ptr(v), w.key_block,
                                   w.topk, ctypes.c_float(0.0), bsa._ptr(out), bsa._ptr(idx),
                                   bsa._stream())
        assert rc == 0, L.bsa_last_error()
        torch.cuda.synchronize()
        if seed == 1:
            # after the first call (which may load the module holding the
            # static array), a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before
        assert bsa.device_status() == 0
        assert torch.equal(idx, ref_idx)
        got = parity.from_device(out).reshape(-1, w.d)
        ref = parity.out_f64(parity.from_device(ref_out).reshape(-1, w.d))
        parity.assert_close(got, ref, "bf16", f"noalloc call seed={seed}")
        assert np.isfinite(parity.out_f64(got)).all()


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    _build.build()
    L = bsa.lib()
    big = bsa.Shape(8, 131072, 128, bsa.BF16)          # needs far more than 32 MiB
    assert L.bsa_forward_workspace_size(big, 64, 32) > (32 << 20)
    fake = ctypes.c_void_p(0x10000)
    rc = L.bsa_forward_noalloc(big, fake, fake, fake, 64, 32, ctypes.c_float(0.0), fake, None,
                               None)
    assert rc == 4                                      # BSA_ERR_WORKSPACE
    assert b"static scratch" in L.bsa_last_error()
    # the 2-head, 1024-token, top-4 problem fits
    assert L.bsa_forward_workspace_size(bsa.Shape(2, 1024, 64, bsa.BF16), 64, 4) <= (32 << 20)
