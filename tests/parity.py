"""Shared parity helpers: tolerances, selection checks, host<->device moves.

Tolerances (stated for the method's outputs; bf16 inputs, fp32 accumulate):
  bf16 outputs  max-abs error <= 2e-2 and relative L2 error <= 5e-3
  fp32 outputs  max-abs error <= 1e-4
  selection     bit-exact block-id sets, except that a block may differ
                when its oracle score lies within 1e-3 relative of the
                oracle's k-th score: |S_b - s_k| <= 1e-3 * max(|s_k|, 1e-3)
"""
from __future__ import annotations

import numpy as np

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
FP32_MAX_ABS = 1e-4
TIE_REL = 1e-3
TIE_FLOOR = 1e-3


def to_device(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def from_device(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def out_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "output"):
    got = out_f64(got).reshape(ref.shape)
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    if dtype == "bf16":
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
            f"{what}: max-abs {max_abs:.3e} (<= {BF16_MAX_ABS}), rel-L2 {rel:.3e} (<= {BF16_REL_L2})"
        return max_abs, rel
    assert max_abs <= FP32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} (<= {FP32_MAX_ABS})"
    return max_abs, None


def check_selection(gpu_idx: np.ndarray, orc_idx: np.ndarray, orc_scores: np.ndarray,
                    kth: np.ndarray, nb: int):
    """Validate GPU top-k rows against the oracle's, with the tie band.

    Returns the number of rows whose sets differ (all within the band)."""
    k = gpu_idx.shape[1]
    kk = min(k, nb)
    differing = 0
    for r in range(gpu_idx.shape[0]):
        g = gpu_idx[r]
        assert (g[kk:] == -1).all(), f"row {r}: padding past min(k, nb) must be -1: {g}"
        gs = g[:kk]
        assert (gs >= 0).all() and (gs < nb).all(), f"row {r}: ids out of range: {g}"
        assert (np.diff(gs) > 0).all(), f"row {r}: ids not strictly ascending: {g}"
        o = orc_idx[r][:kk]
        if np.array_equal(gs, o):
            continue
        differing += 1
        band = TIE_REL * max(abs(kth[r]), TIE_FLOOR)
        for b in np.setxor1d(gs, o):
            assert abs(orc_scores[r, b] - kth[r]) <= band, (
                f"row {r}: block {b} differs but its oracle score {orc_scores[r, b]:.6g} is "
                f"outside the tie band of the k-th score {kth[r]:.6g} (band {band:.3g})")
    return differing
