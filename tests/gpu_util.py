"""Shared helpers for the GPU parity tests: run the library, run the oracle, compare.

Tolerances (GPU bf16 output widened to fp64 vs the fp64 oracle):
    max |d out| <= 2e-2,  mean |d out| <= 2e-3,  max |d lse| <= 1e-3 over finite rows;
    rows whose oracle lse is -inf must come back with lse = -inf and out = 0 exactly.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_OUT_MAX = 2e-2
TOL_OUT_MEAN = 2e-3
TOL_LSE = 1e-3

MASK_IDS = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL,
            "blockdiag": oracle.MASK_BLOCKDIAG, "blockdiag_causal": oracle.MASK_BLOCKDIAG_CAUSAL}


def f32(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a bf16 CPU tensor (numpy has no bf16)."""
    return t.float().cpu().numpy()


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    out_ref = np.asarray(out_ref, dtype=np.float64)
    assert out_gpu.shape == out_ref.shape, f"{what}: out shape {out_gpu.shape} vs {out_ref.shape}"
    assert np.isfinite(out_gpu).all(), f"{what}: non-finite output"
    d = np.abs(out_gpu - out_ref)
    assert d.max() <= TOL_OUT_MAX, f"{what}: max |d out| {d.max():.3e}"
    assert d.mean() <= TOL_OUT_MEAN, f"{what}: mean |d out| {d.mean():.3e}"
    if lse_gpu is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        assert lse_gpu.shape == lse_ref.shape
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), inf_ref), f"{what}: -inf rows differ"
        assert not np.isnan(lse_gpu).any(), f"{what}: NaN lse"
        if (~inf_ref).any():
            dl = np.abs(lse_gpu[~inf_ref] - lse_ref[~inf_ref]).max()
            assert dl <= TOL_LSE, f"{what}: max |d lse| {dl:.3e}"
    return float(d.max()), float(d.mean())


def to_dev(*ts):
    return [t.cuda() for t in ts]
