"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances (bf16 output against the fp64 oracle on the same bf16 inputs):
  O  : max |err| <= 2e-2 and mean |err| <= 2e-3
  lse: |err| / max(|lse_ref|, 1) <= 1e-3, and -inf exactly where the oracle has -inf
"""
from __future__ import annotations

import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, dtype=np.float64)
    lse = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: O max abs err {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean abs err {err.mean():.3e}"
    ref_inf = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), ref_inf), f"{what}: -inf lse pattern differs"
    assert not np.any(np.isnan(lse)), f"{what}: NaN lse"
    fin = ~ref_inf
    if fin.any():
        rel = np.abs(lse[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)
        assert rel.max() <= LSE_REL, f"{what}: lse rel err {rel.max():.3e}"
    return float(err.max()), float(err.mean())
