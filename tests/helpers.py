"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances are the ones the task's acceptance criteria state, in the pages'
own form max|got - ref| / max|ref| ("Inside NVIDIA's cuDNN Graph API",
section 5, rel err; cudnn-frontend PR #554 compares relative to each
tensor's magnitude):
  O (bf16 output)  <= 1e-2 * max|ref|
  O (fp16 output)  <= 2e-3 * max|ref|
  LSE              |got - ref| <= 1e-3 (and -inf exactly where ref is -inf)
  dQ, dK, dV       <= 2e-2 * max|ref|
"""
from __future__ import annotations

import numpy as np
import torch

O_TOL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}
LSE_TOL = 1e-3
GRAD_TOL = 2e-2


def np64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, np.float64)


def rel_err(got, ref) -> float:
    got, ref = np64(got), np64(ref)
    if got.size == 0:
        return 0.0
    denom = np.max(np.abs(ref))
    num = np.max(np.abs(got - ref))
    if denom == 0:
        return float(num)
    return float(num / denom)


def check_rel(got, ref, tol, name):
    got_np = np64(got)
    assert np.all(np.isfinite(got_np)), f"{name}: non-finite values"
    e = rel_err(got_np, ref)
    assert e <= tol, f"{name}: rel err {e:.3e} > {tol:.1e}"
    return e


def check_lse(got, ref, name="lse"):
    got, ref = np64(got), np64(ref)
    dead = np.isneginf(ref)
    assert np.all(np.isneginf(got[dead])), f"{name}: dead rows must be -inf"
    live = ~dead
    if live.any():
        assert np.all(np.isfinite(got[live])), f"{name}: non-finite live rows"
        e = float(np.max(np.abs(got[live] - ref[live])))
        assert e <= LSE_TOL, f"{name}: max |dLSE| {e:.3e} > {LSE_TOL:.0e}"
        return e
    return 0.0
