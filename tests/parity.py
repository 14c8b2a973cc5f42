"""Shared helpers of the parity tests: tolerances, conversions, comparisons.

Tolerances (stated for bf16 inputs with fp32 accumulation):
  O      max|gpu - oracle| <= 1e-2
  LSE    max|gpu - oracle| <= 1e-3
  dQ, dK, dV   max|gpu - oracle| <= 2e-2 * max|oracle|
Integer work (split bounds, tile order) is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2


def np64(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor -> float64 numpy (exact upcast)."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def max_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.size == 0:
        return 0.0
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    d = np.where(np.isnan(d), np.inf, d)
    return float(d.max())


def check_o(gpu, ref, what="O"):
    e = max_err(gpu, ref)
    assert e <= TOL_O, f"{what}: max|diff| {e:.3e} > {TOL_O}"
    return e


def check_lse(gpu, ref, what="LSE"):
    e = max_err(gpu, ref)
    assert e <= TOL_LSE, f"{what}: max|diff| {e:.3e} > {TOL_LSE}"
    return e


def check_grad(gpu, ref, what):
    ref = np.asarray(ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    e = max_err(gpu, ref)
    assert e <= TOL_GRAD_REL * max(scale, 1e-30) or (scale == 0.0 and e == 0.0), \
        f"{what}: max|diff| {e:.3e} > {TOL_GRAD_REL} * max|ref| ({scale:.3e})"
    return e, scale


def to_cuda(d: dict, keys) -> dict:
    out = dict(d)
    for k in keys:
        out[k] = d[k].cuda()
    return out
