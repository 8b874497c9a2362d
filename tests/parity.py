"""Tolerances and comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (bf16 inputs and outputs, fp32 accumulation on the GPU):
  O      per element |o - o_ref| <= max(1e-2, ulp_bf16(o_ref)/2 + 2^-8 * spread + 1e-3)
         where spread_ic = sum_j P_ij |v_jc - O_ic| (from the oracle).  The
         first term is the rounding of the bf16 output (the flat 1e-2 cannot
         hold where |o_ref| >= 4: a correctly rounded bf16 value there can be
         1/64 away from the exact one); the second bounds the effect of the
         bf16 rounding of the weights P that the P V product uses (relative
         error <= 2^-9 per weight, <= 2^-8 after renormalisation).  When no
         spread is given only the first term is used.
  LSE    max-abs <= 1e-3
  dQ, dK, dV  max-abs <= 2e-2 * max|grad_ref| per tensor
"""
from __future__ import annotations

import numpy as np
import torch

O_ABS = 1e-2
LSE_ABS = 1e-3
GRAD_REL = 2e-2


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), np.finfo(np.float64).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def o_bound(o_ref: np.ndarray, spread=None) -> np.ndarray:
    if spread is None:
        return np.maximum(O_ABS, 0.5 * bf16_ulp(o_ref) + 2e-3)
    return np.maximum(O_ABS, 0.5 * bf16_ulp(o_ref) + 2.0 ** -8 * spread + 1e-3)


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def check_o(o_gpu, o_ref, what="", spread=None):
    """Returns (max abs error, number of elements above the flat 1e-2)."""
    o_gpu, o_ref = to_np(o_gpu), to_np(o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    err = np.abs(o_gpu - o_ref)
    bound = o_bound(o_ref, None if spread is None else to_np(spread))
    bad = err > bound
    assert not bad.any(), (f"{what}: O max err {err.max():.3e}, {int(bad.sum())} elements over bound; "
                           f"worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    over_flat = int((err > O_ABS).sum())
    if over_flat:
        print(f"[parity] {what}: {over_flat} of {err.size} O elements above the flat 1e-2 "
              f"(max {err.max():.3e}), all within the derived bound")
    return float(err.max()), over_flat


def check_lse(lse_gpu, lse_ref, what=""):
    lse_gpu, lse_ref = to_np(lse_gpu), to_np(lse_ref)
    assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    err = float(np.max(np.abs(lse_gpu - lse_ref)))
    assert err <= LSE_ABS, f"{what}: LSE max err {err:.3e}"
    return err


def check_grad(g_gpu, g_ref, name, what=""):
    g_gpu, g_ref = to_np(g_gpu), to_np(g_ref)
    assert np.all(np.isfinite(g_gpu)), f"{what}: non-finite {name}"
    scale = float(np.max(np.abs(g_ref)))
    err = float(np.max(np.abs(g_gpu - g_ref)))
    assert err <= GRAD_REL * scale + 1e-6, f"{what}: {name} max err {err:.3e} vs bound {GRAD_REL * scale:.3e}"
    return err, scale
