"""Tolerances and helpers shared by the GPU parity tests.

Tolerances (stated for this method; the readings are explained in the design doc):
  * fp32 inputs: every element satisfies |y - y_ref| <= 1e-4 * max(|y_ref|, rms(y_ref))
    (a relative bound, floored at the output's rms so that outputs that
    cancel to ~0 are not judged by a vanishing denominator);
  * bf16 inputs (fp32 state): max |y - y_ref| <= 2e-3 * rms(y_ref).
The same rules apply to final states, each with its own rms.

Outputs stored in bf16 (the causal convolution with bf16 input) carry their own
rounding: bf16 keeps 8 significant bits, so rounding to nearest is off by at
most 2^-9 relative.  Such outputs pass iff every element has
|out - ref| <= 2^-8 * |ref| + 1e-5 * rms(ref) (twice the rounding bound, for the
fp32 arithmetic before it, plus a floor for outputs that cancel to ~0).
"""
from __future__ import annotations

import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-3
TOL_BF16_OUT = 2.0 ** -8


def rms(a):
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def err_f32(y, ref):
    """Largest |y - ref| / max(|ref|, rms(ref)) over all elements."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = np.maximum(np.abs(ref), max(rms(ref), 1e-30))
    return float(np.max(np.abs(y - ref) / scale))


def err_bf16(y, ref):
    """max |y - ref| / rms(ref)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(y - ref)) / max(rms(ref), 1e-30))


def check(y, ref, bf16: bool, what: str):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite values"
    if bf16:
        e = err_bf16(y, ref)
        assert e <= TOL_BF16, f"{what}: max|err|/rms = {e:.3e} > {TOL_BF16}"
    else:
        e = err_f32(y, ref)
        assert e <= TOL_F32, f"{what}: max err/max(|ref|,rms) = {e:.3e} > {TOL_F32}"
    return e


def host(t):
    return t.detach().float().cpu().numpy()


def check_bf16_out(out, ref, what: str):
    """Per-element check of a bf16-stored output against the fp64 reference."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (what, out.shape, ref.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite values"
    if ref.size == 0:
        return 0.0
    bound = TOL_BF16_OUT * np.abs(ref) + 1e-5 * rms(ref)
    worst = float(np.max(np.abs(out - ref) / bound))
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the bf16 output bound"
    return worst
