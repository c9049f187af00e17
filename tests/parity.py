"""Tolerances and helpers shared by the GPU parity tests.

Tolerances (stated for this method):
  * fp32 inputs: every element satisfies |y - y_ref| <= 1e-4 * max(|y_ref|, rms(y_ref))
    (a relative bound, floored at the output's rms so that outputs that
    cancel to ~0 are not judged by a vanishing denominator);
  * bf16 inputs (fp32 state): max |y - y_ref| <= 2e-3 * rms(y_ref).
The same rules apply to final states, each with its own rms.

Beside the pass/fail figure every comparison also measures the relative error
WITHOUT the rms floor, max |y - y_ref| / |y_ref| over the elements with
|y_ref| >= 1e-2 * rms(y_ref), so that what the floor hides is visible.  When the
environment variable SS_PARITY_LOG names a file, each comparison appends one
JSON line there: the label, the element count, max |err|, rms(ref), the judged
figure and the unfloored relative error.

Outputs stored in bf16 (the causal convolution with bf16 input) carry their own
rounding: bf16 keeps 8 significant bits, so rounding to nearest is off by at
most 2^-9 relative.  Such outputs pass iff every element has
|out - ref| <= 2^-8 * |ref| + 1e-5 * rms(ref) (twice the rounding bound, for the
fp32 arithmetic before it, plus a floor for outputs that cancel to ~0).

Outputs too large to hold twice on the host (the full-size workloads) are
compared block by block with StreamCheck, which reaches exactly the outcome of
check() on the whole array without keeping it.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-3
TOL_BF16_OUT = 2.0 ** -8
UNFLOORED_ABOVE = 1e-2     # the unfloored relative error is taken over |ref| >= this * rms(ref)


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


def rel_unfloored(y, ref, floor_abs):
    """max |y - ref| / |ref| over the elements with |ref| >= floor_abs (0 if there are none)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    keep = np.abs(ref) >= max(floor_abs, 1e-300)
    if not np.any(keep):
        return 0.0
    return float(np.max(np.abs(y[keep] - ref[keep]) / np.abs(ref[keep])))


def log_result(what, **fields):
    path = os.environ.get("SS_PARITY_LOG")
    if not path:
        return
    rec = {"what": what}
    rec.update({k: (float(v) if isinstance(v, (np.floating, float)) else v) for k, v in fields.items()})
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def check(y, ref, bf16: bool, what: str):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite values"
    r = rms(ref)
    if bf16:
        e = err_bf16(y, ref)
    else:
        e = err_f32(y, ref)
    log_result(what, n=int(ref.size), max_abs_err=float(np.max(np.abs(y - ref))) if ref.size else 0.0, rms_ref=r,
               judged=e, rule="max|err|/rms" if bf16 else "max err/max(|ref|,rms)",
               tol=TOL_BF16 if bf16 else TOL_F32, rel_unfloored=rel_unfloored(y, ref, UNFLOORED_ABOVE * r))
    if bf16:
        assert e <= TOL_BF16, f"{what}: max|err|/rms = {e:.3e} > {TOL_BF16}"
    else:
        assert e <= TOL_F32, f"{what}: max err/max(|ref|,rms) = {e:.3e} > {TOL_F32}"
    return e


class StreamCheck:
    """check() over an output delivered in blocks (any split of the elements).

    bf16 rule: max |err| and sum(ref^2) accumulate, so the outcome is exact.
    fp32 rule: an element passes outright when |err| <= tol * |ref|; otherwise
    it needs |err| <= tol * rms(ref).  The largest |err| among the elements that
    did not pass outright is kept, and finish() compares it with tol * rms, which
    is the outcome of check() on the whole array.  The reported figures that
    depend on the final rms (the floored error, the unfloored relative error's
    threshold) use each block's own rms for the split, which only matters for
    the report, not for the outcome."""

    def __init__(self, what: str, bf16: bool, tol: float | None = None):
        self.what, self.bf16 = what, bf16
        self.tol = tol if tol is not None else (TOL_BF16 if bf16 else TOL_F32)
        self.n, self.ss, self.max_err, self.worst_out = 0, 0.0, 0.0, 0.0
        self.rel_unf, self.floored = 0.0, 0.0

    def add(self, y, ref):
        y = np.asarray(y, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert y.shape == ref.shape, (self.what, y.shape, ref.shape)
        if ref.size == 0:
            return
        assert np.all(np.isfinite(y)), f"{self.what}: non-finite values"
        err = np.abs(y - ref)
        aref = np.abs(ref)
        self.n += ref.size
        self.ss += float(np.sum(ref * ref))
        self.max_err = max(self.max_err, float(np.max(err)))
        if not self.bf16:
            out = err > self.tol * aref
            if np.any(out):
                self.worst_out = max(self.worst_out, float(np.max(err[out])))
        rb = math.sqrt(float(np.mean(ref * ref)))
        self.rel_unf = max(self.rel_unf, rel_unfloored(y, ref, UNFLOORED_ABOVE * rb))
        self.floored = max(self.floored, float(np.max(err / np.maximum(aref, max(rb, 1e-30)))))

    def finish(self):
        r = math.sqrt(self.ss / self.n) if self.n else 0.0
        judged = (self.max_err / max(r, 1e-30)) if self.bf16 else self.floored
        log_result(self.what, n=self.n, max_abs_err=self.max_err, rms_ref=r, judged=judged,
                   rule="max|err|/rms" if self.bf16 else "max err/max(|ref|,rms)", tol=self.tol,
                   rel_unfloored=self.rel_unf, streamed=True)
        if self.bf16:
            assert self.max_err <= self.tol * r, f"{self.what}: max|err|/rms = {judged:.3e} > {self.tol}"
        else:
            assert self.worst_out <= self.tol * r, \
                f"{self.what}: an element is off by {self.worst_out:.3e} > {self.tol} * max(|ref|, rms {r:.3e})"
        return judged


class StreamCheckBf16Out:
    """check_bf16_out() over an output delivered in blocks: an element passes outright
    when |err| <= 2^-8 |ref|; the largest excess |err| - 2^-8 |ref| among the others is
    compared with 1e-5 * rms(ref) at the end, the outcome of check_bf16_out on the whole."""

    def __init__(self, what: str):
        self.what, self.n, self.ss, self.excess, self.max_err = what, 0, 0.0, 0.0, 0.0

    def add(self, out, ref):
        out = np.asarray(out, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert out.shape == ref.shape, (self.what, out.shape, ref.shape)
        if ref.size == 0:
            return
        assert np.all(np.isfinite(out)), f"{self.what}: non-finite values"
        err = np.abs(out - ref)
        self.n += ref.size
        self.ss += float(np.sum(ref * ref))
        self.max_err = max(self.max_err, float(np.max(err)))
        self.excess = max(self.excess, float(np.max(err - TOL_BF16_OUT * np.abs(ref))))

    def finish(self):
        r = math.sqrt(self.ss / self.n) if self.n else 0.0
        floor = 1e-5 * r
        log_result(self.what, n=self.n, max_abs_err=self.max_err, rms_ref=r,
                   judged=max(self.excess, 0.0) / max(floor, 1e-300),
                   rule="largest |err| - 2^-8 |ref| over 1e-5 rms", tol=1.0, streamed=True)
        assert self.excess <= floor, f"{self.what}: an element exceeds the bf16 output bound"


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
    log_result(what, n=int(ref.size), max_abs_err=float(np.max(np.abs(out - ref))), rms_ref=rms(ref), judged=worst,
               rule="max |err| / (2^-8 |ref| + 1e-5 rms)", tol=1.0)
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the bf16 output bound"
    return worst
