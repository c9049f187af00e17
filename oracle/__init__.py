"""fp64 CPU oracle for the selective scan (S6) -- TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously correct reference that the CUDA library
is checked against.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The product package never
imports it, and nothing here imports the product package.

The arithmetic lives in ``ss_oracle.c`` (plain C, double precision,
sequential in time; see its header for the equations and their sources).
This module only compiles that file with gcc and marshals numpy arrays.

Inputs are the exact bytes the GPU sees: fp32 arrays, or bf16 passed as raw
``uint16`` bit patterns (``dtype="bf16"``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB = os.path.join(_HERE, "libss_oracle.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ss_oracle.c into libss_oracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.sso_scan.argtypes = [i64, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                             ctypes.c_int, vp, i64, dp, dp, dp, ctypes.c_int, ctypes.c_int]
    lib.sso_scan.restype = ctypes.c_int
    lib.sso_state_update.argtypes = [i64, i64, i64, ctypes.c_int, dp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, ctypes.c_int, vp, i64, dp, ctypes.c_int, ctypes.c_int]
    lib.sso_state_update.restype = ctypes.c_int
    lib.sso_delta.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_int]
    lib.sso_delta.restype = ctypes.c_double
    lib.sso_conv1d.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, ctypes.c_int, dp, ctypes.c_int]
    lib.sso_conv1d.restype = ctypes.c_int
    lib.sso_scan_bwd.argtypes = [i64, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp,
                                 ctypes.c_int, vp, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                 ctypes.c_int, ctypes.c_int]
    lib.sso_scan_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _in(a, dtype_code):
    """Contiguous view of an input array in the oracle's wire format."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = np.float32 if dtype_code == F32 else np.uint16
    if a.dtype != want:
        raise TypeError(f"expected {np.dtype(want).name} input, got {a.dtype}")
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(dtype):
    if dtype in ("f32", "fp32", "float32", F32):
        return F32
    if dtype in ("bf16", "bfloat16", BF16):
        return BF16
    raise ValueError(f"unknown dtype {dtype!r}")


def _threads(nthreads):
    return nthreads if nthreads and nthreads > 0 else (os.cpu_count() or 1)


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *,
         dtype="f32", h0=None, chans=None, nthreads=0, zoh=False, lib=None):
    """Full-sequence scan.  Shapes: u/delta/z (batch, dim, L); B/C (batch, N, L);
    A (dim, N); D/delta_bias (dim,).  Returns (y, h_last) as float64 arrays of
    shape (nchan, L) and (nchan, N), where nchan = batch*dim or len(chans).
    ``zoh`` uses the zero-order-hold input weight (exp(dt A) - 1)/A instead of dt."""
    code = _dtype_code(dtype)
    u, delta, B, C, z = (_in(x, code) for x in (u, delta, B, C, z))
    A, D, delta_bias = _f32(A), _f32(D), _f32(delta_bias)
    batch, dim, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and B.shape == (batch, N, L) and C.shape == (batch, N, L)
    assert A.shape == (dim, N)
    assert z is None or z.shape == u.shape
    ch = None if chans is None else np.ascontiguousarray(chans, dtype=np.int64)
    nch = batch * dim if ch is None else ch.shape[0]
    hh0 = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64).reshape(nch, N)
    y = np.empty((nch, L), dtype=np.float64)
    hl = np.empty((nch, N), dtype=np.float64)
    rc = (lib or _load()).sso_scan(batch, dim, N, L, code, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                          _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(ch), nch,
                          _ptr(hh0), _ptr(y), _ptr(hl), _threads(nthreads), int(bool(zoh)))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y, hl


def scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, dy, dlast=None,
             dtype="f32", h0=None, chans=None, want_BC=True, nthreads=0, zoh=False, lib=None):
    """Gradients of  sum(dy * y) + sum(dlast * h_last)  for the scan of ``scan``.

    ``dy`` is (batch, dim, L) (or (nchan, L) with ``chans``), ``dlast`` and ``h0``
    (nchan, N); all three are taken as float64.  Returns a dict of float64 arrays:
    du, ddelta, dz (None without z) shaped like u; dh0 (nchan, N); dB, dC
    (batch, N, L) over the listed channels (None unless ``want_BC``).  Without
    ``chans``: dA (dim, N), dD, ddelta_bias (dim,) summed over the batch rows.
    With ``chans``: dA_part (nchan, N), dD_part, dbias_part (nchan,) are each
    channel's own terms.  dD, ddelta_bias and dh0 are the gradients at the given
    D, delta_bias and h0, or at zero where those are absent."""
    code = _dtype_code(dtype)
    u, delta, B, C, z = (_in(x, code) for x in (u, delta, B, C, z))
    A, D, delta_bias = _f32(A), _f32(D), _f32(delta_bias)
    batch, dim, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and B.shape == (batch, N, L) and C.shape == (batch, N, L)
    assert A.shape == (dim, N) and (z is None or z.shape == u.shape)
    ch = None if chans is None else np.ascontiguousarray(chans, dtype=np.int64)
    nch = batch * dim if ch is None else ch.shape[0]
    f64 = lambda a, shape: None if a is None else np.ascontiguousarray(a, dtype=np.float64).reshape(shape)
    dyy, dl, hh0 = f64(dy, (nch, L)), f64(dlast, (nch, N)), f64(h0, (nch, N))
    du = np.zeros((nch, L)); ddelta = np.zeros((nch, L))
    dz = np.zeros((nch, L)) if z is not None else None
    dA_part = np.zeros((nch, N)); dD_part = np.zeros(nch); db_part = np.zeros(nch)
    dh0 = np.zeros((nch, N))
    dB = np.zeros((batch, N, L)) if want_BC else None
    dC = np.zeros((batch, N, L)) if want_BC else None
    rc = (lib or _load()).sso_scan_bwd(batch, dim, N, L, code, _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                       _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(ch), nch,
                                       _ptr(hh0), _ptr(dyy), _ptr(dl), _ptr(du), _ptr(ddelta), _ptr(dz),
                                       _ptr(dA_part), _ptr(dD_part), _ptr(db_part), _ptr(dh0), _ptr(dB), _ptr(dC),
                                       _threads(nthreads), int(bool(zoh)))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    out = dict(du=du, ddelta=ddelta, dz=dz, dh0=dh0, dB=dB, dC=dC)
    if ch is None:
        out["du"], out["ddelta"] = du.reshape(batch, dim, L), ddelta.reshape(batch, dim, L)
        if dz is not None:
            out["dz"] = dz.reshape(batch, dim, L)
        out["dA"] = dA_part.reshape(batch, dim, N).sum(axis=0)
        out["dD"] = dD_part.reshape(batch, dim).sum(axis=0)
        out["ddelta_bias"] = db_part.reshape(batch, dim).sum(axis=0)
    else:
        out.update(dA_part=dA_part, dD_part=dD_part, dbias_part=db_part)
    return out


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *,
                 dtype="f32", chans=None, nthreads=0, zoh=False, lib=None):
    """One decode step.  Shapes: u/delta/z (batch, dim); B/C (batch, N);
    state (nchan, N) float64, updated in place.  Returns y (nchan,) float64."""
    code = _dtype_code(dtype)
    u, delta, B, C, z = (_in(x, code) for x in (u, delta, B, C, z))
    A, D, delta_bias = _f32(A), _f32(D), _f32(delta_bias)
    batch, dim = u.shape
    N = A.shape[1]
    assert B.shape == (batch, N) and C.shape == (batch, N) and A.shape == (dim, N)
    ch = None if chans is None else np.ascontiguousarray(chans, dtype=np.int64)
    nch = batch * dim if ch is None else ch.shape[0]
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64 and state.flags.c_contiguous
            and state.shape == (nch, N)):
        raise TypeError("state must be a C-contiguous float64 array of shape (nchan, N)")
    y = np.empty((nch,), dtype=np.float64)
    rc = (lib or _load()).sso_state_update(batch, dim, N, code, _ptr(state), _ptr(u), _ptr(delta), _ptr(A),
                                  _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                  int(bool(softplus)), _ptr(ch), nch, _ptr(y), _threads(nthreads),
                                  int(bool(zoh)))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y


def conv1d(x, w, bias=None, silu=True, *, dtype="f32", nthreads=0, lib=None):
    """Causal depthwise convolution of width 4 (w[:, 3] on the current step), plus
    bias, then SiLU when ``silu``.  x (batch, dim, L) in the wire format of
    ``dtype``; w (dim, 4); bias (dim,).  Returns float64 (batch, dim, L)."""
    code = _dtype_code(dtype)
    x = _in(x, code)
    w, bias = _f32(w), _f32(bias)
    batch, dim, L = x.shape
    assert w.shape == (dim, 4) and (bias is None or bias.shape == (dim,))
    out = np.empty((batch, dim, L), dtype=np.float64)
    rc = (lib or _load()).sso_conv1d(batch, dim, L, code, _ptr(x), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(out),
                                     _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def step_size(draw: float, bias: float = 0.0, softplus: bool = True, lib=None) -> float:
    """dt for one raw value: softplus(draw + bias), or draw + bias when softplus is off."""
    return (lib or _load()).sso_delta(float(draw), float(bias), int(bool(softplus)))


class Variant:
    """The oracle API bound to another build of the same C source (used by the
    mutation tests, which compile deliberately broken copies on the CPU)."""

    def __init__(self, so_path):
        self.lib = _bind(so_path)

    def scan(self, *a, **k):
        return scan(*a, lib=self.lib, **k)

    def state_update(self, *a, **k):
        return state_update(*a, lib=self.lib, **k)

    def step_size(self, *a, **k):
        return step_size(*a, lib=self.lib, **k)

    def scan_bwd(self, *a, **k):
        return scan_bwd(*a, lib=self.lib, **k)

    def conv1d(self, *a, **k):
        return conv1d(*a, lib=self.lib, **k)


class _Default:
    scan = staticmethod(scan)
    scan_bwd = staticmethod(scan_bwd)
    state_update = staticmethod(state_update)
    step_size = staticmethod(step_size)
    conv1d = staticmethod(conv1d)


default = _Default()
