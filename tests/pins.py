"""Pins for the fp64 oracle: checks against facts fixed by the pages and by
mathematics, independent of the oracle's own recurrence code.

Each pin takes an oracle object (``oracle.default`` or an ``oracle.Variant``)
and raises AssertionError when the oracle disagrees.  The same pins are run
against deliberately broken builds of the oracle in ``test_oracle_mutants.py``
to show that a plausible mistake fails at least one of them.

Sources (page titles and sections):
  * "State Space Models and Mamba" (multigrid.ai/learn/mamba-ssm):
    "It is a linear recurrence" (the recurrence and readout), "Why a linear
    recurrence can be trained in parallel" (the unrolled sum and the
    convolution kernel C A^k B), "Selective state" (delta_t, A_t, h_t; large
    delta resets toward the token, small delta keeps the state), "What it
    costs" (scan and recurrence modes must agree).
  * "State Space Models Explained ..." (mernstackdev.com): "A tiny example you
    can run" and "Selectivity, shown in code" (printed outputs, stored under
    tests/golden/).
  * "Mamba: Linear-Time Sequence Modeling with Selective State Spaces"
    (azimuth.plus): the selection mechanism (delta = softplus(Linear(x))) and
    Theorem 1 (N = 1 reduces to a gated RNN).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [float(x) for x in v.split()]
    return out


def f32(x):
    return np.asarray(x, dtype=np.float32)


def softplus64(x):
    x = np.asarray(x, dtype=np.float64)
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)


def silu64(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def rand_problem(seed, batch=2, dim=3, N=4, L=24, gate=True, with_D=True, with_bias=True):
    """Small random problem, every parameter varying with channel and time."""
    r = np.random.default_rng(seed)
    u = f32(r.normal(size=(batch, dim, L)))
    draw = f32(r.normal(size=(batch, dim, L)) - 1.0)
    A = f32(-np.exp(r.uniform(-1.0, 1.5, size=(dim, N))))
    B = f32(r.normal(size=(batch, N, L)))
    C = f32(r.normal(size=(batch, N, L)))
    D = f32(r.normal(size=(dim,))) if with_D else None
    z = f32(r.normal(size=(batch, dim, L))) if gate else None
    bias = f32(r.uniform(-3.0, 0.5, size=(dim,))) if with_bias else None
    return dict(u=u, delta=draw, A=A, B=B, C=C, D=D, z=z, delta_bias=bias)


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- the pins

def pin_tiny_example(orc):
    """Printed outputs of the scalar worked example (tests/golden/tiny_example.txt)."""
    g = read_golden("tiny_example.txt")
    sig = f32(g["signal"]).reshape(1, 1, -1)
    L = sig.shape[-1]
    for key in ("a=0.9", "a=0.3"):
        a = float(key.split("=")[1])
        y, h = orc.scan(sig, f32(np.ones((1, 1, L))), f32([[math.log(a)]]), f32(np.ones((1, 1, L))),
                        f32(np.ones((1, 1, L))), softplus=False)
        err = np.max(np.abs(y[0] - np.asarray(g[key])))
        assert err <= g["tolerance"][0], (key, y[0], g[key])
        assert abs(h[0, 0] - y[0, -1]) < 1e-12      # C = 1: the last output is the state


def pin_selective_toy(orc):
    """Printed outputs of the toy keep/write gate (tests/golden/selective_toy.txt)."""
    g = read_golden("selective_toy.txt")
    vals = np.asarray(g["values"])
    imp = np.asarray(g["important"]) > 0
    L = len(vals)
    lo = math.log(0.95) / math.log(0.2)
    dt = np.where(imp, 1.0, lo)
    B = np.where(imp, 1.0, 0.05 / lo)
    y, _ = orc.scan(f32(vals).reshape(1, 1, L), f32(dt).reshape(1, 1, L), f32([[math.log(0.2)]]),
                    f32(B).reshape(1, 1, L), f32(np.ones((1, 1, L))), softplus=False)
    err = np.max(np.abs(y[0] - np.asarray(g["outputs"])))
    assert err <= g["tolerance"][0], (y[0], g["outputs"])


def pin_lti_convolution(orc):
    """Time-invariant case equals the convolution with kernel K_k = sum_n C_n exp(k dt A_n) dt B_n,
    plus the D skip, times the SiLU gate."""
    r = np.random.default_rng(11)
    batch, dim, N, L = 2, 3, 4, 40
    u = f32(r.normal(size=(batch, dim, L)))
    draw0 = f32(r.normal(size=(batch, dim, 1)))
    bias = f32(r.uniform(-2.0, 0.0, size=(dim,)))
    A = f32(-np.exp(r.uniform(-1.0, 1.0, size=(dim, N))))
    B0 = f32(r.normal(size=(batch, N, 1)))
    C0 = f32(r.normal(size=(batch, N, 1)))
    D = f32(r.normal(size=(dim,)))
    z = f32(r.normal(size=(batch, dim, L)))
    y, _ = orc.scan(u, np.repeat(draw0, L, axis=2), A, np.repeat(B0, L, axis=2), np.repeat(C0, L, axis=2),
                    D=D, z=z, delta_bias=bias, softplus=True)
    y = y.reshape(batch, dim, L)
    k = np.arange(L)
    for b in range(batch):
        for d in range(dim):
            dt = softplus64(float(draw0[b, d, 0]) + float(bias[d]))
            K = np.zeros(L)
            for n in range(N):
                K += float(C0[b, n, 0]) * np.exp(k * dt * float(A[d, n])) * dt * float(B0[b, n, 0])
            conv = np.convolve(u[b, d].astype(np.float64), K)[:L]
            want = (conv + float(D[d]) * u[b, d].astype(np.float64)) * silu64(z[b, d])
            assert rel_err(y[b, d], want) < 1e-11, (b, d, rel_err(y[b, d], want))


def pin_unrolled_sum(orc):
    """Brute-force unrolling: h_t = (prod_{r<=t} Abar_r) h0 + sum_{s<=t} (prod_{s<r<=t} Abar_r) dt_s B_s u_s,
    every quantity varying with channel and time, with an initial state."""
    p = rand_problem(5)
    batch, dim, L = p["u"].shape
    N = p["A"].shape[1]
    r = np.random.default_rng(6)
    h0 = r.normal(size=(batch * dim, N))
    y, hl = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"],
                     delta_bias=p["delta_bias"], softplus=True, h0=h0)
    for b in range(batch):
        for d in range(dim):
            c = b * dim + d
            dt = softplus64(p["delta"][b, d].astype(np.float64) + float(p["delta_bias"][d]))
            logA = dt[:, None] * p["A"][d].astype(np.float64)[None, :]          # (L, N)
            cum = np.cumsum(logA, axis=0)                                          # sum_{r<=t}
            inp = dt[:, None] * p["B"][b].T.astype(np.float64) * p["u"][b, d].astype(np.float64)[:, None]
            for t in range(L):
                h = np.exp(cum[t]) * h0[c]
                for s in range(t + 1):
                    h = h + np.exp(cum[t] - cum[s]) * inp[s]
                yt = float(np.dot(p["C"][b, :, t].astype(np.float64), h)) + float(p["D"][d]) * float(p["u"][b, d, t])
                yt *= float(silu64(p["z"][b, d, t]))
                assert abs(y[c, t] - yt) <= 1e-10 * max(1.0, abs(yt)), (b, d, t, y[c, t], yt)
                if t == L - 1:
                    assert np.max(np.abs(hl[c] - h)) <= 1e-10 * max(1.0, np.max(np.abs(h)))


def pin_zero_step_keeps_state(orc):
    """dt = 0 exactly: Abar = 1 and no input enters, so the state is unchanged and y = C h0 + D u
    (gated); in recurrence mode the state is bitwise unchanged."""
    p = rand_problem(7)
    batch, dim, L = p["u"].shape
    N = p["A"].shape[1]
    h0 = np.random.default_rng(8).normal(size=(batch * dim, N))
    zero = f32(np.zeros_like(p["u"]))
    y, hl = orc.scan(p["u"], zero, p["A"], p["B"], p["C"], D=p["D"], z=p["z"], softplus=False, h0=h0)
    assert np.array_equal(hl, h0)
    for b in range(batch):
        for d in range(dim):
            c = b * dim + d
            want = (p["C"][b].T.astype(np.float64) @ h0[c] + float(p["D"][d]) * p["u"][b, d].astype(np.float64)) \
                * silu64(p["z"][b, d])
            assert rel_err(y[c], want) < 1e-13
    st = h0.copy()
    yd = orc.state_update(st, p["u"][:, :, 0].copy(), zero[:, :, 0].copy(), p["A"], p["B"][:, :, 0].copy(),
                          p["C"][:, :, 0].copy(), D=p["D"], z=p["z"][:, :, 0].copy(), softplus=False)
    assert np.array_equal(st, h0)
    assert rel_err(yd, y[:, 0]) < 1e-13


def pin_large_step_resets(orc):
    """A very large dt with A <= -1 sends Abar to 0, so the state holds only the current token's
    input: h_t = dt B_t u_t and y_t = dt u_t sum_n C_t B_t + D u_t, whatever came before."""
    p = rand_problem(9, gate=False)
    batch, dim, L = p["u"].shape
    A = f32(-1.0 - np.abs(p["A"]))
    big = 1.0e4
    y, hl = orc.scan(p["u"], f32(np.full_like(p["u"], big)), A, p["B"], p["C"], D=p["D"], softplus=False,
                     h0=np.ones((batch * dim, A.shape[1])))
    for b in range(batch):
        for d in range(dim):
            c = b * dim + d
            cb = np.sum(p["C"][b].astype(np.float64) * p["B"][b].astype(np.float64), axis=0)
            u64 = p["u"][b, d].astype(np.float64)
            want = big * u64 * cb + float(p["D"][d]) * u64
            assert rel_err(y[c], want) < 1e-12
            assert rel_err(hl[c], big * p["B"][b, :, -1].astype(np.float64) * float(p["u"][b, d, -1])) < 1e-12


def pin_recurrence_equals_scan(orc):
    """Recurrence mode (one token at a time from a zero state) reproduces the scan: y and final state."""
    p = rand_problem(13)
    batch, dim, L = p["u"].shape
    N = p["A"].shape[1]
    y, hl = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"],
                     delta_bias=p["delta_bias"], softplus=True)
    st = np.zeros((batch * dim, N))
    for t in range(L):
        yt = orc.state_update(st, p["u"][:, :, t].copy(), p["delta"][:, :, t].copy(), p["A"],
                              p["B"][:, :, t].copy(), p["C"][:, :, t].copy(), D=p["D"], z=p["z"][:, :, t].copy(),
                              delta_bias=p["delta_bias"], softplus=True)
        assert rel_err(yt, y[:, t]) < 1e-13, t
    assert rel_err(st, hl) < 1e-13


def pin_linear_and_causal(orc):
    """For fixed dt, B, C, z the map u -> y is linear (no nonlinearity around the state), and
    causal: changing u at t0 leaves every earlier output bitwise unchanged."""
    p = rand_problem(15)
    r = np.random.default_rng(16)
    u2 = f32(r.normal(size=p["u"].shape))
    kw = dict(D=p["D"], z=p["z"], delta_bias=p["delta_bias"], softplus=True)
    y1, _ = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], **kw)
    y2, _ = orc.scan(u2, p["delta"], p["A"], p["B"], p["C"], **kw)
    y12, _ = orc.scan(f32(p["u"].astype(np.float64) + u2), p["delta"], p["A"], p["B"], p["C"], **kw)
    assert np.max(np.abs(y12 - (y1 + y2))) <= 1e-6 * np.max(np.abs(y12))   # u1+u2 rounded to fp32
    t0 = 10
    u3 = p["u"].copy()
    u3[:, :, t0] += 1.0
    y3, _ = orc.scan(u3, p["delta"], p["A"], p["B"], p["C"], **kw)
    assert np.array_equal(y3[:, :t0], y1[:, :t0])
    assert np.all(np.any(y3[:, t0:] != y1[:, t0:], axis=1))


def pin_gated_rnn_decay(orc):
    """Theorem 1 (N = 1, A = -1, dt = softplus(g)): the decay factor exp(-softplus(g)) equals
    1 - sigmoid(g), the forget gate of the gated RNN.  Under the Euler input term dt*B*x the
    input weight is softplus(g), not sigmoid(g): the theorem's input weight needs the
    zero-order-hold term, which this scan does not use."""
    g = f32(np.linspace(-6.0, 6.0, 25)).reshape(1, 25)
    one = f32(np.ones((1, 25)))
    A = f32(-np.ones((25, 1)))
    st = np.ones((25, 1))
    orc.state_update(st, f32(np.zeros((1, 25))), g, A, f32(np.ones((1, 1))), f32(np.ones((1, 1))), softplus=True)
    sig = 1.0 / (1.0 + np.exp(-g[0].astype(np.float64)))
    assert np.max(np.abs(st[:, 0] - (1.0 - sig))) < 1e-14
    st = np.zeros((25, 1))
    orc.state_update(st, one, g, A, f32(np.ones((1, 1))), f32(np.ones((1, 1))), softplus=True)
    assert np.max(np.abs(st[:, 0] - np.log1p(np.exp(g[0].astype(np.float64))))) < 1e-12
    assert np.max(np.abs(st[:, 0] - sig)) > 0.1


def pin_inverse_softplus_bias(orc):
    """delta_bias = log(expm1(x)) with a zero raw delta gives dt = x: the bias enters before the
    softplus.  Observed through the scan with A = 0, B = C = u = 1, L = 1 (then y = dt)."""
    xs = np.linspace(1e-3, 1e-1, 17)
    bias = f32(np.log(np.expm1(xs)))
    dim = len(xs)
    one = f32(np.ones((1, dim, 1)))
    y, _ = orc.scan(one, f32(np.zeros((1, dim, 1))), f32(np.zeros((dim, 1))), f32(np.ones((1, 1, 1))),
                    f32(np.ones((1, 1, 1))), delta_bias=bias, softplus=True)
    want = softplus64(bias.astype(np.float64))
    assert rel_err(y[:, 0], want) < 1e-14
    assert np.max(np.abs(y[:, 0] - xs) / xs) < 1e-6          # fp32 rounding of the bias only
    for x, b in zip(xs, bias):
        assert abs(orc.step_size(0.0, float(b), True) - x) / x < 1e-6
    # large and very negative arguments: softplus(x) -> x and -> exp(x)
    assert abs(orc.step_size(40.0, 0.0, True) - 40.0) < 1e-12
    assert abs(orc.step_size(-40.0, 0.0, True) - math.exp(-40.0)) < 1e-28
    assert orc.step_size(-2.5, 0.5, False) == -2.0


def pin_bf16_widening(orc):
    """bf16 inputs are widened exactly: a bf16 problem and the fp32 problem holding the same
    values give bitwise identical results."""
    p = rand_problem(17)
    def to_bf16_bits(a):
        bits = np.asarray(a, dtype=np.float32).view(np.uint32)
        return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    def from_bits(b):
        return (b.astype(np.uint32) << 16).view(np.float32)
    wires = {k: to_bf16_bits(p[k]) for k in ("u", "delta", "B", "C", "z")}
    vals = {k: from_bits(v) for k, v in wires.items()}
    kw = dict(D=p["D"], delta_bias=p["delta_bias"], softplus=True)
    yb, hb = orc.scan(wires["u"], wires["delta"], p["A"], wires["B"], wires["C"], z=wires["z"], dtype="bf16", **kw)
    yf, hf = orc.scan(vals["u"], vals["delta"], p["A"], vals["B"], vals["C"], z=vals["z"], dtype="f32", **kw)
    assert np.array_equal(yb, yf) and np.array_equal(hb, hf)
    # spot values: 1.0, -2.0, 0.15625 (exact in bf16)
    for v in (1.0, -2.0, 0.15625):
        assert from_bits(to_bf16_bits(np.float32(v)).reshape(1))[0] == v


def pin_channel_subset(orc):
    """Computing a list of channels one by one gives the same rows as the full problem."""
    p = rand_problem(19, batch=2, dim=5)
    y, hl = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], delta_bias=p["delta_bias"])
    chans = np.array([7, 0, 9, 3])
    ys, hs = orc.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], delta_bias=p["delta_bias"],
                      chans=chans)
    assert np.array_equal(ys, y[chans]) and np.array_equal(hs, hl[chans])


def pin_degenerate_sizes(orc):
    """L = 0 returns the initial state; N = 0 leaves only the gated skip term D u."""
    p = rand_problem(21, L=6)
    h0 = np.random.default_rng(22).normal(size=(6, 4))
    y, hl = orc.scan(p["u"][:, :, :0], p["delta"][:, :, :0], p["A"], p["B"][:, :, :0], p["C"][:, :, :0],
                     D=p["D"], z=p["z"][:, :, :0], delta_bias=p["delta_bias"], h0=h0)
    assert y.shape == (6, 0) and np.array_equal(hl, h0)
    y, hl = orc.scan(p["u"], p["delta"], f32(np.zeros((3, 0))), f32(np.zeros((2, 0, 6))), f32(np.zeros((2, 0, 6))),
                     D=p["D"], z=p["z"], delta_bias=p["delta_bias"])
    want = (p["D"][None, :, None] * p["u"].astype(np.float64)) * silu64(p["z"])
    assert rel_err(y, want.reshape(6, 6)) < 1e-14 and hl.shape == (6, 0)


# ---------------------------------------------------------------- zero-order hold

def pin_zoh_theorem1(orc):
    """Theorem 1 ("Mamba: Linear-Time Sequence Modeling with Selective State
    Spaces", azimuth.plus): with N = 1, A = -1, B = C = 1 and dt = softplus(g_t),
    the zero-order-hold scan is the gated RNN h_t = (1 - s_t) h_{t-1} + s_t x_t
    with s_t = sigmoid(g_t), exactly (1 - exp(-softplus(g)) = sigmoid(g))."""
    r = np.random.default_rng(41)
    L = 50
    x = f32(r.normal(size=(1, 2, L)))
    g = f32(r.normal(scale=2.0, size=(1, 2, L)))
    one = f32(np.ones((1, 1, L)))
    y, hl = orc.scan(x, g, f32(-np.ones((2, 1))), one, one, softplus=True, zoh=True)
    for d in range(2):
        s = 1.0 / (1.0 + np.exp(-g[0, d].astype(np.float64)))
        h, want = 0.0, []
        for t in range(L):
            h = (1.0 - s[t]) * h + s[t] * float(x[0, d, t])
            want.append(h)
        assert rel_err(y[d], want) < 1e-12, (d, rel_err(y[d], want))
        assert abs(hl[d, 0] - want[-1]) < 1e-12


def pin_zoh_limits(orc):
    """A = 0 exactly: the hold weight is its limit dt, so ZOH and the printed
    (Euler) update agree bitwise; |A dt| ~ 1e-9: they agree to 1e-8 relative.
    Large |A dt|: the weight tends to -1/A, the steady state of the held input."""
    p = rand_problem(42, batch=1, dim=3, N=4, L=16, gate=False, with_D=False)
    A0 = f32(np.zeros((3, 4)))
    ye, he = orc.scan(p["u"], p["delta"], A0, p["B"], p["C"], delta_bias=p["delta_bias"])
    yz, hz = orc.scan(p["u"], p["delta"], A0, p["B"], p["C"], delta_bias=p["delta_bias"], zoh=True)
    assert np.array_equal(ye, yz) and np.array_equal(he, hz)
    At = f32(np.full((3, 4), -1e-9))
    ye, _ = orc.scan(p["u"], p["delta"], At, p["B"], p["C"], delta_bias=p["delta_bias"])
    yz, _ = orc.scan(p["u"], p["delta"], At, p["B"], p["C"], delta_bias=p["delta_bias"], zoh=True)
    assert rel_err(yz, ye) < 1e-8
    # one step with dt = 40, A = -2 from h = 0: h = (exp(-80) - 1)/(-2) * B u ~ B u / 2
    y, h = orc.scan(f32([[[3.0]]]), f32([[[40.0]]]), f32([[-2.0]]), f32([[[5.0]]]), f32([[[1.0]]]),
                    softplus=False, zoh=True)
    assert abs(h[0, 0] - 7.5) < 1e-12 and abs(y[0, 0] - 7.5) < 1e-12


def pin_zoh_lti_convolution(orc):
    """Time-invariant zero-order hold: y_t = sum_k C Abar^k Bbar u_{t-k} with
    Abar = exp(dt A) and Bbar = (exp(dt A) - 1)/A B, as an O(L^2) convolution."""
    r = np.random.default_rng(43)
    dim, N, L = 2, 3, 30
    u = f32(r.normal(size=(1, dim, L)))
    draw = f32(r.normal(size=(1, dim, 1)))
    A = f32(-np.exp(r.uniform(-1.0, 1.0, size=(dim, N))))
    B0 = f32(r.normal(size=(1, N, 1)))
    C0 = f32(r.normal(size=(1, N, 1)))
    y, _ = orc.scan(u, np.repeat(draw, L, axis=2), A, np.repeat(B0, L, axis=2), np.repeat(C0, L, axis=2),
                    softplus=True, zoh=True)
    k = np.arange(L)
    for d in range(dim):
        dt = softplus64(float(draw[0, d, 0]))
        K = np.zeros(L)
        for n in range(N):
            a = float(A[d, n])
            K += float(C0[0, n, 0]) * np.exp(k * dt * a) * (np.expm1(dt * a) / a) * float(B0[0, n, 0])
        want = np.convolve(u[0, d].astype(np.float64), K)[:L]
        assert rel_err(y[d], want) < 1e-11


# ---------------------------------------------------------------- the short convolution

def pin_conv_impulse_response(orc):
    """A unit impulse at t0 returns the taps in causal order: out[t0 + j] = w[3 - j]
    for j = 0..3 and zero everywhere else (no bias, no SiLU)."""
    L, t0 = 12, 5
    x = np.zeros((1, 3, L), dtype=np.float32)
    x[0, :, t0] = 1.0
    w = f32([[1.0, 10.0, 100.0, 1000.0], [-2.0, 0.5, 3.0, -7.0], [4.0, -1.0, 0.25, 2.0]])
    out = orc.conv1d(x, w, silu=False)
    for d in range(3):
        want = np.zeros(L)
        for j in range(4):
            want[t0 + j] = w[d, 3 - j]
        assert np.array_equal(out[0, d], want), (d, out[0, d], want)


def pin_conv_worked_sum(orc):
    """x = 1..5 with taps (1, 10, 100, 1000): each output reads the last four
    inputs as decimal digits, 1000, 2100, 3210, 4321, 5432 (the sum written out)."""
    x = f32([1, 2, 3, 4, 5]).reshape(1, 1, 5)
    out = orc.conv1d(x, f32([[1.0, 10.0, 100.0, 1000.0]]), silu=False)
    assert np.array_equal(out[0, 0], [1000.0, 2100.0, 3210.0, 4321.0, 5432.0]), out


def pin_conv_identity_silu(orc):
    """Taps (0, 0, 0, 1) with a bias pass x + b through: the output is
    silu(x + b) = (x + b) / (1 + exp(-(x + b)))."""
    r = np.random.default_rng(31)
    x = f32(r.normal(size=(2, 3, 20)))
    b = f32(r.normal(size=(3,)))
    w = f32(np.tile([0.0, 0.0, 0.0, 1.0], (3, 1)))
    out = orc.conv1d(x, w, bias=b, silu=True)
    s = x.astype(np.float64) + b[None, :, None].astype(np.float64)
    assert rel_err(out, silu64(s)) < 1e-15


def pin_conv_linear_causal(orc):
    """Without the SiLU the convolution is linear in x, and a change at t0 leaves every
    output before t0 bitwise unchanged."""
    r = np.random.default_rng(32)
    x1 = f32(r.normal(size=(1, 4, 30)))
    x2 = f32(r.normal(size=(1, 4, 30)))
    w = f32(r.normal(size=(4, 4)))
    o1, o2 = orc.conv1d(x1, w, silu=False), orc.conv1d(x2, w, silu=False)
    o12 = orc.conv1d(f32(x1.astype(np.float64) + x2.astype(np.float64)), w, silu=False)
    assert rel_err(o12, o1 + o2) < 1e-6          # x1 + x2 rounded to fp32
    x3 = x1.copy()
    x3[0, :, 17] += 1.0
    o3 = orc.conv1d(x3, w, silu=False)
    assert np.array_equal(o3[:, :, :17], o1[:, :, :17]) and not np.array_equal(o3[:, :, 17:21], o1[:, :, 17:21])


# ---------------------------------------------------------------- backward pass
#
# The gradients are pinned by finite differences of the forward oracle, which
# the pins above fix independently: for every input element x, the fourth-order
# central difference  (8 (L(x+h) - L(x-h)) - (L(x+2h) - L(x-2h))) / (12 h)  of
#     L = sum(dy * y) + sum(dlast * h_last)
# must match the oracle's adjoint.  h = 2^-10 keeps every perturbed fp32 input
# exact (inputs are multiples of 2^-12 below 2^12 in size), so the difference quotient has only
# its O(h^4) truncation error, far below the tolerance.

FD_H = 2.0 ** -10


def _fd_case(seed, softplus=True, zoh=False, gate=True, with_D=True, with_bias=True, h0=True, dlast=True):
    p = rand_problem(seed, batch=2, dim=2, N=3, L=7, gate=gate, with_D=with_D, with_bias=with_bias)
    r = np.random.default_rng(seed + 100)
    if not softplus:                     # dt = raw + bias must stay positive without the softplus
        p["delta"] = f32(np.abs(r.normal(size=p["u"].shape)) * 0.4 + 0.05)
        if with_bias:
            p["delta_bias"] = f32(r.uniform(0.0, 0.2, size=p["delta_bias"].shape))
    for k, v in p.items():               # snap to a 2^-12 grid: x +- h, x +- 2h are then exact in fp32
        if v is not None:
            p[k] = f32(np.round(v.astype(np.float64) * 4096.0) / 4096.0)
    nch = 4
    extra = dict(
        dy=r.normal(size=(2, 2, 7)),
        dlast=r.normal(size=(nch, 3)) if dlast else None,
        h0=r.normal(size=(nch, 3)) if h0 else None,
    )
    return p, extra, softplus, zoh


def _fd_loss(orc, p, extra, softplus, zoh):
    y, hl = orc.scan(**p, softplus=softplus, h0=extra["h0"], zoh=zoh)
    out = float(np.sum(extra["dy"].reshape(y.shape) * y))
    if extra["dlast"] is not None:
        out += float(np.sum(extra["dlast"] * hl))
    return out


def _fd_check(orc, case, tol=1e-9):
    p, extra, softplus, zoh = case
    g = orc.scan_bwd(**p, softplus=softplus, dy=extra["dy"], dlast=extra["dlast"], h0=extra["h0"], zoh=zoh)
    names = {"u": "du", "delta": "ddelta", "z": "dz", "B": "dB", "C": "dC", "A": "dA", "D": "dD",
             "delta_bias": "ddelta_bias"}
    checked = 0
    for key, gkey in list(names.items()) + [("h0", "dh0")]:
        src = extra if key == "h0" else p
        if src[key] is None:
            continue
        base = src[key]
        adj = np.asarray(g[gkey], dtype=np.float64).reshape(base.shape)
        fd = np.zeros(base.shape)
        for idx in np.ndindex(base.shape):
            vals = []
            for k in (1, -1, 2, -2):
                pert = base.copy()
                pert[idx] = pert[idx] + k * FD_H
                assert float(pert[idx]) - float(base[idx]) == k * FD_H     # exact perturbation
                if key == "h0":
                    e2 = dict(extra, h0=pert)
                    vals.append(_fd_loss(orc, p, e2, softplus, zoh))
                else:
                    vals.append(_fd_loss(orc, dict(p, **{key: pert}), extra, softplus, zoh))
            fd[idx] = (8.0 * (vals[0] - vals[1]) - (vals[2] - vals[3])) / (12.0 * FD_H)
        scale = max(1.0, float(np.max(np.abs(fd))))
        err = float(np.max(np.abs(adj - fd)))
        assert err <= tol * scale, f"d{key}: adjoint vs finite difference {err:.3e} (scale {scale:.3e})"
        checked += 1
    return checked


def pin_bwd_finite_difference(orc):
    """Every gradient of the full model (softplus step, bias, D, gate, h0, dlast)."""
    assert _fd_check(orc, _fd_case(11)) == 9


def pin_bwd_finite_difference_plain(orc):
    """Softplus off, no bias, no D, no gate, zero initial state: the bare recurrence."""
    assert _fd_check(orc, _fd_case(12, softplus=False, gate=False, with_D=False, with_bias=False, h0=False)) == 5


def pin_bwd_finite_difference_zoh(orc):
    """Zero-order-hold input weight: its derivatives in dt and A enter ddelta and dA."""
    assert _fd_check(orc, _fd_case(13, zoh=True)) == 9


def pin_bwd_finite_difference_zoh_small_A(orc):
    """Zero-order hold where dt*A is tiny or zero (A = 0 and A = -2^-12): the
    series form of the hold weight's A-derivative, including its A -> 0 limit dt^2/2."""
    case = _fd_case(16, zoh=True)
    case[0]["A"][:, 0] = 0.0
    case[0]["A"][:, 1] = -(2.0 ** -12)
    assert _fd_check(orc, case) == 9


def pin_bwd_zero_cotangent(orc):
    """Zero cotangents give exactly zero gradients (the map is linear in (dy, dlast))."""
    p, extra, softplus, zoh = _fd_case(14)
    g = orc.scan_bwd(**p, dy=np.zeros_like(extra["dy"]), dlast=None, h0=extra["h0"])
    for k in ("du", "ddelta", "dz", "dB", "dC", "dA", "dD", "ddelta_bias", "dh0"):
        assert np.all(g[k] == 0.0), k


def pin_bwd_channel_subset(orc):
    """Per-channel outputs for a subset of channels equal those of the full call."""
    p, extra, softplus, zoh = _fd_case(15)
    full = orc.scan_bwd(**p, dy=extra["dy"], dlast=extra["dlast"], h0=extra["h0"])
    chans = np.array([3, 0])
    sub = orc.scan_bwd(**p, dy=extra["dy"].reshape(4, 7)[chans], dlast=extra["dlast"][chans],
                       h0=extra["h0"][chans], chans=chans, want_BC=False)
    assert np.array_equal(sub["du"], full["du"].reshape(4, 7)[chans])
    assert np.array_equal(sub["dh0"], full["dh0"][chans])
    dA = sub["dA_part"]
    assert np.allclose(full["dA"][1], dA[0] + orc.scan_bwd(**p, dy=extra["dy"].reshape(4, 7)[[1]],
                                                            dlast=extra["dlast"][[1]], h0=extra["h0"][[1]],
                                                            chans=[1], want_BC=False)["dA_part"][0],
                       rtol=1e-14, atol=1e-14)


PINS = [pin_tiny_example, pin_selective_toy, pin_lti_convolution, pin_unrolled_sum, pin_zero_step_keeps_state,
        pin_large_step_resets, pin_recurrence_equals_scan, pin_linear_and_causal, pin_gated_rnn_decay,
        pin_inverse_softplus_bias, pin_bf16_widening, pin_channel_subset, pin_degenerate_sizes,
        pin_conv_impulse_response, pin_conv_worked_sum, pin_conv_identity_silu, pin_conv_linear_causal,
        pin_zoh_theorem1, pin_zoh_limits, pin_zoh_lti_convolution,
        pin_bwd_finite_difference, pin_bwd_finite_difference_plain, pin_bwd_finite_difference_zoh,
        pin_bwd_finite_difference_zoh_small_A, pin_bwd_zero_cotangent, pin_bwd_channel_subset]
