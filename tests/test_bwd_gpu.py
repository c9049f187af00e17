"""GPU parity of the backward pass (ss_scan_bwd) against the fp64 oracle's
adjoint, which the finite-difference pins fix.

Every gradient is compared element by element:
    |g - g_ref| <= TOL_GRAD * max(|g_ref|, rms(g_ref))
for fp32 and bf16 inputs alike (both sides read the same bf16 bytes; the
arithmetic is fp32 on the GPU).  TOL_GRAD = 1e-4, the bound of the fp32
forward scan: the adjoint and the recomputed states chain decays that are each
a MUFU.EX2 with ~2^-22 relative error, and dA, dD, ddelta_bias, dB, dC are fp32
sums of up to L or dim terms.  The errors measured on B300 stay below 4e-6.

At the long-sequence size (batch 1, dim 5120, N 16, L 65536, bf16) the oracle
computes every channel, in blocks of 512, and every gradient is compared; dB,
dC and du are also checked by Euler's identity for functions homogeneous of
degree one: y and h_last are linear in B, in C and in u (with h0 = 0), so
    sum dB B = sum dC C = sum dy (y - D u silu(z)) + sum dlast h_last   (dC: without dlast)
    sum du u = sum dy y + sum dlast h_last.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import StreamCheck, host, log_result, rms
from fullsize import wire_problem

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_GRAD = 1e-4
NAMES = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


def grad_err(g, ref):
    g = np.asarray(g, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g))
    if ref.size == 0:
        return 0.0
    scale = np.maximum(np.abs(ref), max(rms(ref), 1e-30))
    return float(np.max(np.abs(g - ref) / scale))


def make(seed, batch, dim, N, L, dtype, gate=True, with_D=True, with_bias=True, h0=True, dlast=True, softplus=True,
         zoh=False):
    p = I.selective_problem("bwd", seed=seed, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=dtype, bc_std=0.5,
                            d_mode="normal", gate=gate, device=DEV, gen_device="cpu")
    p.extra["zoh"] = zoh
    if zoh:   # decay rates from -0.01 to -50: both branches of the hold weight and of its A-derivative
        n = torch.arange(N, dtype=torch.float32)
        row = -0.01 * torch.exp(n * (math.log(5000.0) / max(N - 1, 1)))
        p.A = row.unsqueeze(0).expand(dim, N).contiguous().to(DEV)
    if not with_D:
        p.D = None
    if not with_bias:
        p.delta_bias = None
    if not softplus:     # dt = raw (+ bias) is then used as is: keep it positive
        g = torch.Generator().manual_seed(seed + 7)
        p.delta = (torch.rand((batch, dim, L), generator=g) * 0.2 + 0.005).to(dtype).to(DEV)
        if with_bias:
            p.delta_bias = torch.full((dim,), 0.01, device=DEV)
        p.softplus = False
    ct = I.cotangents(seed=seed + 1000, batch=batch, dim=dim, dstate=N, seqlen=L, with_dlast=dlast, with_h0=h0,
                      device=DEV, gen_device="cpu")
    return p, ct


def gpu_grads(p, ct):
    return ss.scan_bwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus,
                       dy=ct.dy, dlast=ct.dlast, h0=ct.h0, want_dh0=True, zoh=p.extra.get("zoh", False))


def oracle_grads(p, ct, chans=None):
    w = I.to_wire
    nb, nd, N = p.batch, p.dim, p.dstate
    dy, dl, h0 = host(ct.dy).reshape(nb * nd, -1), ct.dlast, ct.h0
    dl = None if dl is None else host(dl).reshape(nb * nd, N)
    h0 = None if h0 is None else host(h0).reshape(nb * nd, N)
    if chans is not None:
        dy = dy[chans]
        dl = None if dl is None else dl[chans]
        h0 = None if h0 is None else h0[chans]
    return oracle.scan_bwd(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z),
                           delta_bias=w(p.delta_bias), softplus=p.softplus,
                           dtype="bf16" if p.in_dtype == I.BF16 else "f32", dy=dy, dlast=dl, h0=h0,
                           chans=chans, want_BC=chans is None, zoh=p.extra.get("zoh", False))


def compare_all(g, r, p):
    """Every gradient; dD, ddelta_bias and dh0 are the gradients at 0 where D, delta_bias or h0 are absent,
    on both sides."""
    errs = {}
    for k in NAMES:
        got = g[k]
        want = r[k]
        if k == "dz" and p.z is None:
            assert got is None and want is None
            continue
        errs[k] = grad_err(host(got), np.asarray(want).reshape(tuple(got.shape)))
        assert errs[k] <= TOL_GRAD, f"{k}: error {errs[k]:.3e} > {TOL_GRAD}"
    return errs


CASES = [
    # seed, batch, dim, N, L, dtype, options
    (1, 2, 70, 16, 200, torch.float32, {}),                                   # 3 channel tiles, ragged last chunk
    (2, 1, 64, 16, 2048, torch.bfloat16, {}),                                 # 32 chunks
    (3, 2, 33, 13, 77, torch.float32, {}),                                    # padded states, L % 8 != 0 (no vectors)
    (4, 1, 40, 4, 130, torch.bfloat16, dict(gate=False, with_D=False)),
    (5, 1, 20, 8, 64, torch.float32, dict(h0=False, dlast=False)),            # exactly one chunk
    (6, 1, 24, 32, 96, torch.bfloat16, {}),
    (7, 1, 10, 64, 72, torch.float32, dict(with_bias=False)),
    (8, 2, 17, 16, 1, torch.float32, {}),                                     # one step
    (9, 1, 30, 16, 150, torch.float32, dict(softplus=False)),
    (10, 3, 100, 16, 520, torch.bfloat16, dict(h0=False)),
    # 16 chunks in two groups of the local passes' blocks, the last chunk 40 steps (two and a
    # half tiles), a partial last channel tile, padded states
    (11, 2, 130, 12, 1000, torch.bfloat16, {}),
    (12, 1, 200, 16, 1000, torch.float32, dict(with_bias=False)),
    # the narrowest state width through the TMA local passes (one lane per channel in the
    # main pass, N padded from 3 to 4)
    (13, 2, 50, 3, 136, torch.bfloat16, {}),
    # zero-order-hold input weight
    (20, 2, 70, 16, 200, torch.float32, dict(zoh=True)),
    (21, 1, 64, 16, 2048, torch.bfloat16, dict(zoh=True)),
    (22, 2, 33, 13, 77, torch.float32, dict(zoh=True, with_D=False)),
    (23, 1, 24, 64, 96, torch.bfloat16, dict(zoh=True, h0=False)),
    (24, 1, 30, 16, 150, torch.float32, dict(zoh=True, softplus=False)),
    (26, 2, 130, 12, 1000, torch.bfloat16, dict(zoh=True)),
    (27, 1, 70, 4, 200, torch.float32, dict(zoh=True)),
    # the medium fp32 configuration's shape
    (25, 2, 256, 16, 2048, torch.float32, {}),
]


@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}b{c[1]}d{c[2]}n{c[3]}L{c[4]}{'zoh' if c[6].get('zoh') else ''}"
                                              for c in CASES])
def test_bwd_matches_oracle(case):
    seed, batch, dim, N, L, dtype, opt = case
    p, ct = make(seed, batch, dim, N, L, dtype, **opt)
    g = gpu_grads(p, ct)
    torch.cuda.synchronize()
    r = oracle_grads(p.to("cpu"), ct)
    compare_all(g, r, p)
    assert ss.device_status() == ss.SS_OK


def test_bwd_zero_cotangent_gives_zero():
    p, ct = make(11, 1, 40, 16, 128, torch.float32)
    ct.dy.zero_()
    ct.dlast.zero_()
    g = gpu_grads(p, ct)
    for k in NAMES:
        assert torch.count_nonzero(g[k]).item() == 0, k


def test_bwd_length_zero():
    p, ct = make(12, 2, 8, 16, 0, torch.float32)
    g = gpu_grads(p, ct)
    assert torch.equal(g["dh0"], ct.dlast)
    assert torch.count_nonzero(g["dA"]).item() == 0


def test_bwd_repeated_calls_agree():
    """Only the atomically accumulated sums may differ between runs, and only in the last bits."""
    p, ct = make(13, 1, 96, 16, 512, torch.bfloat16)
    g1, g2 = gpu_grads(p, ct), gpu_grads(p, ct)
    for k in ("du", "ddelta", "dz", "dh0"):
        assert torch.equal(g1[k], g2[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        assert grad_err(host(g1[k]), host(g2[k])) <= 1e-5, k


def full_size_grads_vs_oracle(p, ct, label):
    """Every gradient of a batch-1 problem against the oracle's adjoint, the oracle running over
    blocks of 512 channels: du, ddelta, dz element by element (streamed), dA, dD, ddelta_bias per
    channel, and dB, dC as the sums of every block's share.  Returns the GPU gradients."""
    assert p.batch == 1
    g = gpu_grads(p, ct)
    torch.cuda.synchronize()
    wp = wire_problem(p)
    N, L = p.dstate, p.seqlen
    dy = host(ct.dy).reshape(p.dim, L)
    dl = host(ct.dlast).reshape(p.dim, N)
    zoh = p.extra.get("zoh", False)
    chk = {k: StreamCheck(f"{label} {k}", False, tol=TOL_GRAD) for k in ("du", "ddelta", "dz")}
    dB = np.zeros((1, N, L))
    dC = np.zeros((1, N, L))
    dA = np.zeros((p.dim, N))
    dD = np.zeros(p.dim)
    db = np.zeros(p.dim)
    for d0 in range(0, p.dim, 512):
        d1 = min(p.dim, d0 + 512)
        chans = np.arange(d0, d1, dtype=np.int64)
        r = oracle.scan_bwd(wp["u"], wp["delta"], wp["A"], wp["B"], wp["C"], D=wp["D"], z=wp["z"],
                            delta_bias=wp["delta_bias"], softplus=p.softplus, dtype=wp["dtype"], dy=dy[d0:d1],
                            dlast=dl[d0:d1], chans=chans, want_BC=True, zoh=zoh)
        for k in chk:
            chk[k].add(host(g[k][0, d0:d1]), r[k])
        dB += r["dB"]
        dC += r["dC"]
        dA[d0:d1], dD[d0:d1], db[d0:d1] = r["dA_part"], r["dD_part"], r["dbias_part"]
    for k in chk:
        chk[k].finish()
    for k, ref in (("dA", dA), ("dD", dD), ("ddelta_bias", db), ("dB", dB), ("dC", dC)):
        e = grad_err(host(g[k]).reshape(ref.shape), ref)
        log_result(f"{label} {k}", n=int(ref.size), judged=e, rule="max err/max(|ref|,rms)", tol=TOL_GRAD)
        assert e <= TOL_GRAD, f"{label} {k}: {e:.3e}"
    return g


def test_bwd_long_sequence_full_and_identities():
    """Batch 1, dim 5120, N 16, L 65536 (bf16, gate): the size and call the benchmark times.
    Every gradient against the oracle (all channels), then Euler's identity for dB, dC and du."""
    p = I.workload("mamba2p8b_long_bf16", device=DEV, gen_device="cuda")
    ct = I.cotangents(seed=103, batch=1, dim=p.dim, dstate=p.dstate, seqlen=p.seqlen, with_h0=False, device=DEV,
                      gen_device="cuda")
    g = full_size_grads_vs_oracle(p, ct, "bwd mamba2p8b_long")
    y, hl = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, chunk_len=2048,
                            return_last_state=True)
    torch.cuda.synchronize()
    # Euler's identity for dB, dC, du over every channel (float64 sums on the GPU)
    f = lambda t: t.double()
    ds_u = f(p.D)[None, :, None] * f(p.u) * torch.nn.functional.silu(f(p.z))
    lin_y = (f(ct.dy) * (f(y) - ds_u)).sum()
    lin_last = (f(ct.dlast) * f(hl)).sum()
    checks = {
        "dB": ((f(g["dB"]) * f(p.B)).sum(), lin_y + lin_last, (f(g["dB"]) * f(p.B)).abs().sum()),
        "dC": ((f(g["dC"]) * f(p.C)).sum(), lin_y, (f(g["dC"]) * f(p.C)).abs().sum()),
        "du": ((f(g["du"]) * f(p.u)).sum(), (f(ct.dy) * f(y)).sum() + lin_last, (f(g["du"]) * f(p.u)).abs().sum()),
    }
    for k, (lhs, rhs, scale) in checks.items():
        rel = abs(float(lhs - rhs)) / float(scale)
        assert rel <= 1e-4, f"{k}: Euler identity off by {rel:.3e} of sum |terms|"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_bwd_unaligned_pointers(dtype):
    """Every array one element past a 16-byte boundary (L a multiple of 8): the kernels take
    their element-by-element paths and scalar atomics; the gradients are the same."""
    p, ct = make(31, 2, 40, 16, 136, dtype)
    shift = lambda t: None if t is None else _offset_copy(t)
    q = I.Problem(p.name, shift(p.u), shift(p.delta), shift(p.A), shift(p.B), shift(p.C), shift(p.D), shift(p.z),
                  shift(p.delta_bias), p.softplus, 0, dict(p.extra))
    cq = I.Cotangents(shift(ct.dy), shift(ct.dlast), shift(ct.h0))
    for t in (q.u, q.B, cq.dy):
        assert t.data_ptr() % 16 != 0
    g = gpu_grads(q, cq)
    torch.cuda.synchronize()
    r = oracle_grads(p.to("cpu"), ct)
    compare_all(g, r, p)


def _offset_copy(t):
    """A copy of t whose storage starts one element past a 16-byte aligned address."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    out = buf[1:].view(t.shape)
    out.copy_(t)
    return out


def test_bwd_long_sequence_zoh_full():
    """The zero-order-hold backward pass at batch 1, dim 5120, N 16, L 65536 (bf16, gate):
    every gradient against the oracle (all channels)."""
    p = I.workload("mamba2p8b_long_bf16", device=DEV, gen_device="cuda")
    p.extra["zoh"] = True
    ct = I.cotangents(seed=104, batch=1, dim=p.dim, dstate=p.dstate, seqlen=p.seqlen, with_h0=False, device=DEV,
                      gen_device="cuda")
    full_size_grads_vs_oracle(p, ct, "zoh bwd mamba2p8b_long")


@pytest.mark.parametrize("chunk", [None, 64], ids=["fwd", "chunked64"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_selective_scan_autograd(chunk, dtype):
    """ss.selective_scan through torch.autograd, from an initial state h0: the leaves' .grad (h0's
    included) of sum(dy y) + sum(dlast h_last) against the oracle's adjoint.  Gradients of bf16 inputs come back rounded to bf16, so they are
    held to twice bf16's rounding bound, 2^-8 of max(|ref|, rms(ref)); fp32 ones to TOL_GRAD."""
    p, ct = make(501, 2, 40, 16, 136, dtype, h0=True)
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
    leaf = {k: getattr(p, k).detach().clone().requires_grad_(True) for k in names}
    leaf["h0"] = ct.h0.detach().clone().requires_grad_(True)
    y, h = ss.selective_scan(*(leaf[k] for k in names), softplus=p.softplus, h0=leaf["h0"], chunk_len=chunk)
    ((y * ct.dy).sum() + (h * ct.dlast).sum()).backward()
    r = oracle_grads(p, ct)
    for k, key in zip(names + ("h0",), ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dh0")):
        got = leaf[k].grad
        assert got is not None and got.dtype == leaf[k].dtype, k
        tol = 2.0 ** -8 if got.dtype == torch.bfloat16 else TOL_GRAD
        e = grad_err(host(got.float()), np.asarray(r[key]).reshape(tuple(got.shape)))
        assert e <= tol, f"{k}: error {e:.3e} > {tol}"
