"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Every case draws seeded inputs from selective_state_space_117_b300.inputs,
runs the library on the GPU, runs the oracle on the host on the same bytes,
and compares element by element under the tolerances of tests/parity.py.
Large workloads run at full size on the GPU in the launch configuration the
benchmark times; the oracle then computes every channel, block by block
(tests/fullsize.py), and every output element is compared.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import StreamCheck, check, host
from fullsize import compare_scans
from pins import read_golden

pytestmark = pytest.mark.gpu
DEV = "cuda"


# ------------------------------------------------------------------ helpers

def oracle_scan(p: I.Problem, h0=None):
    w = I.to_wire
    return oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z), delta_bias=w(p.delta_bias),
                       softplus=p.softplus, dtype="bf16" if p.in_dtype == I.BF16 else "f32", h0=h0)


def run(p: I.Problem, impl: str, chunk_len=None):
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus, return_last_state=True)
    if impl == "fwd":
        return ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, **kw)
    if impl in ("fwd_thread", "fwd_warp"):
        return ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, schedule=impl[4:], **kw)
    return ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, chunk_len=chunk_len, **kw)


def compare(p: I.Problem, y, hl, what):
    bf = p.in_dtype == I.BF16
    yr, hr = oracle_scan(p.to("cpu"))
    B, Dm, L = p.u.shape
    N = p.A.shape[1]
    ey = check(host(y).reshape(B * Dm, L), yr, bf, what + " y")
    eh = check(host(hl).reshape(B * Dm, N), hr, bf, what + " last_state")
    return ey, eh


def custom(seed, batch, dim, N, L, dtype=torch.float32, gate=True, with_D=True, with_bias=True, softplus=True):
    p = I.selective_problem("custom", seed=seed, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=dtype, bc_std=0.5,
                            d_mode="normal", gate=gate, device=DEV, gen_device="cpu")
    # vary A across channels as well as states
    g = torch.Generator().manual_seed(seed + 1000)
    p.A = (-torch.exp(torch.rand((dim, N), generator=g) * 2.5 - 1.0)).to(DEV)
    if not with_D:
        p.D = None
    if not with_bias:
        p.delta_bias = None
    p.softplus = softplus
    if not softplus:   # raw step sizes must stay small and positive without the softplus
        p.delta = (torch.rand(p.u.shape, generator=g) * 0.2).to(dtype).to(DEV)
        p.delta_bias = None
    return p


# ------------------------------------------------------------ worked examples

@pytest.mark.parametrize("impl", ["fwd", "chunked3", "decode"])
def test_worked_examples(impl):
    g = read_golden("tiny_example.txt")
    sig = torch.tensor(g["signal"], dtype=torch.float32, device=DEV).view(1, 1, -1)
    L = sig.shape[-1]
    one = torch.ones((1, 1, L), device=DEV)
    for key in ("a=0.9", "a=0.3"):
        A = torch.tensor([[math.log(float(key.split("=")[1]))]], device=DEV)
        if impl == "decode":
            st = torch.zeros((1, 1, 1), device=DEV)
            ys = [ss.state_update(st, sig[:, :, t].contiguous(), one[:, :, t].contiguous(), A, one[:, 0, t:t + 1].contiguous(),
                                  one[:, 0, t:t + 1].contiguous(), softplus=False)[0, 0].item() for t in range(L)]
        elif impl == "fwd":
            ys = host(ss.scan_fwd(sig, one, A, one, one, softplus=False))[0, 0]
        else:
            ys = host(ss.scan_chunked(sig, one, A, one, one, softplus=False, chunk_len=3))[0, 0]
        assert np.max(np.abs(np.asarray(ys) - np.asarray(g[key]))) <= g["tolerance"][0], (key, ys)
    t = read_golden("selective_toy.txt")
    vals = torch.tensor(t["values"], device=DEV).view(1, 1, -1)
    imp = torch.tensor(t["important"], device=DEV).view(1, 1, -1) > 0
    lo = math.log(0.95) / math.log(0.2)
    dt = torch.where(imp, torch.tensor(1.0, device=DEV), torch.tensor(lo, device=DEV)).float()
    Bv = torch.where(imp, torch.tensor(1.0, device=DEV), torch.tensor(0.05 / lo, device=DEV)).float()
    A = torch.tensor([[math.log(0.2)]], device=DEV)
    one4 = torch.ones_like(vals)
    if impl == "chunked3":
        y = ss.scan_chunked(vals, dt, A, Bv, one4, softplus=False, chunk_len=3)
    else:
        y = ss.scan_fwd(vals, dt, A, Bv, one4, softplus=False)
    assert np.max(np.abs(host(y)[0, 0] - np.asarray(t["outputs"]))) <= t["tolerance"][0]


# ------------------------------------------------------------ the workloads

@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("fwd_thread", None), ("fwd_warp", None), ("chunked", 1),
                                        ("chunked", 7), ("chunked", 16), ("chunked", 64)])
def test_tiny_fp32(impl, chunk):
    p = I.workload("tiny_fp32", device=DEV, gen_device="cpu")
    y, hl = run(p, impl, chunk)
    compare(p, y, hl, f"tiny_fp32/{impl}{chunk or ''}")


@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("fwd_thread", None), ("fwd_warp", None), ("chunked", 2048),
                                        ("chunked", 256), ("chunked", 100)])
def test_medium_fp32_gate(impl, chunk):
    p = I.workload("medium_fp32_gate", device=DEV, gen_device="cpu")
    y, hl = run(p, impl, chunk)
    compare(p, y, hl, f"medium_fp32_gate/{impl}{chunk or ''}")


def test_medium_lti_closed_form():
    """Time-invariant variant: library vs oracle, and library vs the convolution closed form
    y_t = silu(z_t) * (sum_k K_k u_{t-k} + D u_t),  K_k = sum_n C_n exp(k dt A_n) dt B_n."""
    p = I.lti_problem(device=DEV, gen_device="cpu")
    y, hl = run(p, "fwd")
    compare(p, y, hl, "medium_lti/fwd")
    yc, _ = run(p, "chunked", 256)
    compare(p, yc, hl, "medium_lti/chunked256")
    pc = p.to("cpu")
    Bn, Dm, L = pc.u.shape
    yh = host(y)
    k = np.arange(L, dtype=np.float64)
    worst = 0.0
    for b in range(Bn):
        for d in range(0, Dm, 8):
            x = float(pc.delta[b, d, 0]) + float(pc.delta_bias[d])
            dt = math.log1p(math.exp(-abs(x))) + max(x, 0.0)
            K = np.zeros(L)
            for n in range(pc.A.shape[1]):
                K += float(pc.C[b, n, 0]) * np.exp(k * dt * float(pc.A[d, n])) * dt * float(pc.B[b, n, 0])
            u = pc.u[b, d].double().numpy()
            z = pc.z[b, d].double().numpy()
            want = (np.convolve(u, K)[:L] + float(pc.D[d]) * u) * (z / (1.0 + np.exp(-z)))
            from parity import err_f32
            worst = max(worst, err_f32(yh[b, d], want))
    assert worst <= 1e-4, worst


@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("fwd_warp", None), ("chunked", 512), ("chunked", 2048)])
def test_mamba130m_layer_bf16(impl, chunk):
    """The Mamba-130M-shaped layer (8 x 1536 x 16 x 2048, bf16): every element of y and every
    final state against the oracle."""
    p = I.workload("mamba130m_layer_bf16", device=DEV, gen_device="cuda")
    y, hl = run(p, impl, chunk)
    compare_scans(p, {f"{impl}{chunk or ''}": (y, hl)}, "mamba130m")


def test_mamba2p8b_long_bf16():
    """The Mamba-2.8B-shaped long sequence (1 x 5120 x 16 x 65536, bf16) through the chunked
    scan at chunk 2048 (the launch configuration the benchmark times) and through ss_scan_fwd
    under its default and thread schedules: every element of y (335.5 M per run) and every
    final state against the oracle, which computes each channel block once for all runs."""
    p = I.workload("mamba2p8b_long_bf16", device=DEV, gen_device="cuda")
    outs = {name: run(p, impl, chunk) for name, impl, chunk in
            (("chunked2048", "chunked", 2048), ("fwd", "fwd", None), ("fwd_thread", "fwd_thread", None))}
    torch.cuda.synchronize()
    compare_scans(p, outs, "mamba2p8b_long")
    del outs, p
    torch.cuda.empty_cache()


def test_decode_stream_256x5120():
    """1024 sequential decode steps on a (256, 5120, 16) fp32 state: every step's y over all
    256 x 5120 channels and the whole final state against the oracle's recurrence, which
    advances its own fp64 state through the same 1024 steps."""
    cfg = I.DECODE
    st_in = I.decode_stream(seed=cfg["seed"], batch=cfg["batch"], dim=cfg["dim"], dstate=cfg["dstate"],
                            steps=cfg["steps"], device=DEV, gen_device="cuda")
    nb, nd, N = cfg["batch"], cfg["dim"], cfg["dstate"]
    state = torch.zeros((nb, nd, N), device=DEV)
    y = torch.empty((nb, nd), device=DEV)
    w = I.to_wire
    A, Dv, bias = w(st_in.A), w(st_in.D), w(st_in.delta_bias)
    sref = np.zeros((nb * nd, N))
    cy = StreamCheck("decode_256x5120 y (all steps, all channels)", True)
    for t in range(cfg["steps"]):
        ss.state_update(state, st_in.u[t], st_in.delta[t], st_in.A, st_in.B[t], st_in.C[t], D=st_in.D, z=st_in.z[t],
                        delta_bias=st_in.delta_bias, y=y)
        yg = host(y).reshape(-1)
        yr = oracle.state_update(sref, w(st_in.u[t]), w(st_in.delta[t]), A, w(st_in.B[t]), w(st_in.C[t]), D=Dv,
                                 z=w(st_in.z[t]), delta_bias=bias, dtype="bf16")
        cy.add(yg, yr)
    cy.finish()
    check(host(state).reshape(nb * nd, N), sref, True, "decode_256x5120 final state (all channels)")
    del st_in, state
    torch.cuda.empty_cache()


# ------------------------------------------------------------ edge cases

RAGGED = [
    # seed, batch, dim, N, L, dtype, gate, with_D, with_bias, softplus
    (21, 1, 130, 1, 63, torch.float32, True, True, True, True),
    (22, 3, 33, 5, 100, torch.float32, False, True, False, True),
    (23, 2, 17, 17, 1, torch.float32, True, False, True, True),
    (24, 1, 257, 33, 77, torch.bfloat16, True, True, True, True),
    (25, 2, 5, 64, 40, torch.float32, True, True, True, False),
    (26, 1, 9, 3, 1000, torch.bfloat16, False, False, True, True),
    (27, 2, 129, 16, 333, torch.bfloat16, True, True, True, True),
    (28, 1, 64, 8, 257, torch.float32, True, True, True, True),
]


@pytest.mark.parametrize("case", RAGGED, ids=[f"b{c[1]}d{c[2]}n{c[3]}L{c[4]}{'bf' if c[5] == torch.bfloat16 else 'f'}"
                                              for c in RAGGED])
@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("chunked", 7), ("chunked", 32)])
def test_ragged(case, impl, chunk):
    seed, batch, dim, N, L, dt, gate, wd, wb, sp = case
    p = custom(seed, batch, dim, N, L, dt, gate, wd, wb, sp)
    y, hl = run(p, impl, chunk)
    compare(p, y, hl, f"ragged/{impl}{chunk or ''}")


# Shapes for the TMA paths (L a multiple of 8, chunk a multiple of 16): partial
# last tiles (L = 16 k + 8), channel tiles cut short (dim % 64 != 0), several
# batch rows, every padded state width, and both input dtypes.
TMA_SHAPES = [
    # seed, batch, dim, N, L, dtype, chunk
    (41, 3, 100, 16, 328, torch.bfloat16, 64),
    (42, 2, 70, 16, 200, torch.float32, 48),
    (43, 1, 64, 64, 96, torch.bfloat16, 32),
    (44, 2, 200, 32, 136, torch.bfloat16, 16),
    (45, 1, 33, 8, 1032, torch.float32, 512),
    (46, 4, 128, 4, 72, torch.bfloat16, 16),
]


@pytest.mark.parametrize("case", TMA_SHAPES, ids=[f"b{c[1]}d{c[2]}n{c[3]}L{c[4]}c{c[6]}" for c in TMA_SHAPES])
@pytest.mark.parametrize("impl", ["fwd", "fwd_thread", "chunked"])
def test_tma_shapes(case, impl):
    seed, batch, dim, N, L, dt, chunk = case
    p = custom(seed, batch, dim, N, L, dt)
    y, hl = run(p, impl, chunk)
    compare(p, y, hl, f"tma/{impl}")


# Shapes for the one-warp-per-channel schedule (512-step segments, 16 steps per lane):
# L = 8 (one lane busy), a last segment holding 8 steps, empty lanes in the last
# segment, exact segment multiples, odd and small N, channel counts that leave the
# last 12-warp block part-empty, and each optional input off.
WARP_SHAPES = [
    # seed, batch, dim, N, L, dtype, gate, with_D, with_bias, softplus
    (61, 1, 5, 1, 8, torch.float32, True, True, True, True),
    (62, 2, 13, 3, 24, torch.bfloat16, True, True, True, True),
    (63, 1, 25, 16, 520, torch.float32, True, True, True, True),
    (64, 3, 12, 8, 1536, torch.bfloat16, False, False, False, True),
    (65, 1, 7, 16, 1032, torch.bfloat16, True, True, True, False),
    (66, 2, 40, 5, 2000, torch.float32, True, False, True, True),
    (67, 1, 3, 16, 4104, torch.bfloat16, True, True, True, True),
]


@pytest.mark.parametrize("case", WARP_SHAPES, ids=[f"b{c[1]}d{c[2]}n{c[3]}L{c[4]}{'bf' if c[5] == torch.bfloat16 else 'f'}"
                                                   for c in WARP_SHAPES])
def test_warp_schedule_shapes(case):
    seed, batch, dim, N, L, dt, gate, wd, wb, sp = case
    p = custom(seed, batch, dim, N, L, dt, gate, wd, wb, sp)
    y, hl = run(p, "fwd_warp")
    compare(p, y, hl, "warp")


def _random_warp_cases(n=12, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        cases.append((300 + i, int(rng.integers(1, 4)), int(rng.integers(1, 41)), int(rng.integers(1, 17)),
                      8 * int(rng.integers(1, 201)), torch.bfloat16 if rng.random() < 0.5 else torch.float32,
                      bool(rng.random() < 0.7), bool(rng.random() < 0.7), bool(rng.random() < 0.7),
                      bool(rng.random() < 0.8)))
    return cases


@pytest.mark.parametrize("case", _random_warp_cases(), ids=lambda c: f"s{c[0]}b{c[1]}d{c[2]}n{c[3]}L{c[4]}")
def test_warp_schedule_random_shapes(case):
    """Seeded random shapes (batch 1-3, D 1-40, N 1-16, L a multiple of 8 up to 1600, either
    dtype, each optional input on or off) under the warp schedule, with and without h0."""
    seed, batch, dim, N, L, dt, gate, wd, wb, sp = case
    p = custom(seed, batch, dim, N, L, dt, gate, wd, wb, sp)
    y, hl = run(p, "fwd_warp")
    compare(p, y, hl, "warp/random")
    g = torch.Generator().manual_seed(seed + 7)
    h0 = torch.randn((batch, dim, N), generator=g)
    y, hl = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus,
                        return_last_state=True, h0=h0.to(DEV), schedule="warp")
    yr, hr = oracle_scan(p.to("cpu"), h0=h0.double().numpy().reshape(batch * dim, N))
    bf = dt == torch.bfloat16
    check(host(y).reshape(batch * dim, L), yr, bf, "warp/random h0 y")
    check(host(hl).reshape(batch * dim, N), hr, bf, "warp/random h0 last_state")


def test_warp_schedule_refuses_unaligned_rows():
    p = custom(68, 1, 4, 16, 64, torch.bfloat16)
    u = torch.empty(p.u.numel() + 1, dtype=p.u.dtype, device=DEV)[1:].view_as(p.u)
    u.copy_(p.u)
    with pytest.raises(ss.SSError) as ei:
        ss.scan_fwd(u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, schedule="warp")
    assert ei.value.status == ss.SS_EINVAL
    # without the flag the library runs the thread schedule on the same arrays
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True)
    y, hl = ss.scan_fwd(u, p.delta, p.A, p.B, p.C, **kw)
    compare(p, y, hl, "unaligned u, default schedule")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_local_pass_wide_decay_spread(dtype):
    """A spread of decay rates (A from -0.05 to -40) and of step sizes across
    channels: going back from a chunk's end, the fast states' weights underflow long
    before the slow ones' (the early stop of the local pass then depends on the
    slowest channel of each block).  The result must still match the oracle."""
    p = custom(47, 2, 192, 16, 4096, dtype)
    n = torch.arange(16, dtype=torch.float32)
    p.A = (-0.05 * torch.exp(n * (math.log(800.0) / 15.0))).unsqueeze(0).expand(192, 16).contiguous().to(DEV)
    p.delta_bias = torch.linspace(-1.0, 1.5, 192, device=DEV)
    for chunk in (1024, 256):
        y, hl = run(p, "chunked", chunk)
        compare(p, y, hl, f"decay-spread/chunked{chunk}")


@pytest.mark.parametrize("impl", ["fwd", "chunked"])
def test_unaligned_rows_and_pointers(impl):
    """Tensors that start 1 element past an allocation (not 16-byte aligned) take the scalar path."""
    p = custom(31, 2, 40, 16, 96, torch.bfloat16)
    def shift(t):
        if t is None:
            return None
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
        v = flat[1:].view(t.shape)
        v.copy_(t)
        return v
    q = I.Problem("shifted", shift(p.u), shift(p.delta), p.A, shift(p.B), shift(p.C), p.D, shift(p.z), p.delta_bias)
    y, hl = run(q, impl, 16)
    compare(q, y, hl, f"unaligned/{impl}")


@pytest.mark.parametrize("impl", ["fwd", "chunked"])
def test_empty_and_degenerate(impl):
    # L = 0: nothing to scan; the final state is the zero start
    p = custom(41, 2, 8, 4, 0)
    hl = torch.full((2, 8, 4), 7.0, device=DEV)
    y = run_out = (ss.scan_fwd if impl == "fwd" else ss.scan_chunked)(
        p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, last_state=hl)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hl).item() == 0 and run_out[0].numel() == 0
    # batch = 0 and dim = 0: no-ops
    for bsz, dim in ((0, 8), (2, 0)):
        q = custom(42, max(bsz, 1), max(dim, 1), 4, 16)
        u = torch.empty((bsz, dim, 16), device=DEV)
        A = torch.empty((dim, 4), device=DEV)
        BC = torch.empty((bsz, 4, 16), device=DEV)
        out = ss.scan_fwd(u, u, A, BC, BC)
        assert out.shape == (bsz, dim, 16)
    # N = 0: only the gated skip term remains
    q = custom(43, 2, 12, 0, 50)
    y, hl = run(q, impl, 8)
    compare(q, y, hl, f"N=0/{impl}")


def test_degenerate_sizes_decode_conv_bwd():
    """Zero batch rows, channels or steps on the decode step, the convolution and the backward
    pass: no error, empty outputs, and the backward pass's gradients of an empty sum are zero."""
    # decode: batch 0 or dim 0
    for bsz, dim in ((0, 8), (3, 0)):
        st = torch.empty((bsz, dim, 4), device=DEV)
        v = torch.empty((bsz, dim), device=DEV)
        bc = torch.empty((bsz, 4), device=DEV)
        y = ss.state_update(st, v, v, torch.empty((dim, 4), device=DEV), bc, bc)
        assert y.shape == (bsz, dim)
    # convolution: L = 0 and dim = 0
    for shape in ((2, 8, 0), (2, 0, 64)):
        x = torch.empty(shape, device=DEV, dtype=torch.bfloat16)
        out = ss.causal_conv1d(x, torch.zeros((shape[1], 4), device=DEV))
        assert out.shape == shape
    # backward with dim = 0: dB and dC (sums over channels) are exactly zero
    bsz, N, L = 2, 4, 16
    u = torch.empty((bsz, 0, L), device=DEV)
    BC = torch.randn((bsz, N, L), device=DEV)
    g = ss.scan_bwd(u, u, torch.empty((0, N), device=DEV), BC, BC, dy=torch.empty((bsz, 0, L), device=DEV))
    torch.cuda.synchronize()
    assert g["dB"].shape == (bsz, N, L) and torch.count_nonzero(g["dB"]).item() == 0
    assert g["dC"].shape == (bsz, N, L) and torch.count_nonzero(g["dC"]).item() == 0
    assert ss.device_status() == ss.SS_OK


def test_two_faces_agree():
    """L decode steps from a zero state == scan_fwd == scan_chunked at several chunk lengths."""
    p = custom(51, 2, 70, 16, 129, torch.float32)
    yf, hf = run(p, "fwd")
    for c in (1, 7, 64, 2048):
        yc, hc = run(p, "chunked", c)
        check(host(yc), host(yf), False, f"chunked{c} vs fwd y")
        check(host(hc), host(hf), False, f"chunked{c} vs fwd state")
    st = torch.zeros((2, 70, 16), device=DEV)
    ys = []
    for t in range(p.seqlen):
        ys.append(ss.state_update(st, p.u[:, :, t].contiguous(), p.delta[:, :, t].contiguous(), p.A,
                                  p.B[:, :, t].contiguous(), p.C[:, :, t].contiguous(), D=p.D, z=p.z[:, :, t].contiguous(),
                                  delta_bias=p.delta_bias))
    yd = torch.stack(ys, dim=2)
    check(host(yd), host(yf), False, "decode x L vs fwd y")
    check(host(st), host(hf), False, "decode x L vs fwd state")
    compare(p, yf, hf, "two-faces/fwd")


def test_zero_step_keeps_state_bitwise():
    """dt = 0 (softplus off, raw delta 0, no bias): Abar = 1 and nothing is written into the state."""
    g = torch.Generator(device=DEV).manual_seed(61)
    st = torch.randn((4, 300, 16), device=DEV, generator=g)
    before = st.clone()
    u = torch.randn((4, 300), device=DEV, generator=g)
    BC = torch.randn((4, 16), device=DEV, generator=g)
    A = -torch.rand((300, 16), device=DEV, generator=g) - 0.5
    y = ss.state_update(st, u, torch.zeros_like(u), A, BC, BC, D=torch.ones(300, device=DEV), softplus=False)
    torch.cuda.synchronize()
    assert torch.equal(st, before)
    want = torch.einsum("bdn,bn->bd", before.double(), BC.double()) + u.double()
    assert torch.max(torch.abs(y.double() - want)).item() <= 1e-5 * torch.max(torch.abs(want)).item()


def test_status_codes_on_device():
    p = custom(71, 1, 16, 16, 64)
    with pytest.raises(ss.SSError) as e:
        ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, chunk_len=16, workspace=torch.empty(8, dtype=torch.uint8, device=DEV))
    assert e.value.status == ss.SS_EWORKSPACE
    A65 = torch.zeros((16, 65), device=DEV)
    BC65 = torch.zeros((1, 65, 64), device=DEV)
    with pytest.raises(ss.SSError) as e:
        ss.scan_fwd(p.u, p.delta, A65, BC65, BC65)
    assert e.value.status == ss.SS_EINVAL


@pytest.mark.parametrize("N", [1, 5, 16, 20, 33, 64])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("shift", [False, True], ids=["aligned", "unaligned"])
def test_decode_ragged(N, dtype, shift):
    """Several decode steps from a random state, for state sizes that pad to the next
    supported width, against the oracle's recurrence step by step."""
    g = torch.Generator().manual_seed(80 + N)
    batch, dim, steps = 3, 70, 6
    st0 = torch.randn((batch, dim, N), generator=g)
    if shift:                                  # state rows not 16-byte aligned: scalar path
        flat = torch.empty(st0.numel() + 1, device=DEV)
        state = flat[1:].view(batch, dim, N)
        state.copy_(st0.to(DEV))
    else:
        state = st0.to(DEV).clone()
    A = (-torch.exp(torch.rand((dim, N), generator=g) * 2.0 - 1.0)).to(DEV)
    D = torch.randn((dim,), generator=g).to(DEV)
    bias = (torch.rand((dim,), generator=g) * 2.0 - 3.0).to(DEV)
    sref = st0.double().numpy().reshape(batch * dim, N).copy()
    w = I.to_wire
    for t in range(steps):
        u = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        dl = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        z = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        Bm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
        Cm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
        y = ss.state_update(state, u, dl, A, Bm, Cm, D=D, z=z, delta_bias=bias)
        yr = oracle.state_update(sref, w(u), w(dl), w(A), w(Bm), w(Cm), D=w(D), z=w(z), delta_bias=w(bias),
                                 dtype="bf16" if dtype == torch.bfloat16 else "f32")
        bf = dtype == torch.bfloat16
        check(host(y).reshape(-1), yr, bf, f"decode N={N} step {t} y")
    check(host(state).reshape(batch * dim, N), sref, dtype == torch.bfloat16, f"decode N={N} state")


@pytest.mark.parametrize("zoh", [False, True], ids=["euler", "zoh"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_many_ranges(dtype, zoh):
    """More (batch row, channel range) blocks than the GPU holds at once, with a partial last
    range in every batch row: 40 rows x 5000 channels (the last range of 128 channels holds
    8), N = 16, from a random state, against the oracle."""
    g = torch.Generator().manual_seed(211)
    batch, dim, N, steps = 40, 5000, 16, 3
    st0 = torch.randn((batch, dim, N), generator=g)
    state = st0.to(DEV).clone()
    A = (-torch.exp(torch.rand((dim, N), generator=g) * 3.0 - 1.5)).to(DEV)
    D = torch.randn((dim,), generator=g).to(DEV)
    bias = (torch.rand((dim,), generator=g) * 2.0 - 3.0).to(DEV)
    sref = st0.double().numpy().reshape(batch * dim, N).copy()
    w = I.to_wire
    bf = dtype == torch.bfloat16
    for t in range(steps):
        u = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        dl = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        z = torch.randn((batch, dim), generator=g).to(dtype).to(DEV)
        Bm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
        Cm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
        y = ss.state_update(state, u, dl, A, Bm, Cm, D=D, z=z, delta_bias=bias, zoh=zoh)
        yr = oracle.state_update(sref, w(u), w(dl), w(A), w(Bm), w(Cm), D=w(D), z=w(z), delta_bias=w(bias),
                                 dtype="bf16" if bf else "f32", zoh=zoh)
        check(host(y).reshape(-1), yr, bf, f"decode many ranges step {t} y")
    check(host(state).reshape(batch * dim, N), sref, bf, "decode many ranges state")
    assert ss.device_status(clear=True) == ss.SS_OK


@pytest.mark.parametrize("zoh", [False, True], ids=["euler", "zoh"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 5], ids=["bulk", "per_thread"])
def test_decode_order_does_not_change_results(N, dtype, zoh):
    """Consecutive ss_state_update calls on one state array take its ranges in opposite
    orders.  The same step from the same state on a second array, twice in a row (its
    contents restored in between, so the two runs take opposite orders and one of them the
    order opposite to the first array's), must give bitwise equal states and outputs."""
    g = torch.Generator().manual_seed(900 + N)
    batch, dim = 37, 700
    st0 = torch.randn((batch, dim, N), generator=g).to(DEV)
    A = (-torch.exp(torch.rand((dim, N), generator=g) * 2.0 - 1.0)).to(DEV)
    D = torch.randn((dim,), generator=g).to(DEV)
    bias = (torch.rand((dim,), generator=g) * 2.0 - 3.0).to(DEV)
    ins = [torch.randn((batch, dim), generator=g).to(dtype).to(DEV) for _ in range(3)]
    Bm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
    Cm = (torch.randn((batch, N), generator=g) * 0.5).to(dtype).to(DEV)
    kw = dict(D=D, z=ins[2], delta_bias=bias, zoh=zoh)
    p = st0.clone()
    y_p = ss.state_update(p, ins[0], ins[1], A, Bm, Cm, **kw)
    q = st0.clone()
    for _ in range(2):
        q.copy_(st0)
        y_q = ss.state_update(q, ins[0], ins[1], A, Bm, Cm, **kw)
        torch.cuda.synchronize()
        assert torch.equal(p, q)
        assert torch.equal(y_p, y_q)
    assert ss.device_status(clear=True) == ss.SS_OK


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_chunked_local_pass_cutoff(dtype):
    """Large steps (dt ~ 2..5): every state's weight underflows a few dozen steps back from a
    chunk's end, so the local pass stops early; the result must still match the oracle."""
    p = custom(91, 2, 200, 16, 1024, dtype)
    p.delta_bias = torch.full((200,), 2.5, device=DEV)
    for chunk in (256, 64):
        y, hl = run(p, "chunked", chunk)
        compare(p, y, hl, f"cutoff/chunked{chunk}")


def test_device_status_clean_after_runs():
    """No bounded wait gave up during any of the launches above (or in this test)."""
    p = custom(101, 2, 130, 16, 4096, torch.bfloat16)
    run(p, "fwd")
    run(p, "chunked", 1024)
    assert ss.device_status(clear=True) == ss.SS_OK


@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("fwd_thread", None), ("chunked", 64), ("chunked", 7)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_initial_state(impl, chunk, dtype):
    """Scans started from a given state h0 against the oracle started from the same state."""
    p = custom(111, 2, 90, 16, 296, dtype)
    g = torch.Generator().manual_seed(112)
    h0 = torch.randn((2, 90, 16), generator=g)
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus, return_last_state=True, h0=h0.to(DEV))
    if impl.startswith("fwd"):
        y, hl = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, schedule=impl[4:] or None, **kw)
    else:
        y, hl = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, chunk_len=chunk, **kw)
    yr, hr = oracle_scan(p.to("cpu"), h0=h0.double().numpy().reshape(180, 16))
    bf = dtype == torch.bfloat16
    check(host(y).reshape(180, 296), yr, bf, f"h0/{impl} y")
    check(host(hl).reshape(180, 16), hr, bf, f"h0/{impl} last_state")


@pytest.mark.parametrize("impl", ["fwd", "chunked"])
def test_prompt_state_handoff(impl):
    """A prompt's state, computed once and handed to the next call through h0, gives
    the same outputs as one scan over prompt + continuation; the state then continues
    in decode steps."""
    p = custom(113, 1, 130, 16, 512, torch.bfloat16)
    kw = dict(D=p.D, delta_bias=p.delta_bias, return_last_state=True)
    split = 320

    def part(t, a, b):
        return t[:, :, a:b].contiguous()

    def call(lo, hi, h0=None):
        args = [part(t, lo, hi) for t in (p.u, p.delta)] + [p.A] + [part(t, lo, hi) for t in (p.B, p.C)]
        extra = dict(z=part(p.z, lo, hi), h0=h0, **kw)
        if impl == "fwd":
            return ss.scan_fwd(*args, **extra)
        return ss.scan_chunked(*args, chunk_len=64, **extra)

    y_all, h_all = call(0, 512)
    y1, h1 = call(0, split)
    y2, h2 = call(split, 512, h0=h1)
    check(host(torch.cat([y1, y2], dim=2)), host(y_all), True, "handoff y")
    check(host(h2), host(h_all), True, "handoff state")
    # L = 0 returns the initial state
    _, h_empty = call(512, 512, h0=h2)
    assert torch.equal(h_empty, h2)


def test_decode_cuda_graph_matches_eager():
    """The multi-step decode replayed from a CUDA graph (as a server would run it) gives
    bitwise the eager steps' y and final state, and both match the oracle's recurrence."""
    batch, dim, N, steps = 4, 300, 16, 64
    st_in = I.decode_stream(seed=41, batch=batch, dim=dim, dstate=N, steps=steps, device=DEV, gen_device="cpu")

    def run(state, ys):
        for t in range(steps):
            ss.state_update(state, st_in.u[t], st_in.delta[t], st_in.A, st_in.B[t], st_in.C[t], D=st_in.D,
                            z=st_in.z[t], delta_bias=st_in.delta_bias, y=ys[t])

    s_e = torch.zeros((batch, dim, N), device=DEV)
    y_e = torch.empty((steps, batch, dim), device=DEV)
    run(s_e, y_e)
    s_g = torch.zeros((batch, dim, N), device=DEV)
    y_g = torch.empty((steps, batch, dim), device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(s_g, y_g)                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(s_g, y_g)
    for _ in range(2):                                  # replays start from a reset state
        s_g.zero_()
        y_g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_g, y_e) and torch.equal(s_g, s_e)
    w = I.to_wire
    sref = np.zeros((batch * dim, N))
    yref = np.empty((steps, batch * dim))
    for t in range(steps):
        yref[t] = oracle.state_update(sref, w(st_in.u[t]), w(st_in.delta[t]), w(st_in.A), w(st_in.B[t]),
                                      w(st_in.C[t]), D=w(st_in.D), z=w(st_in.z[t]), delta_bias=w(st_in.delta_bias),
                                      dtype="bf16")
    check(y_e.reshape(steps, -1).cpu().numpy(), yref, True, "graph decode y")
    check(s_e.reshape(-1, N).cpu().numpy(), sref, True, "graph decode state")
