"""Run by tests/test_debug_bounds_gpu.py in a child process with SS_LIBRARY=debug: every kernel
family of the debug build (device-side index checks) on small problems, against the oracle, and
then the status word, which must show no failed check; finally the self-test check that records
one.  Prints one line per case and exits non-zero on the first failure."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import check, check_bf16_out, host

DEV = "cuda"
w = I.to_wire


def problem(seed, batch, dim, N, L, dtype):
    p = I.selective_problem("dbg", seed=seed, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=dtype, bc_std=0.5,
                            d_mode="normal", gate=True, device=DEV, gen_device="cpu")
    g = torch.Generator().manual_seed(seed + 9)
    p.A = (-torch.exp(torch.rand((dim, N), generator=g) * 3.0 - 1.0)).to(DEV)
    return p


def shifted(t):
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    v = flat[1:].view(t.shape)
    v.copy_(t)
    return v


def scan_case(name, p, run, zoh=False):
    y, hl = run(p)
    torch.cuda.synchronize()
    bf = p.in_dtype == I.BF16
    yr, hr = oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z), delta_bias=w(p.delta_bias),
                         dtype="bf16" if bf else "f32", zoh=zoh)
    n = p.batch * p.dim
    check(host(y).reshape(n, p.seqlen), yr, bf, name + " y")
    check(host(hl).reshape(n, p.dstate), hr, bf, name + " state")
    print("ok", name, flush=True)


def main():
    assert ss.debug_bounds_build(), "the debug build is not the loaded library"
    assert ss.device_status(clear=True) in (ss.SS_OK, ss.SS_ETIMEOUT, ss.SS_EBOUNDS)
    kw = lambda p, **o: dict(D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True, **o)
    for dt in (torch.bfloat16, torch.float32):
        tag = "bf16" if dt == torch.bfloat16 else "f32"
        p = problem(1, 2, 70, 16, 328, dt)
        scan_case(f"fwd thread {tag}", p, lambda q: ss.scan_fwd(q.u, q.delta, q.A, q.B, q.C, schedule="thread", **kw(q)))
        scan_case(f"fwd warp {tag}", p, lambda q: ss.scan_fwd(q.u, q.delta, q.A, q.B, q.C, schedule="warp", **kw(q)))
        scan_case(f"chunked grouped {tag}", p,
                  lambda q: ss.scan_chunked(q.u, q.delta, q.A, q.B, q.C, chunk_len=64, **kw(q)))
        scan_case(f"chunked grouped zoh {tag}", p,
                  lambda q: ss.scan_chunked(q.u, q.delta, q.A, q.B, q.C, chunk_len=64, **kw(q, zoh=True)), zoh=True)
        p32 = problem(2, 1, 40, 32, 136, dt)
        scan_case(f"chunked tma local N=32 {tag}", p32,
                  lambda q: ss.scan_chunked(q.u, q.delta, q.A, q.B, q.C, chunk_len=48, **kw(q)))
        pr = problem(3, 2, 33, 5, 77, dt)
        scan_case(f"fwd ring ragged {tag}", pr, lambda q: ss.scan_fwd(q.u, q.delta, q.A, q.B, q.C, **kw(q)))
        scan_case(f"chunked ring ragged {tag}", pr,
                  lambda q: ss.scan_chunked(q.u, q.delta, q.A, q.B, q.C, chunk_len=7, **kw(q)))
        pu = problem(4, 1, 24, 16, 96, dt)
        q = I.Problem("dbg_shift", shifted(pu.u), shifted(pu.delta), pu.A, shifted(pu.B), shifted(pu.C), pu.D,
                      shifted(pu.z), pu.delta_bias)
        scan_case(f"chunked unaligned {tag}", q,
                  lambda r: ss.scan_chunked(r.u, r.delta, r.A, r.B, r.C, chunk_len=16, **kw(r)))
        # decode: bulk path (aligned, N % 4 == 0) and per-thread path (N = 5)
        for N in (16, 5):
            st = torch.zeros((3, 50, N), device=DEV)
            sref = np.zeros((150, N))
            pd = problem(5 + N, 3, 50, N, 4, dt)
            for t in range(4):
                col = lambda x: x[:, :, t].contiguous()
                y = ss.state_update(st, col(pd.u), col(pd.delta), pd.A, col(pd.B), col(pd.C), D=pd.D, z=col(pd.z),
                                    delta_bias=pd.delta_bias)
                yr = oracle.state_update(sref, w(col(pd.u)), w(col(pd.delta)), w(pd.A), w(col(pd.B)), w(col(pd.C)),
                                         D=w(pd.D), z=w(col(pd.z)), delta_bias=w(pd.delta_bias),
                                         dtype="bf16" if dt == torch.bfloat16 else "f32")
                check(host(y).reshape(-1), yr, dt == torch.bfloat16, f"decode N={N} {tag}")
            print("ok", f"decode N={N} {tag}", flush=True)
        # causal conv1d
        x = problem(6, 2, 40, 4, 600, dt).u
        wt = torch.randn((40, 4), generator=torch.Generator().manual_seed(7)).to(DEV) * 0.5
        out = ss.causal_conv1d(x, wt)
        ref = oracle.conv1d(w(x), w(wt), None, dtype="bf16" if dt == torch.bfloat16 else "f32")
        if dt == torch.bfloat16:
            check_bf16_out(host(out), ref, f"conv1d {tag}")
        else:
            check(host(out), ref, False, f"conv1d {tag}")
        print("ok", f"conv1d {tag}", flush=True)
        # backward pass
        pb = problem(8, 2, 40, 16, 136, dt)
        ct = I.cotangents(seed=9, batch=2, dim=40, dstate=16, seqlen=136, device=DEV, gen_device="cpu")
        g = ss.scan_bwd(pb.u, pb.delta, pb.A, pb.B, pb.C, D=pb.D, z=pb.z, delta_bias=pb.delta_bias, dy=ct.dy,
                        dlast=ct.dlast, h0=ct.h0, want_dh0=True)
        torch.cuda.synchronize()
        r = oracle.scan_bwd(w(pb.u), w(pb.delta), w(pb.A), w(pb.B), w(pb.C), D=w(pb.D), z=w(pb.z),
                            delta_bias=w(pb.delta_bias), dtype="bf16" if dt == torch.bfloat16 else "f32",
                            dy=host(ct.dy).reshape(80, -1), dlast=host(ct.dlast).reshape(80, 16),
                            h0=host(ct.h0).reshape(80, 16))
        for k in ("du", "ddelta", "dz", "dB", "dC", "dA", "dh0"):
            got = host(g[k]).astype(np.float64)
            ref = np.asarray(r[k]).reshape(got.shape)
            sc = np.maximum(np.abs(ref), np.sqrt(np.mean(ref * ref)))
            e = float(np.max(np.abs(got - ref) / sc))
            assert e <= 1e-4, f"bwd {k} {tag}: {e}"
        print("ok", f"bwd {tag}", flush=True)
    st = ss.device_status(clear=True)
    assert st == ss.SS_OK, f"status word after the cases: {ss.lib().ss_status_string(st).decode()}"
    print("ok status clean", flush=True)
    ss.selftest_bounds()
    assert ss.device_status(clear=True) == ss.SS_EBOUNDS
    assert ss.device_status() == ss.SS_OK
    print("ok selftest records SS_EBOUNDS", flush=True)


if __name__ == "__main__":
    main()
