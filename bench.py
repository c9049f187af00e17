#!/usr/bin/env python3
"""Benchmark of the B300 selective scan (Mamba S6).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One "step" is one chunked forward scan (local pass, carry, fix-up: every row
of the forward hot path) over the Mamba-2.8B-shaped long-sequence workload:
batch 1, D = 5120 channels, N = 16 states, L = 65536 steps, chunk 2048, bf16
u/delta/B/C/z, fp32 A/D/delta_bias/state/y, synthetic seeded inputs resident
in HBM.  The inputs (3.4 GB) are far larger than the 126 MB L2, so no flush
is needed between steps.

Rank 0 prints one JSON line.  `value` is B*D*L elements per second for the
whole job (every rank runs its own replica of the workload: the scan shards
over independent channels and batch rows, with no collective on the data
path).  The line also carries the roofline of the dominant kernel, the whole
step's roofline, per-kernel times measured with CUDA events inside the timed
region, the end-to-end figure through host buffers (and the same host copies
timed without the scan), clocks sampled during the timed region, side
measurements (decode, causal conv1d, the zero-order-hold step, ss_scan_fwd on
the 130M-shaped layer and under both of its schedules, the backward pass), the
ex2 throughput of the running GPU (the SFU peak that the exponential roofline
divides by, `sfu`), and the fp64 oracle timed on the host cores as a CPU
baseline, whose sample channels are also compared with the bench's own outputs
(`cpu_baseline.parity_sample`).

`--impl reference` times the fp64 CPU oracle instead (the reference arm):
same metric and workload, a bounded sample of channels per step.

Profiling aids (one JSON object, no bench line): `--bwd-only` times only the
backward pass, `--schedules-only` only ss_scan_fwd under its two schedules;
`--dim` / `--seqlen` shrink the workload; `--no-decode`, `--no-e2e`,
`--no-sfu` and `--no-cpu-baseline` drop legs.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

METRIC = "scan throughput (B·D·L elems/s, HBM GB/s) and % of HBM/SFU roofline, 1×B300"
WORKLOAD = "mamba2p8b_long_bf16"
CHUNK = 2048
SMS = 148
SM_MAX_MHZ = 2032.0
# Fallback only, used when the ex2 throughput leg below cannot run: 32 MUFU.EX2 lanes per
# clock per SM, the rate ncu's pipe_xu utilisation implies for the scan kernels.  The bench
# line's SFU peak is normally the rate that leg measures on the running GPU.
EX2_PER_CLK_PER_SM_FALLBACK = 32


# ----------------------------------------------------------------- measured DRAM traffic

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# kernel of the chunked step, from one ncu capture of this workload at full
# size (the summary and its command are under profiles/).  The figures belong
# to the kernel sources with the hash below; after any change to those sources
# they no longer describe the running kernels and the bench reports null.
TRAFFIC = {
    "sources": "501695340deecda3",
    # local phase = order_channels_kernel (0.00036 GB read) + local_sorted_kernel
    # (0.96253 GB read + 0.00856 GB written): rows of channels whose weights have
    # underflowed are never fetched, so it reads less than the 1.30 GB of u and delta.
    "local": 971450000,
    "carry": 11490000,       # carry_kernel: 0.01149 GB read (writes stay in L2)
    "fixup": 3340000000,     # scan_tma_kernel (fix-up): 2.03 GB read + 1.31 GB written
}


# The files that define the chunked step's three kernels and how they are launched.
STEP_SOURCES = ("ss_device.cuh", "ss_kernels.cuh", "ss_kernels_tma.cuh", "ss_tma.cuh", "ss_tma_launch.cuh",
                "ss_scan_tma.cu", "ss_scan_local.cu", "ss_occupancy.cuh", "ss_types.h", "ss_dispatch.cuh",
                "ss_local_sorted.cu")


def kernel_sources_hash():
    """sha256 (first 16 hex digits) over the sources of the chunked step's kernels."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(HERE, "selective_state_space_117_b300", "csrc")
    for f in STEP_SOURCES:
        h.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, L):
    if TRAFFIC["sources"] != kernel_sources_hash() or L != 65536:
        return None
    return TRAFFIC.get(kernel)


# ----------------------------------------------------------------- roofline model

def workload_counts(batch, dim, dstate, seqlen, in_bytes=2, gate=True):
    """Algorithmic bytes and exponentials of one forward scan.
    bytes: u, delta (and z) read once, y written once (fp32), B and C read once per
    batch row, A, D, delta_bias read once, the final state written once.
    exps: N discretization exps per element, one in the softplus, one in the SiLU gate."""
    elems = batch * dim * seqlen
    per_elem = in_bytes * (3 if gate else 2) + 4
    byts = elems * per_elem + batch * 2 * dstate * seqlen * in_bytes + dim * dstate * 4 + 2 * dim * 4 \
        + batch * dim * dstate * 4
    exps = elems * (dstate + 1 + (1 if gate else 0))
    return elems, byts, exps


def peaks(sfu=None):
    """HBM peak from MEASURED_PEAKS.json; the SFU (ex2) peak from the throughput leg when it
    ran (`sfu`), else the fallback rate at the maximum SM clock."""
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    hbm, src = 6400.0, "fallback"
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        hbm, src = float(pk.get("hbm_gbs", hbm)), "measured"
    if sfu and sfu.get("texps"):
        return {"hbm_gbs": hbm, "hbm_src": src, "sfu_texps": sfu["texps"],
                "sfu_src": "measured: ex2.approx.ftz.f32 throughput loop (ss_measure_ex2), best of "
                           f"{sfu['launches']} launches at {sfu['sm_mhz']} MHz"}
    texps = SMS * EX2_PER_CLK_PER_SM_FALLBACK * SM_MAX_MHZ * 1e6 / 1e12
    return {"hbm_gbs": hbm, "hbm_src": src, "sfu_texps": texps,
            "sfu_src": f"fallback: {SMS} SMs x {EX2_PER_CLK_PER_SM_FALLBACK}/clk/SM x {SM_MAX_MHZ:.0f} MHz"}


def measure_sfu(ss, torch, launches=20, iters=4096):
    """The ex2.approx.ftz.f32 throughput of the running GPU (ss_measure_ex2): 8 blocks of 256
    threads per SM, each thread 8 independent chains; every launch timed with CUDA events on
    the current stream; the best launch gives the peak.  Clocks are sampled meanwhile so the
    rate can also be stated per clock and per SM."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    blocks = 8 * sms
    sink = torch.empty((blocks,), dtype=torch.float32, device="cuda")
    for _ in range(3):
        n = ss.measure_ex2(blocks, iters, sink=sink)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    with ClockSampler(device_index_for_smi(torch)) as clk:
        for e0, e1 in ev:
            e0.record()
            ss.measure_ex2(blocks, iters, sink=sink)
            e1.record()
        torch.cuda.synchronize()
    ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
    best, med = ms[0], ms[len(ms) // 2]
    c = clk.summary()
    mhz = c["sm_mhz"] or SM_MAX_MHZ
    texps = n / (best * 1e-3) / 1e12
    return {"texps": round(texps, 4), "texps_median": round(n / (med * 1e-3) / 1e12, 4),
            "per_clk_per_sm": round(texps * 1e12 / (sms * mhz * 1e6), 3), "sm_mhz": mhz, "sms": sms,
            "ex2_per_launch": n, "ms_best": round(best, 4), "launches": launches,
            "clock_reasons": c["reasons"], "gpu_launches": launches + 3}


def roofline_terms(byts, exps, ms, pk):
    t = ms * 1e-3
    gbs = byts / t / 1e9
    texps = exps / t / 1e12
    t_hbm = byts / (pk["hbm_gbs"] * 1e9)
    t_sfu = exps / (pk["sfu_texps"] * 1e12)
    if t_sfu >= t_hbm:
        return {"bound": "alu", "achieved": round(texps, 4), "peak": round(pk["sfu_texps"], 4), "unit": "Texp/s",
                "frac": round(texps / pk["sfu_texps"], 4), "hbm_gbs": round(gbs, 1),
                "hbm_frac": round(gbs / pk["hbm_gbs"], 4)}
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / pk["hbm_gbs"], 4), "texps": round(texps, 4)}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) while the timed region runs.  Entering waits (up to
    10 s) for the first sample, so that the sampler's start-up, which can hold up the
    process's own CUDA calls for a moment, falls before the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.idx = device_index
        self.out = ""
        self.lines = []
        self.reader = None

    def __enter__(self):
        import threading
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.idx is not None:
            cmd += ["-i", str(self.idx)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        first = threading.Event()

        def pump():
            for line in self.proc.stdout:
                self.lines.append(line)
                first.set()
            first.set()

        self.reader = threading.Thread(target=pump, daemon=True)
        self.reader.start()
        first.wait(timeout=10.0)
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self.reader is not None:
                self.reader.join(timeout=5)
            self.out = "".join(self.lines)

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), float(f[2]), float(f[3]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [r for r in rows if r[3] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(busy), "power_w_max": max(r[2] for r in busy)}


def device_index_for_smi(torch):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    local = torch.cuda.current_device()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return local


# ----------------------------------------------------------------- distributed helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def barrier_and_max(value: float, world: int):
    """The maximum of `value` over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU baseline (oracle)

def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(p, nchan):
    """Host copies of the first `nchan` channels of a problem (wire format for the oracle)."""
    from selective_state_space_117_b300 import inputs as I
    sub = lambda t: I.to_wire(t[:, :nchan].contiguous()) if t is not None else None
    sub0 = lambda t: I.to_wire(t[:nchan].contiguous()) if t is not None else None
    return dict(u=sub(p.u), delta=sub(p.delta), z=sub(p.z), A=sub0(p.A), D=sub0(p.D), delta_bias=sub0(p.delta_bias),
                B=I.to_wire(p.B), C=I.to_wire(p.C))


def time_oracle(sample, threads, out=None):
    """Seconds the oracle takes on the sample; its (y, last_state) go into `out` when given."""
    import oracle
    t0 = time.perf_counter()
    r = oracle.scan(sample["u"], sample["delta"], sample["A"], sample["B"], sample["C"], D=sample["D"],
                    z=sample["z"], delta_bias=sample["delta_bias"], softplus=True, dtype="bf16", nthreads=threads)
    dt = time.perf_counter() - t0
    if out is not None:
        out["y"], out["h"] = r
    return dt


def parity_of_sample(res, y, hl, nchan):
    """The bench's own outputs on the oracle's sample channels (batch row 0), under the bf16 rule
    max |err| <= 2e-3 rms(ref), with the unfloored relative error over |ref| >= 1e-2 rms."""
    import numpy as np
    out = {"channels": nchan, "rule": "max|err|/rms(ref) <= 2e-3 (bf16 inputs)"}
    for key, got, ref in (("y", y[0, :nchan].float().cpu().numpy(), res["y"]),
                          ("last_state", hl[0, :nchan].float().cpu().numpy(), res["h"])):
        ref = np.asarray(ref, dtype=np.float64).reshape(got.shape)
        err = np.abs(got.astype(np.float64) - ref)
        r = float(np.sqrt(np.mean(ref * ref)))
        keep = np.abs(ref) >= 1e-2 * r
        out[key] = {"max_abs_err": float(err.max()), "rms_ref": r, "max_err_over_rms": float(err.max() / r),
                    "rel_unfloored": float(np.max(err[keep] / np.abs(ref[keep]))) if keep.any() else 0.0}
    return out


def cpu_baseline(p, budget_s=20.0, y=None, hl=None):
    """The oracle on the host cores over a bounded channel sample (about `budget_s` of wall time).
    With the GPU's y and final state of the same workload, the sample's outputs are also compared
    with them (`parity_sample`)."""
    import oracle
    oracle.build()
    threads = host_threads()
    L = p.seqlen
    probe = oracle_sample(p, min(threads, p.dim))
    per_chan = time_oracle(probe, threads) / min(threads, p.dim)
    nchan = int(min(p.dim, max(threads, budget_s / max(per_chan, 1e-9))))
    nchan = min(p.dim, max(threads, (nchan // threads) * threads))
    sample = oracle_sample(p, nchan)
    res = {}
    dt = time_oracle(sample, threads, res)
    elems = p.batch * nchan * L
    # one core, on a few channels; per-channel work is the same for every channel, so the
    # whole workload's single-core time is this scaled linearly
    n1 = 4
    t1 = time_oracle(oracle_sample(p, n1), 1)
    one = p.batch * n1 * L / t1
    return {"value": elems / dt, "unit": "elem/s", "cores": threads, "kind": "oracle",
            "sample": f"{nchan} of {p.dim} channels x L={L} (fp64 C oracle, OpenMP over channels), {dt:.1f} s",
            "single_core": {"value": one, "unit": "elem/s", "sample": f"{n1} channels x L={L} on 1 thread, {t1:.2f} s",
                            "scaled_workload_s": round(p.batch * p.dim * L / one, 1),
                            "note": "scaled linearly from the sample to all channels"},
            **({"parity_sample": parity_of_sample(res, y, hl, nchan)} if y is not None else {})}


# ----------------------------------------------------------------- the reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from selective_state_space_117_b300 import inputs as I
    import oracle
    oracle.build()
    p = I.workload(WORKLOAD, device="cpu", gen_device="cpu", dim=512)   # the channels the samples draw from
    threads = host_threads()
    probe = oracle_sample(p, threads)
    per_chan = time_oracle(probe, threads) / threads
    budget = 150.0 / max(1, args.steps + args.warmup)
    nchan = max(1, int(min(512, max(threads, budget / max(per_chan, 1e-9)))))
    sample = oracle_sample(p, nchan)
    for _ in range(args.warmup):
        time_oracle(sample, threads)
    t = [time_oracle(sample, threads) for _ in range(args.steps)]
    tot = sum(t)
    elems = nchan * p.seqlen
    value = elems * args.steps / tot
    cfg = {"workload": f"{WORKLOAD}: batch=1, D=5120, N=16, L=65536, chunk {CHUNK}; bf16 inputs, fp32 state",
           "sample_per_step": f"{nchan} channels x L={p.seqlen}"}
    line = {"metric": METRIC, "value": value, "unit": "elem/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "elem/s", "cores": threads, "kind": "oracle",
                             "sample": f"{nchan} channels x L={p.seqlen} per step"},
            "e2e": {"value": value, "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    import selective_state_space_117_b300 as ss
    from selective_state_space_117_b300 import inputs as I

    sfu = None
    if not args.no_sfu:
        try:
            sfu = measure_sfu(ss, torch)
        except Exception as e:   # the line then states the fallback peak it used
            sfu = {"error": str(e)}
    pk = peaks(sfu)
    if args.schedules_only:            # the ss_scan_fwd schedule comparison alone (for profiling it)
        if rank == 0:
            print(json.dumps({"fwd_schedules": bench_fwd_schedules(ss, I, torch)}), flush=True)
        return 0
    p = I.workload(WORKLOAD, device="cuda", gen_device="cuda", dim=args.dim, seqlen=args.seqlen)
    Bt, Dm, N, L = p.batch, p.dim, p.dstate, p.seqlen
    if args.bwd_only:                  # the backward leg alone (for profiling it); one JSON line
        if rank == 0:
            print(json.dumps({"bwd": bench_bwd(ss, I, torch, p, pk, None, reps=max(1, args.steps))}), flush=True)
        return 0
    elems, byts, exps = workload_counts(Bt, Dm, N, L)
    y = torch.empty((Bt, Dm, L), dtype=torch.float32, device="cuda")
    hl = torch.empty((Bt, Dm, N), dtype=torch.float32, device="cuda")
    ws = torch.empty((ss.chunked_workspace_bytes(Bt, Dm, N, L, CHUNK),), dtype=torch.uint8, device="cuda")
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, chunk_len=CHUNK, y=y, last_state=hl, workspace=ws)
    phases = [(ss.PHASE_LOCAL, "local"), (ss.PHASE_CARRY, "carry"), (ss.PHASE_FIXUP, "fixup")]

    def step(evs=None):
        for i, (ph, _) in enumerate(phases):
            ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, phase=ph, **kw)
            if evs is not None:
                evs[i + 1].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device_index_for_smi(torch)) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0.record()
        for k in range(args.steps):
            ev[k][0].record()
            step(ev[k])
        t1.record()
        torch.cuda.synchronize()
        barrier(world)
    total_ms = barrier_and_max(t0.elapsed_time(t1), world)
    ms = total_ms / args.steps
    per_kernel = {name: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps))
                  for i, (_, name) in enumerate(phases)}
    step_median = statistics.median(ev[k][0].elapsed_time(ev[k][len(phases)]) for k in range(args.steps))
    ksum = sum(per_kernel.values())
    dominant = max(per_kernel, key=per_kernel.get)
    value = elems * world / (ms * 1e-3)

    # Roofline of the dominant kernel.  The fix-up pass produces every output, so its algorithmic
    # work is the whole forward scan's; the local and carry passes are the overhead of chunking.
    line_kernels = {n: {"ms": round(v, 4), "share": round(v / ksum, 4), "traffic": traffic_for(n, L)}
                    for n, v in per_kernel.items()}
    roof_dom = roofline_terms(byts, exps, per_kernel[dominant], pk)
    roof_dom.update({"kernel": f"{dominant} pass", "traffic": traffic_for(dominant, L),
                     "peak_src": pk["sfu_src"] if roof_dom["bound"] == "alu" else pk["hbm_src"]})
    roof_step = roofline_terms(byts, exps, ms, pk)

    e2e = None if args.no_e2e else bench_e2e(ss, torch, p, y, hl, ws, world, elems, min(8, args.steps))
    dec = None if args.no_decode else bench_decode(ss, I, torch, pk)
    conv = None if args.no_decode else bench_conv(ss, torch, pk)
    side = {}
    if not args.no_decode:
        side["zoh"] = bench_zoh_step(ss, torch, p, kw, elems)
        side["fwd_layer"] = bench_fwd_layer(ss, I, torch, pk)
        side["fwd_schedules"] = bench_fwd_schedules(ss, I, torch)
        side["bwd"] = bench_bwd(ss, I, torch, p, pk, ms)

    line = {
        "metric": METRIC, "value": value, "unit": "elem/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": round(step_median, 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: batch=1, D={Dm}, N=16, L={L}, chunk {CHUNK}",
                   "entry_point": "ss_scan_chunked (phases local, carry, fixup)",
                   "inputs": "bf16 u/delta/B/C/z; fp32 A/D/delta_bias/state/y; arithmetic fp32",
                   "l2": f"no flush: inputs {byts / 1e9:.2f} GB per step >> 126 MB L2",
                   "parallelism": f"replicas x{world}"},
        "hbm_gbs": round(byts / (ms * 1e-3) / 1e9, 1),
        "roofline": roof_dom,
        "roofline_step": roof_step,
        "kernels": line_kernels,
        "kernel_sources": kernel_sources_hash(),
        "e2e": e2e,
        "gpu_launches": args.steps * (len(phases) + 1),   # the local phase orders the channels first
        "clocks": clk.summary(),
        "peaks": pk,
        "sfu": sfu,
    }
    if dec is not None:
        line["decode"] = dec
    if conv is not None:
        line["conv1d"] = conv
    line.update(side)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        step()                       # y and the final state of the workload again (the side legs reused them)
        torch.cuda.synchronize()
        line["cpu_baseline"] = cpu_baseline(p, y=y, hl=hl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def bench_e2e(ss, torch, p, y, hl, ws, world, elems, e2e_steps):
    """The same scan through the public API with pinned host buffers: every step copies its
    inputs host->device and its outputs (y, final state) device->host inside the timed region.
    Steps are pipelined over three streams with two buffer sets, so step i+1's upload and step
    i-1's download overlap step i's scan; each step still moves all of its own bytes."""
    e2e_steps = max(2, e2e_steps)
    Bt, Dm, N, L = p.batch, p.dim, p.dstate, p.seqlen
    names = ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")
    hp = {k: getattr(p, k).cpu().pin_memory() for k in names}
    hy = [torch.empty((Bt, Dm, L), dtype=torch.float32).pin_memory() for _ in range(2)]
    hh = [torch.empty((Bt, Dm, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    dp = [{k: torch.empty_like(v, device="cuda") for k, v in hp.items()} for _ in range(2)]
    dy = [y, torch.empty_like(y)]
    dh = [hl, torch.empty_like(hl)]
    wss = [ws, torch.empty_like(ws)]
    h2d = sum(v.numel() * v.element_size() for v in hp.values())
    d2h = hy[0].numel() * 4 + hh[0].numel() * 4
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]     # the scan has finished reading buffer set b

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev_free[b])
            for k, v in hp.items():
                dp[b][k].copy_(v, non_blocking=True)
            ev_up[b].record(s_up)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_up[b])
            s_run.wait_event(ev_down[b])                  # step i-2's outputs have left buffer set b
            d = dp[b]
            ss.scan_chunked(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                            delta_bias=d["delta_bias"], chunk_len=CHUNK, y=dy[b], last_state=dh[b],
                            workspace=wss[b], stream=s_run)
            ev_run[b].record(s_run)
            ev_free[b].record(s_run)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_run[b])
            hy[b].copy_(dy[b], non_blocking=True)
            hh[b].copy_(dh[b], non_blocking=True)
            ev_down[b].record(s_down)

    for e in ev_free + ev_down:
        e.record(torch.cuda.current_stream())
    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    barrier(world)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    a0.record(cur)
    for st in (s_up, s_run, s_down):
        st.wait_event(a0)
    for i in range(e2e_steps):
        e2e_step(i)
    for st in (s_up, s_run, s_down):
        cur.wait_stream(st)
    a1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = barrier_and_max(a0.elapsed_time(a1), world) / e2e_steps

    # The host link alone: the same uploads and downloads on the same streams, no scan.
    def copies(i):
        b = i % 2
        with torch.cuda.stream(s_up):
            for k, v in hp.items():
                dp[b][k].copy_(v, non_blocking=True)
        with torch.cuda.stream(s_down):
            hy[b].copy_(dy[b], non_blocking=True)
            hh[b].copy_(dh[b], non_blocking=True)

    copies(0)
    torch.cuda.synchronize()
    a0.record(cur)
    for st in (s_up, s_down):
        st.wait_event(a0)
    for i in range(e2e_steps):
        copies(i)
    for st in (s_up, s_down):
        cur.wait_stream(st)
    a1.record(cur)
    torch.cuda.synchronize()
    link_ms = a0.elapsed_time(a1) / e2e_steps
    del dp, hp, hy, hh
    return {"value": elems * world / (e2e_ms * 1e-3), "unit": "elem/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
            "pipelined": "upload / scan / download on three streams, two buffer sets",
            "copies_only_ms_per_step": round(link_ms, 3),
            "copies_only_gbs": round((h2d + d2h) / (link_ms * 1e-3) / 1e9, 1)}


def time_scan_fwd(ss, torch, p, schedule, reps):
    """Average ms of ss_scan_fwd over reps calls (CUDA events around the loop)."""
    y = torch.empty((p.batch, p.dim, p.seqlen), device="cuda")
    hl = torch.empty((p.batch, p.dim, p.dstate), device="cuda")
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus, y=y, last_state=hl, schedule=schedule)
    for _ in range(3):
        ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, **kw)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, **kw)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def time_scan_chunked(ss, torch, p, chunk, reps):
    """Average ms of ss_scan_chunked at `chunk` over reps calls (CUDA events around the loop)."""
    y = torch.empty((p.batch, p.dim, p.seqlen), device="cuda")
    hl = torch.empty((p.batch, p.dim, p.dstate), device="cuda")
    ws = torch.empty((ss.chunked_workspace_bytes(p.batch, p.dim, p.dstate, p.seqlen, chunk),), dtype=torch.uint8,
                     device="cuda")
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, softplus=p.softplus, y=y, last_state=hl, chunk_len=chunk,
              workspace=ws)
    for _ in range(3):
        ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, **kw)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, **kw)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def bench_fwd_layer(ss, I, torch, pk, reps=20):
    """The Mamba-130M-shaped layer (batch 8, D 1536, N 16, L 2048, bf16 inputs, gate):
    ss_scan_fwd (one pass; 12288 channels at one thread each fill 2.6 warps per SM) and
    ss_scan_chunked at chunks of 256, 512 and 1024 steps (4 to 8 times the threads, plus a
    local pass and a carry); the roofline is stated for the faster entry point."""
    p = I.workload("mamba130m_layer_bf16", device="cuda", gen_device="cuda")
    elems, byts, exps = workload_counts(p.batch, p.dim, p.dstate, p.seqlen)
    ms = time_scan_fwd(ss, torch, p, None, reps)
    chunked = {c: time_scan_chunked(ss, torch, p, c, reps) for c in (256, 512, 1024)}
    best_c = min(chunked, key=chunked.get)
    best = ("ss_scan_fwd", ms) if ms <= chunked[best_c] else (f"ss_scan_chunked (chunk {best_c})", chunked[best_c])
    roof = roofline_terms(byts, exps, best[1], pk)
    return {"workload": "mamba130m_layer_bf16: batch=8, D=1536, N=16, L=2048, bf16 inputs, gate",
            "entry_point": "ss_scan_fwd", "schedule": "thread (12288 channels)", "ms": round(ms, 4),
            "chunked_ms": {str(c): round(v, 4) for c, v in chunked.items()},
            "best": best[0], "best_ms": round(best[1], 4), "elem_per_s": elems / (best[1] * 1e-3), "roofline": roof,
            "roofline_fwd": roofline_terms(byts, exps, ms, pk),
            "note": "inputs 0.25 GB, about twice the L2: no flush between repetitions",
            "gpu_launches": reps * (1 + 3 * 4) + 9 * 4 + 3}


def bench_fwd_schedules(ss, I, torch, reps=50):
    """ss_scan_fwd under both schedules (SS_FLAG_SCHED_WARP first, then _THREAD) on the
    medium workload (batch 2, D 256, N 16, L 2048, fp32 inputs, gate: 512 channels, too
    few to fill the GPU one thread each) and on the Mamba-130M-shaped layer (12288
    channels, where one thread per channel wins).  Each schedule runs 3 untimed and
    `reps` timed calls."""
    out = {"entry_point": "ss_scan_fwd", "gpu_launches": 4 * reps}
    for key, name, desc, note in (
            ("medium", "medium_fp32_gate", "batch=2, D=256, N=16, L=2048, fp32 inputs, gate",
             "inputs 13 MB stay in L2 between repetitions"),
            ("mamba130m", "mamba130m_layer_bf16", "batch=8, D=1536, N=16, L=2048, bf16 inputs, gate",
             "inputs 0.25 GB, about twice the L2")):
        p = I.workload(name, device="cuda", gen_device="cuda")
        elems = p.batch * p.dim * p.seqlen
        r = {"workload": f"{name}: {desc}", "note": note}
        for sched in ("warp", "thread"):
            ms = time_scan_fwd(ss, torch, p, sched, reps)
            r[f"ms_{sched}"] = round(ms, 4)
            r[f"elem_per_s_{sched}"] = elems / (ms * 1e-3)
        out[key] = r
        del p
    return out


def bench_zoh_step(ss, torch, p, kw, elems, reps=5):
    """The long-sequence chunked step with the zero-order-hold input weight."""
    for _ in range(2):
        ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, zoh=True, **kw)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, zoh=True, **kw)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    return {"entry_point": "ss_scan_chunked with SS_FLAG_ZOH, same workload", "ms_per_step": round(ms, 4),
            "elem_per_s": elems / (ms * 1e-3), "gpu_launches": 3 * reps}


def bwd_counts(batch, dim, dstate, seqlen, in_bytes=2):
    """Algorithmic bytes and exponentials of one backward pass with a gate.
    bytes: u, delta, z read once (in_bytes each) and dy once (fp32); du, ddelta, dz written
    once (fp32); B, C read and dB, dC written once per batch row; A, D, delta_bias, dlast read
    and dA, dD, ddelta_bias, dh0 written once.
    exps: N decays per element (each needed by both the state and its adjoint), and one each
    for the step size, its derivative sigmoid(x) and the gate's sigmoid(z)."""
    elems = batch * dim * seqlen
    byts = elems * (3 * in_bytes + 4 + 3 * 4) + batch * dstate * seqlen * (2 * in_bytes + 2 * 4) \
        + dim * dstate * 4 * 2 + dim * 4 * 4 + batch * dim * dstate * 4 * 2
    exps = elems * (dstate + 3)
    return elems, byts, exps


def bench_bwd(ss, I, torch, p, pk, fwd_ms, reps=5):
    """ss_scan_bwd on the long-sequence workload: the gradients of sum(dy y) + sum(dlast h_last)
    for every input (both local passes in one kernel at 64-step chunks, the forward and the
    adjoint carry, main pass: four kernels and five memsets per call)."""
    ct = I.cotangents(seed=103, batch=p.batch, dim=p.dim, dstate=p.dstate, seqlen=p.seqlen, with_h0=False,
                      device="cuda", gen_device="cuda")
    ws = torch.empty((ss.bwd_workspace_bytes(p.batch, p.dim, p.dstate, p.seqlen, ss.BF16),), dtype=torch.uint8,
                     device="cuda")

    def call():
        return ss.scan_bwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, dy=ct.dy,
                           dlast=ct.dlast, workspace=ws)

    for _ in range(2):
        g = call()
    del g
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the same call with the zero-order-hold input weight
    zcall = lambda: ss.scan_bwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, dy=ct.dy,
                                dlast=ct.dlast, workspace=ws, zoh=True)
    zcall()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        zcall()
    e1.record()
    torch.cuda.synchronize()
    zoh_ms = e0.elapsed_time(e1) / reps
    elems, byts, exps = bwd_counts(p.batch, p.dim, p.dstate, p.seqlen)
    roof = roofline_terms(byts, exps, ms, pk)
    del ct, ws
    return {"workload": f"{WORKLOAD}: batch={p.batch}, D={p.dim}, N={p.dstate}, L={p.seqlen}, bf16 inputs, gate, "
                        "fp32 gradients",
            "entry_point": "ss_scan_bwd", "ms": round(ms, 4), "elem_per_s": elems / (ms * 1e-3),
            "algorithmic_bytes": byts, "exps": exps, "roofline": roof,
            "time_vs_forward_step": round(ms / fwd_ms, 2) if fwd_ms else None,
            "zoh_ms": round(zoh_ms, 4), "gpu_launches": 4 * (2 * reps + 1)}


def bench_conv(ss, torch, pk, batch=1, dim=5120, seqlen=65536, reps=20):
    """The short convolution in front of the scan (ss_causal_conv1d with SiLU) on the
    long-sequence shape, bf16 in and out: 2 x 2 B of traffic per element."""
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((batch, dim, seqlen), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.randn((dim, 4), generator=g, device="cuda") * 0.5
    b = torch.randn((dim,), generator=g, device="cuda") * 0.1
    out = torch.empty_like(x)
    for _ in range(3):
        ss.causal_conv1d(x, w, b, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ss.causal_conv1d(x, w, b, out=out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    byts = batch * dim * seqlen * 4 + dim * 5 * 4
    gbs = byts / (ms * 1e-3) / 1e9
    del x, out
    return {"workload": f"conv1d_silu: batch={batch}, D={dim}, L={seqlen}, width 4, bf16 in and out",
            "entry_point": "ss_causal_conv1d", "ms": round(ms, 4), "algorithmic_bytes": byts, "gbs": round(gbs, 1),
            "hbm_frac": round(gbs / pk["hbm_gbs"], 4), "gpu_launches": reps}


def bench_decode(ss, I, torch, pk, steps=1024, batch=256, dim=5120, dstate=16):
    """The recurrence face: 1024 sequential decode steps on a (256, 5120, 16) fp32 state,
    captured once in a CUDA graph and replayed."""
    s = I.decode_stream(batch=batch, dim=dim, dstate=dstate, steps=steps, device="cuda", gen_device="cuda")
    state = torch.zeros((batch, dim, dstate), dtype=torch.float32, device="cuda")
    y = torch.empty((batch, dim), dtype=torch.float32, device="cuda")

    def run_all():
        for t in range(steps):
            ss.state_update(state, s.u[t], s.delta[t], s.A, s.B[t], s.C[t], D=s.D, z=s.z[t], delta_bias=s.delta_bias,
                            y=y)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run_all()                                   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_all()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    state.zero_()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    per_step_bytes = batch * dim * (2 * dstate * 4 + 3 * 2 + 4) + batch * 2 * dstate * 2 + dim * (dstate + 2) * 4
    us = ms * 1e3 / steps
    gbs = per_step_bytes / (us * 1e-6) / 1e9
    del s
    return {"workload": f"decode_256x5120: batch={batch}, D={dim}, N={dstate}, {steps} sequential steps, bf16 "
                        "inputs drawn per step, fp32 state", "entry_point": "ss_state_update (CUDA-graph replay)",
            "us_per_step": round(us, 2), "algorithmic_bytes_per_step": per_step_bytes,
            "gbs": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm_gbs"], 4),
            "note": "the 83.9 MB state fits in the 126 MB L2, so steps can exceed the HBM roofline",
            "gpu_launches": steps}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the side measurements (decode, conv1d, ZOH step, single-pass layer)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sfu", action="store_true", help="skip the ex2 throughput leg (the SFU peak then falls back)")
    ap.add_argument("--dim", type=int, default=5120, help="channels (5120 = the workload; smaller only for profiling)")
    ap.add_argument("--seqlen", type=int, default=65536, help="steps (65536 = the workload; shorter only for profiling)")
    ap.add_argument("--bwd-only", action="store_true",
                    help="time only the backward pass (ss_scan_bwd), --steps calls after 2 warm-ups")
    ap.add_argument("--schedules-only", action="store_true",
                    help="time only ss_scan_fwd under its two schedules (medium workload, then the 130M layer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
