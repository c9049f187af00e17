"""Multi-rank host logic of bench.py on CPU: two gloo ranks, barrier and max over ranks."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    bench.barrier(w)
    out[r] = bench.barrier_and_max(10.0 + r * 5.0, w)
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    assert bench.barrier_and_max(3.5, 1) == 3.5


def test_roofline_model_counts():
    elems, byts, exps = bench.workload_counts(1, 5120, 16, 65536)
    assert elems == 335544320
    assert exps == elems * 18
    # 10 bytes per element plus B, C, A, D, bias and the final state
    assert byts == elems * 10 + 2 * 16 * 65536 * 2 + 5120 * 16 * 4 + 2 * 5120 * 4 + 5120 * 16 * 4
    pk = {"hbm_gbs": 6471.4, "sfu_texps": 148 * 32 * 2032e6 / 1e12, "hbm_src": "measured"}
    r = bench.roofline_terms(byts, exps, 1.0, pk)
    assert r["bound"] == "alu" and abs(r["achieved"] - exps / 1e-3 / 1e12) < 1e-3
