"""The benchmark's multi-rank host logic on CPU, as two gloo ranks: the
whole-job value is the work summed over ranks divided by the slowest rank's
time, each rank draws its own requests, and a rank that dies ends the other
rank's next collective with an error instead of a hang."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, ws: int, port: int, timeout_s: float = 60.0):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      PKV_DIST_TIMEOUT_S=str(timeout_s))


def _aggregate_worker(rank: int, ws: int, port: int, q):
    _env(rank, ws, port)
    import torch
    import torch.distributed as dist
    import bench
    got_ws, got_rank, _ = bench.dist_setup(ws)
    assert (got_ws, got_rank) == (ws, rank)
    # rank r: decode part 2 ms + r ms moving (r + 1) GB; prefill part 1 ms, 1e12 FLOP
    stats = [("decode", 2.0 + rank, 1e9 * (rank + 1), "GB/s"), ("prefill", 1.0, 1e12, "TFLOP/s")]
    bench.barrier(ws)
    out = bench.aggregate_parts(stats, ws, torch.device("cpu"), PEAKS)
    q.put((rank, out))
    dist.destroy_process_group()


def test_two_ranks_sum_work_over_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_aggregate_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res[0] == res[1]  # every rank computes the same whole-job numbers
    dec, pre = res[0]["decode"], res[0]["prefill"]
    assert dec["ms"] == 3.0                       # the slowest rank's time
    assert dec["work"] == int(3e9)                # 1 GB + 2 GB
    assert dec["value"] == pytest.approx(3e9 / 3e-3 / 1e9, rel=1e-6)  # 1000 GB/s
    assert dec["roofline_frac"] == pytest.approx(1000.0 / 6000.0 / 2, abs=1e-4)
    assert pre["value"] == pytest.approx(2e12 / 1e-3 / 1e12, rel=1e-6)  # 2000 TFLOP/s
    assert pre["roofline_frac"] == pytest.approx(0.5, abs=1e-4)


def test_ranks_draw_different_requests_of_the_same_shape():
    import bench
    from paged_kv_cache_316_gb300 import workloads as wl
    a = wl.llama_decode(seed=0 + bench.rank_seed(0))
    b = wl.llama_decode(seed=0 + bench.rank_seed(1))
    assert a.query.shape == b.query.shape and len(a.pt.lengths) == len(b.pt.lengths)
    assert a.pt.lengths != b.pt.lengths


def _dying_worker(rank: int, ws: int, port: int, q):
    _env(rank, ws, port, timeout_s=20.0)
    import torch
    import bench
    bench.dist_setup(ws)
    bench.barrier(ws)
    if rank == 1:
        os._exit(3)  # dies between steps, before the next collective
    try:
        bench.allreduce_max(1.0, ws, torch.device("cpu"))
        q.put((rank, "no error"))
    except Exception as e:  # noqa: BLE001 - any collective failure is the expected outcome
        q.put((rank, type(e).__name__))


def test_dead_rank_fails_the_next_collective():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_dying_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert procs[1].exitcode == 3
    rank, outcome = q.get()
    assert rank == 0 and outcome != "no error"
