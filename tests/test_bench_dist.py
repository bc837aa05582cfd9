"""The benchmark's multi-rank logic on CPU: world_size 2 over gloo (127.0.0.1).

Each rank runs an independent replica (no data-path collective); the timed region is the
slowest rank's and the work is summed over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        ms, units = bench.reduce_over_ranks(dist, 10.0 + 5.0 * rank, 100.0 * (rank + 1))
        dist.barrier()
        q.put((r, ws, local, ms, units))
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, ws, local, ms, units) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert ms == 15.0          # the slowest rank's time
        assert units == 300.0      # the work of both replicas


def test_single_process_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_over_ranks(None, 3.0, 7.0) == (3.0, 7.0)
    cfg = bench.decode_config(bench.synth_workload(), 2)
    assert cfg["batch_rows"] == 64 and cfg["v_heads"] == 48 and "x2" in cfg["parallelism"]
