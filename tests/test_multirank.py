"""The N > 1 benchmark path runs independent replicas (one per GPU) whose only
shared steps are a barrier and a max-reduction of the timed region over ranks.
That host logic is exercised here with the gloo backend, world size 2, on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), W4A16_BENCH_BACKEND="gloo")
    import bench
    r, local, w, pg = bench.dist_setup()
    assert (r, w) == (rank, world) and pg is not None
    # each rank "times" a different duration; every rank must see the maximum
    ms = 10.0 + 5.0 * rank
    bench.barrier(pg)
    m = bench.reduce_max(pg, ms, torch.device("cpu"))
    # whole-job value: all ranks' bytes over the slowest rank's time
    bytes_per_step, steps = 8_929_280, 200
    value = w * bytes_per_step * steps / (m * 1e-3) / 1e9
    q.put((rank, m, value))
    dist.destroy_process_group()


def test_replicas_max_reduce_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[1] for g in got] == [15.0, 15.0]
    expect = world * 8_929_280 * 200 / 15e-3 / 1e9
    assert all(abs(g[2] - expect) < 1e-9 for g in got)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    r, local, w, pg = bench.dist_setup()
    assert (r, local, w, pg) == (0, 0, 1, None)
    assert bench.reduce_max(None, 3.0, None) == 3.0
