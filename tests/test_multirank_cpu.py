"""The multi-process path of bench.py on CPU (gloo, world size 2): process-group
set-up from the launcher's environment, the barrier, and the max-over-ranks
reduction that turns per-rank times into the job's time.  The attention path
itself needs no exchange between ranks: each rank runs an independent
replica (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    r, w, local = bench.dist_setup()
    bench.barrier(w)
    t = bench.reduce_max(1.5 + r, w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, local, t))


def test_two_rank_max_reduction_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[3] == pytest.approx(2.5) for g in got)  # every rank sees the slowest rank's time
