"""The N > 1 host path of bench.py on CPU: two gloo ranks (world_size 2) run
the replica set-up, the barrier and the max-over-ranks reduction that turn
per-rank step times into the whole-job number.  No GPU is touched."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each replica reports its own step time; the job takes the slowest
    got = bench.reduce_max(1.5 + rank, w)
    results[rank] = got
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_reduce_to_the_max_time():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        assert codes == [0, 0], codes
        assert dict(results) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.reduce_max(3.25, 1) == 3.25
