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
    # every timed window is taken at its slowest rank
    wins = bench.reduce_max_windows([1.0 + rank, 3.0 - rank, 2.0], w)
    results[rank] = (got, wins)
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
        assert dict(results) == {0: (2.5, [2.0, 3.0, 2.0]), 1: (2.5, [2.0, 3.0, 2.0])}


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.reduce_max(3.25, 1) == 3.25


def test_rotation_copies_continue_across_windows():
    import bench
    # 20 steps x 8 launches: 16 copies divide the window, so windows run back to back
    assert bench.rotation_copies(12, 160) == (16, False)
    assert bench.rotation_copies(12, 24) == (12, False)
    # no divisor in [r_min, 4 r_min]: the L2 is flushed between windows instead
    assert bench.rotation_copies(12, 8) == (12, True)
    assert bench.rotation_copies(12, 97) == (12, True)


def test_both_arms_report_the_same_config():
    import bench
    for world in (1, 2, 8):
        cfg = bench.workload_config(world)
        assert cfg["M"] == [1, 2, 4, 8, 16, 32, 48, 64] and cfg["parallelism"] == f"replicas x{world}"
        assert set(cfg) == {"workload", "N", "K", "M", "out", "parallelism"}
