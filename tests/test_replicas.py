"""The multi-replica path of bench.py (one process per GPU, no collective on
the data path): the job time is the slowest rank's and the job throughput is
the sum over replicas.  Runs as two gloo ranks on the CPU."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = bench.max_over_ranks(2.0 + rank, w, "cpu")  # rank 1 is the slower one
        # A parity failure on one rank stops every rank before the timing.
        agree = (bench.all_ranks_ok(True, w, "cpu"), bench.all_ranks_ok(rank == 0, w, "cpu"))
        q.put((r, w, local, ms, bench.job_tokens_per_s(w, 512, ms), agree))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_slowest_time_and_summed_throughput():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, local, ms, tps, agree) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert agree == (True, False)
        assert ms == pytest.approx(3.0)
        assert tps == pytest.approx(2 * 512 / 3.0e-3)


def test_single_process_defaults():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5


def test_step_stats():
    import bench
    st = bench.step_stats([float(v) for v in range(1, 101)])
    assert st["n"] == 100 and st["min"] == 1.0 and st["max"] == 100.0
    assert st["median"] == 50.5 and st["mean"] == 50.5
    assert st["p10"] == 11.0 and st["p90"] == 90.0
