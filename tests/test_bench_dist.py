"""Host logic of the multi-GPU benchmark (replicas), run as two gloo ranks on CPU.

Each rank of `bench.py --gpus N` runs the whole workload on its own GPU; the
only cross-rank steps are barriers and the max over ranks of the timed
duration, from which rank 0 reports all ranks' work / the slowest rank's time.
These tests run exactly those steps with world_size 2 over gloo, no GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    r, local, w, dist = bench.dist_setup()
    assert (r, local, w) == (rank, rank, world) and dist is not None
    bench.barrier(dist)
    ms = [2.0, 3.5][rank]                       # rank 1 is the slower replica
    slowest = bench.max_over_ranks(dist, ms)
    value = bench.job_throughput(1.0e12, w, slowest)
    # the reference arm: rank 0 alone runs it; the others return without work
    ran = None
    if rank != 0:
        import time
        t = time.perf_counter()
        bench.run_reference(None, rank, w, dist)
        ran = time.perf_counter() - t
    bench.barrier(dist)
    out.put((rank, slowest, value, ran))
    dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks_and_value_aggregates_all_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ran in res:
        assert slowest == 3.5                   # both ranks see the slowest rank's time
        # 2 ranks x 1e12 FLOP in 3.5 ms = 571.43 TFLOP/s
        assert value == pytest.approx(2 * 1.0e12 / 3.5e-3 / 1e12)
    assert res[1][3] is not None and res[1][3] < 1.0   # non-zero rank: no reference work


def test_single_rank_has_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_setup() == (0, 0, 1, None)
    assert bench.max_over_ranks(None, 1.25) == 1.25
    assert bench.job_throughput(5.0e12, 1, 1000.0) == pytest.approx(5.0)
