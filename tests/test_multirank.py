"""The benchmark's multi-rank host logic (rank discovery, barrier, max-over-
ranks timing, independent per-rank problems) on two CPU processes over gloo."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.dist_barrier(dist)
    # each rank reports its own step time; every rank must see the maximum
    t = bench.dist_max(dist, 10.0 + 5.0 * r)
    # weak scaling: whole-job value counts every rank's (identical-size) problem
    import workloads as W
    d = W.make_fused(seed=3, n=500, dmax=64)
    value = w * d["n_edges"] * d["H"] / (t * 1e-3)
    q.put((r, w, local, t, value, d["n_edges"]))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_gloo_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 and x[0] == x[2] for x in res)
    assert all(x[3] == 15.0 for x in res)          # max over ranks on every rank
    assert res[0][4] == res[1][4]                    # same whole-job value
    assert res[0][5] == res[1][5]                    # same per-rank problem size


def test_single_rank_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    r, w, _ = bench.dist_env()
    assert w == 1
    assert bench.dist_init(1, "gloo") is None
    assert bench.dist_max(None, 3.5) == 3.5
