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


def _shard_worker(rank, world, port, q):
    """One rank of the row-sharded layer on CPU: its rows of the partition,
    k / v all-gathered from node shards over gloo, the oracle on its own rows
    (the shard as a graph of its own); rank 0 stitches every rank's rows."""
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch
    import torch.distributed as dist
    import bench
    import oracle
    import workloads as W
    import sparse_graph_attention_head_gb300 as gat
    dist.init_process_group("gloo")
    d = W.make_fused(seed=5, n=900, dmax=300, dtype="f32", H=2, Dh=16)
    rpn = d["row_ptr"]
    rb = gat.gat_partition_rows(rpn, world)
    r0, r1, e0, e1 = bench.shard_bounds(rb, rpn, rank)
    a, b, per = bench.node_shard(d["n_rows"], world, rank)
    full = []
    for x in ("k", "v"):
        pad = torch.zeros((per,) + d[x].shape[1:], dtype=torch.float32)
        pad[: b - a] = torch.from_numpy(d[x][a:b])
        parts = [torch.empty_like(pad) for _ in range(world)]
        dist.all_gather(parts, pad)
        full.append(torch.cat(parts)[: d["n_rows"]].numpy())
    local_rp = (rpn[r0:r1 + 1] - rpn[r0]).astype(np.int32)
    out = oracle.fused_layer(local_rp, d["col_idx"][e0:e1], d["q"][r0:r1], full[0], full[1],
                             d["H"], d["Dh"], d["scale"])
    gathered = [None] * world
    dist.all_gather_object(gathered, (r0, r1, out))
    if rank == 0:
        ref = oracle.fused_layer(rpn, d["col_idx"], d["q"], d["k"], d["v"], d["H"], d["Dh"],
                                 d["scale"])
        stitched = np.concatenate([o for (_, _, o) in sorted(gathered, key=lambda t: t[0])])
        q.put((np.array_equal(stitched, ref), [(g0, g1) for (g0, g1, _) in gathered],
               bool(np.array_equal(full[0], d["k"]) and np.array_equal(full[1], d["v"]))))
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_rank_row_shards_stitch_to_the_full_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    equal, ranges, kv_ok = q.get(timeout=150)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert kv_ok                      # the all-gather rebuilt the full k and v
    assert equal                      # rows are independent: shards stitch bit for bit
    assert sorted(ranges)[0][0] == 0 and sorted(ranges)[-1][1] == 900
    assert sorted(ranges)[0][1] == sorted(ranges)[1][0]


def test_partition_rows_tiles_and_balances():
    import numpy as np
    import workloads as W
    import sparse_graph_attention_head_gb300 as gat
    rng = np.random.default_rng(4)
    for n, parts in ((1, 1), (1, 4), (10, 3), (5000, 7), (20000, 8)):
        deg = W.zipf_degrees(rng, n, dmax=2000)
        if n > 10:
            deg[rng.integers(0, n, 5)] = 0
        rp = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
        rb = gat.gat_partition_rows(rp, parts)
        assert rb.shape == (parts + 1,) and rb[0] == 0 and rb[-1] == n
        assert (np.diff(rb) >= 0).all()
        wgt = np.arange(n + 1) + rp                     # prefix weight: rows + edges
        per = np.diff(wgt[rb])
        # each part is within one row's weight of the ideal share
        assert per.max() - wgt[-1] / parts <= (1 + deg.max()), (per, wgt[-1] / parts)
    with pytest.raises(gat.GatError):
        gat.gat_partition_rows(np.array([0, 5, 3], dtype=np.int32), 2)
