"""GPU parity: every entry point of libgat against the fp64 oracle on the same
seeded inputs, through the C ABI (Python binding = argument marshalling).

Small cases span several tiles and ragged tails and are compared element by
element; the full-size workloads are compared on sampled outputs the oracle
computes one by one, in the launch configuration the benchmark times.
Integer outputs (the plan) are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_bf16, assert_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gat():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_graph_attention_head_gb300 as g
    return g


DEV = "cuda"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def dev_bf16(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host(t):
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


# ----------------------------------------------------------------------------
# edge softmax (multi-head CSR softmax workload)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("use_plan", [False, True])
def test_edge_softmax_workload(gat, use_plan):
    d = W.make_edge_softmax()  # 384 rows, degrees 0..36, H=4, scores N(0, 2^2)
    rp = dev(d["row_ptr"])
    s = dev(d["scores"])
    plan = gat.Plan(rp, heavy_threshold=20) if use_plan else None
    out = gat.gat_edge_softmax(rp, s, 4, plan=plan)
    o = oracle.edge_softmax(d["row_ptr"], d["scores"], 4)
    assert_fp32(host(out), o, name="edge_softmax")


@pytest.mark.parametrize("H", [1, 3, 4, 5, 8, 12, 32, 40, 64, 128])
def test_edge_softmax_heads_in_place_and_long_rows(gat, H):
    deg = np.array([0, 1, 2, 31, 32, 33, 300, 0, 5000, 7])
    d = W.make_edge_softmax(seed=40 + H, deg=deg, H=H)
    rp = dev(d["row_ptr"])
    s = dev(d["scores"])
    o = oracle.edge_softmax(d["row_ptr"], d["scores"], H)
    for plan in (None, gat.Plan(rp, heavy_threshold=40)):
        buf = s.clone()
        gat.gat_edge_softmax(rp, buf, H, out=buf, plan=plan)  # in place
        assert_fp32(host(buf), o, name=f"edge_softmax H={H}")


def test_edge_softmax_plan_reused_across_calls_and_head_counts(gat):
    """One plan serves consecutive launches: its work counters are reset by
    the last block of each launch. Every call writes into a NaN-filled
    buffer, so a batch or heavy row skipped by a stale counter would show."""
    deg = W.zipf_degrees(np.random.default_rng(21), 20_000, dmax=3000, mean=16.0)
    deg[[5, 6, 7]] = [2500, 1100, 300]  # heavy rows: two-pass, one-pass, just past a warp buffer
    rp_h = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    rp = dev(rp_h)
    plan = gat.Plan(rp)
    first = {}
    for H in (8, 4, 8, 16, 8):
        d = W.make_edge_softmax(seed=70 + H, deg=deg, H=H)
        s = dev(d["scores"])
        out = torch.full_like(s, float("nan"))
        gat.gat_edge_softmax(rp, s, H, out=out, plan=plan)
        g = host(out)
        if H not in first:
            first[H] = g
            assert_fp32(g, oracle.edge_softmax(d["row_ptr"], d["scores"], H),
                        name=f"edge_softmax plan reuse H={H}")
        else:  # deterministic: the same launch gives the same bits
            assert np.array_equal(g, first[H])


@pytest.mark.parametrize("H", [8, 4, 32, 64, 128])
def test_edge_softmax_neg_inf_heads_on_every_row_path(gat, H):
    """-inf scores on every row path of the 8-head kernel (thread tiers, the
    8-per-lane warp tier, the whole-warp shared-memory rows, rows streamed
    twice through a warp buffer, one-chunk and multi-chunk block rows; the
    warp-from-global rows without a plan): head 0 of every row all -inf (NaN,
    as the two-pass definition), head 1 -inf but for one edge (that edge 1,
    the rest 0), head 2 -inf on every other edge; scores ~ N(0, 30^2)."""
    deg = np.array([3, 8, 9, 100, 200, 300, 600, 1500, 3000, 0, 2, 40], np.int32)
    rng = np.random.default_rng(11 + H)
    rp_h = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    E = int(rp_h[-1])
    s_h = rng.normal(0.0, 30.0, size=(E, H)).astype(np.float32)
    for r in range(deg.size):
        e0, e1 = rp_h[r], rp_h[r + 1]
        if e1 == e0:
            continue
        s_h[e0:e1, 0] = -np.inf
        keep = e0 + (e1 - e0) // 2
        s_h[e0:e1, 1] = -np.inf
        s_h[keep, 1] = 5.0
        s_h[e0:e1:2, 2] = -np.inf
    o = oracle.edge_softmax(rp_h, s_h, H)
    rp = dev(rp_h)
    for plan in (None, gat.Plan(rp)):
        buf = dev(s_h)
        gat.gat_edge_softmax(rp, buf, H, out=buf, plan=plan)  # in place
        g = host(buf)
        assert_fp32(g, o, name=f"edge_softmax -inf heads H={H} plan={plan is not None}")
        for r in range(deg.size):
            e0, e1 = rp_h[r], rp_h[r + 1]
            if e1 > e0:
                assert np.isnan(g[e0:e1, 0]).all()
                assert abs(g[e0 + (e1 - e0) // 2, 1] - 1.0) <= 1e-6


@pytest.mark.parametrize("H", [8, 4])
def test_edge_softmax_heavy_ring_boundaries_and_many_heavy_rows(gat, H):
    """The heavy rows' chunk ring: 20,000 plan-heavy rows at H = 8 (more than
    32 list entries per block of the grid, so blocks take several 32-entry
    groups; 6,000 at H = 4) cycling through the ring's boundaries in chunks
    of 2048/H edges: one
    edge past a warp buffer, exactly 2 and 4 chunks (the largest row kept in
    its slots), 4 chunks + 1 (the first row read twice), and long rows; an
    all -inf head on some rows. Every element against the oracle."""
    ce = 2048 // H
    cyc = np.array([ce + 1, 2 * ce, 2 * ce + 1, 4 * ce, 4 * ce + 1, 9 * ce + 3, ce + 7, 3 * ce])
    deg = np.tile(cyc, 20000 // cyc.size + 1)[:20000].astype(np.int64)
    if H == 4:  # keep the edge count moderate at the wider chunks
        deg = deg[:6000]
    rng = np.random.default_rng(90 + H)
    rp_h = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    E = int(rp_h[-1])
    s_h = (2.0 * rng.standard_normal((E, H))).astype(np.float32)
    for r in range(0, deg.size, 997):
        s_h[rp_h[r]:rp_h[r + 1], 0] = -np.inf
    rp = dev(rp_h)
    plan = gat.Plan(rp)
    assert plan.info()["n_heavy"] == deg.size
    o = oracle.edge_softmax(rp_h, s_h, H)
    g = host(gat.gat_edge_softmax(rp, dev(s_h), H, plan=plan))
    nan_rows = np.zeros(E, dtype=bool)
    for r in range(0, deg.size, 997):
        nan_rows[rp_h[r]:rp_h[r + 1]] = True
    assert np.isnan(g[nan_rows, 0]).all()
    keep = np.ones(g.shape, dtype=bool)
    keep[nan_rows, 0] = False
    assert_fp32(g[keep], o[keep], name=f"edge_softmax heavy ring H={H}")


def test_edge_softmax_unaligned_buffers(gat):
    """Scores and output 4 bytes off a 16-byte boundary (H = 8): the 4-byte
    copy path, with and without a plan, against the oracle."""
    deg = np.array([5, 0, 300, 40, 2000, 7, 129, 1], np.int32)
    d = W.make_edge_softmax(seed=91, deg=deg, H=8)
    rp = dev(d["row_ptr"])
    o = oracle.edge_softmax(d["row_ptr"], d["scores"], 8)
    E = d["scores"].shape[0]
    for plan in (None, gat.Plan(rp)):
        sbuf = torch.empty(E * 8 + 1, device=DEV)
        obuf = torch.empty(E * 8 + 1, device=DEV)
        s = sbuf[1:].view(E, 8)
        s.copy_(dev(d["scores"]))
        out = obuf[1:].view(E, 8)
        assert s.data_ptr() % 16 != 0 and out.data_ptr() % 16 != 0
        gat.gat_edge_softmax(rp, s, 8, out=out, plan=plan)
        assert_fp32(host(out), o, name="edge_softmax unaligned")


def test_edge_softmax_extreme_scores_and_neg_inf_row(gat):
    rp_h = np.array([0, 3, 5, 8], np.int32)
    s_h = np.array([[80.0], [-80.0], [79.0], [-np.inf], [-np.inf], [3.0], [3.0], [3.0]],
                   np.float32)
    out = gat.gat_edge_softmax(dev(rp_h), dev(s_h), 1)
    o = oracle.edge_softmax(rp_h, s_h, 1)
    g = host(out)
    assert np.isnan(g[3:5]).all() and np.isnan(o[3:5]).all()  # all -inf row -> NaN
    assert_fp32(g[[0, 1, 2, 5, 6, 7]], o[[0, 1, 2, 5, 6, 7]])
    np.testing.assert_allclose(g[5:8, 0], 1 / 3, rtol=1e-6)


# ----------------------------------------------------------------------------
# softmax + aggregation workload (edge softmax H=1 then weighted SpMM)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("use_plan", [False, True])
def test_aggregate_workload(gat, use_plan):
    d = W.make_aggregate()  # 384 rows, degrees 0..36, col_idx unsorted, values [384,64]
    rp, ci = dev(d["row_ptr"]), dev(d["col_idx"])
    plan = gat.Plan(rp, heavy_threshold=24) if use_plan else None
    w = gat.gat_edge_softmax(rp, dev(d["scores"]).reshape(-1, 1), 1, plan=plan)
    out = gat.gat_spmm_weighted(rp, ci, w, dev(d["values"]).reshape(384, 1, 64), 1, 64,
                                plan=plan)
    w_o = oracle.edge_softmax(d["row_ptr"], d["scores"], 1)
    o, c = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], w_o, d["values"], 1, 64,
                                want_cond=True)
    n = np.diff(d["row_ptr"]).astype(np.float64)[:, None, None]
    g = host(out)
    assert (g[np.diff(d["row_ptr"]) == 0] == 0).all()  # zero-degree rows are exact zeros
    rate = assert_fp32(g, o, c, n, name="aggregate")
    assert rate > 0.99


@pytest.mark.parametrize("use_plan", [False, True])
def test_softmax_aggregate_workload_one_launch(gat, use_plan):
    """The same operation (softmax of given scores, then the weighted sum) in
    one pass: the 384-row workload against the oracle's softmax followed by
    its aggregation."""
    d = W.make_aggregate()
    rp, ci = dev(d["row_ptr"]), dev(d["col_idx"])
    plan = gat.Plan(rp, heavy_threshold=24, chunk_edges=8) if use_plan else None
    if use_plan:
        assert plan.info()["n_chunks"] > 0
    out = gat.gat_softmax_aggregate(rp, ci, dev(d["scores"]).reshape(-1, 1),
                                    dev(d["values"]).reshape(384, 1, 64), 1, 64, plan=plan)
    w_o = oracle.edge_softmax(d["row_ptr"], d["scores"], 1)
    o, c = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], w_o, d["values"], 1, 64,
                                want_cond=True)
    n = np.maximum(np.diff(d["row_ptr"]), 1).astype(np.float64)[:, None, None]
    g = host(out)
    assert (g[np.diff(d["row_ptr"]) == 0] == 0).all()
    rate = assert_fp32(g, o, c, n, name="aggregate one pass")
    assert rate > 0.99


@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "bf16"), (4, 32, "f32"), (12, 64, "bf16"),
                                         (1, 64, "f32"), (2, 8, "f32")])
def test_softmax_aggregate_heads_heavy_rows_masked_head(gat, H, Dh, dtype):
    """Multi-head one-pass softmax + aggregation on a power-law graph with a
    chunked heavy row, an empty row, and a row whose head 0 is all -inf (NaN
    there, as the softmax of the composition gives)."""
    rng = np.random.default_rng(80 + H * Dh)
    deg = W.zipf_degrees(rng, 3000, dmax=500)
    deg[[4, 9, 20]] = [2500, 0, 7]
    rp, ci = W.make_csr(rng, deg, 2000, sort_within_rows=False)
    E = int(rp[-1])
    sc = (2.0 * rng.standard_normal((E, H))).astype(np.float32)
    sc[rp[20]:rp[21], 0] = -np.inf
    f32 = rng.standard_normal((2000, H, Dh)).astype(np.float32)
    if dtype == "bf16":
        fb = W.bf16_bits_from_f32(f32)
        fd, fo = dev_bf16(fb), fb
    else:
        fd, fo = dev(f32), f32
    rpd = dev(rp)
    plan = gat.Plan(rpd)
    assert plan.info()["n_chunks"] > 0
    w_o = oracle.edge_softmax(rp, sc, H)
    o, c = oracle.spmm_weighted(rp, ci, w_o, fo, H, Dh, want_cond=True)
    assert np.isnan(o[20, 0]).all()
    keep = np.ones(o.shape, dtype=bool)
    keep[20, 0] = False
    for pl in (None, plan):
        g = host(gat.gat_softmax_aggregate(rpd, dev(ci), dev(sc), fd, H, Dh, plan=pl))
        assert np.isnan(g[20, 0]).all() and not np.isnan(g[keep]).any()
        assert (g[9] == 0).all()
        if dtype == "bf16":
            assert_bf16(g[keep], o[keep], c[keep], name=f"aggregate one pass {H}x{Dh} bf16")
        else:
            n = np.broadcast_to(np.maximum(deg, 1).astype(np.float64)[:, None, None], o.shape)
            assert_fp32(g[keep], o[keep], c[keep], n[keep], name=f"aggregate one pass {H}x{Dh}")


def test_softmax_aggregate_errors(gat):
    """Shapes outside the vector engine are refused (the two-launch
    composition covers them); a plan for another graph is refused."""
    rp = dev(np.array([0, 2, 3], np.int32))
    ci = dev(np.array([0, 1, 1], np.int32))
    sc = dev(np.zeros((3, 1), np.float32))
    with pytest.raises(gat.GatError, match="GAT_ERR_UNSUPPORTED"):
        gat.gat_softmax_aggregate(rp, ci, sc, dev(np.zeros((2, 1, 5), np.float32)), 1, 5)
    other = gat.Plan(dev(np.array([0, 1, 2, 3], np.int32)))
    with pytest.raises(gat.GatError, match="GAT_ERR_PLAN_MISMATCH"):
        gat.gat_softmax_aggregate(rp, ci, sc, dev(np.zeros((2, 1, 8), np.float32)), 1, 8,
                                  plan=other)


@pytest.mark.parametrize("H,Dh,dtype", [(1, 64, "f32"), (4, 32, "f32"), (8, 64, "f32"),
                                         (8, 64, "bf16"), (2, 64, "bf16"), (1, 32, "bf16"),
                                         (3, 24, "f32"), (5, 6, "bf16"),
                                         # head groups: 2 x 8, 3 x 4, 2 x 16 heads
                                         (16, 64, "f32"), (12, 32, "bf16"), (32, 32, "f32")])
def test_spmm_shapes(gat, H, Dh, dtype):
    rng = np.random.default_rng(50 + H * Dh)
    deg = np.concatenate([rng.integers(0, 40, 300), [0, 65, 64, 200, 1500]])
    n, n_src = deg.size, 257
    rp, ci = W.make_csr(rng, deg, n_src, sort_within_rows=False)
    E = int(rp[-1])
    w = rng.standard_normal((E, H)).astype(np.float32)
    f32 = rng.standard_normal((n_src, H, Dh)).astype(np.float32)
    if dtype == "bf16":
        bits = W.bf16_bits_from_f32(f32)
        feat_d, feat_o = dev_bf16(bits), bits
    else:
        feat_d, feat_o = dev(f32), f32
    o, c = oracle.spmm_weighted(rp, ci, w.astype(np.float64), feat_o, H, Dh, want_cond=True)
    rpd = dev(rp)
    for plan, no_ws in ((None, False), (gat.Plan(rpd, heavy_threshold=64), False),
                        (gat.Plan(rpd, heavy_threshold=64, chunk_edges=50), False),
                        (gat.Plan(rpd, heavy_threshold=64), True)):
        out = gat.gat_spmm_weighted(rpd, dev(ci), dev(w), feat_d, H, Dh, plan=plan,
                                    no_workspace=no_ws)
        g = host(out)
        if dtype == "bf16":
            assert_bf16(g, o, c, name=f"spmm {H}x{Dh} bf16")
        else:
            assert_fp32(g, o, c, deg.astype(np.float64)[:, None, None], name=f"spmm {H}x{Dh}")


# ----------------------------------------------------------------------------
# SDDMM workload (COO) and CSR / multi-head / bf16 forms
# ----------------------------------------------------------------------------
def test_sddmm_workload(gat):
    d = W.make_sddmm()  # src [1024,128], dst [768,128], 16384 edges
    out = gat.gat_sddmm(dev(d["src_idx"]), dev(d["src_feat"]), dev(d["dst_feat"]), 1, 128,
                        dst_idx=dev(d["dst_idx"]))
    o, c = oracle.sddmm(d["src_idx"], d["src_feat"], d["dst_feat"], 1, 128,
                        dst_idx=d["dst_idx"], want_cond=True)
    rate = assert_fp32(host(out), o, c, 128, name="sddmm")
    assert rate > 0.98


@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "bf16"), (4, 32, "f32"), (3, 5, "f32"),
                                         (2, 24, "bf16")])
def test_sddmm_csr_multihead(gat, H, Dh, dtype):
    rng = np.random.default_rng(60 + Dh)
    deg = np.concatenate([rng.integers(0, 30, 200), [0, 0, 300]])
    rp, ci = W.make_csr(rng, deg, 150, sort_within_rows=True)
    n = deg.size
    k32 = rng.standard_normal((150, H, Dh)).astype(np.float32)
    q32 = rng.standard_normal((n, H, Dh)).astype(np.float32)
    if dtype == "bf16":
        kb, qb = W.bf16_bits_from_f32(k32), W.bf16_bits_from_f32(q32)
        kd, qd, ko, qo = dev_bf16(kb), dev_bf16(qb), kb, qb
    else:
        kd, qd, ko, qo = dev(k32), dev(q32), k32, q32
    out = gat.gat_sddmm(dev(ci), kd, qd, H, Dh, scale=0.3, row_ptr=dev(rp))
    o, c = oracle.sddmm(ci, ko, qo, H, Dh, scale=0.3, row_ptr=rp, want_cond=True)
    assert_fp32(host(out), o, c, Dh, name="sddmm csr")


# ----------------------------------------------------------------------------
# degree-bucket plan: bit-exact against the oracle's definition
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("T,C", [(64, 64), (16, 32), (1, 1), (4095, 4096)])
def test_plan_bit_exact(gat, T, C):
    rng = np.random.default_rng(70)
    deg = np.concatenate([W.zipf_degrees(rng, 30000), [0, T, T + 1, C, C + 1, 2 * C, 9000],
                          np.zeros(5000, np.int64)])
    rp = W.row_ptr_from_degrees(deg)
    plan = gat.Plan(dev(rp), heavy_threshold=T, chunk_edges=C)
    hr, cs, cr = (host(t).astype(np.int64) for t in plan.export())
    ohr, ocs, ocr = oracle.plan(rp, T, C)
    np.testing.assert_array_equal(hr, ohr)
    np.testing.assert_array_equal(cs, ocs)
    np.testing.assert_array_equal(cr, ocr)


def test_plan_empty_and_all_light(gat):
    rp = np.zeros(11, np.int32)
    plan = gat.Plan(dev(rp), n_edges=0)
    assert plan.info()["n_heavy"] == 0 and plan.info()["n_chunks"] == 0
    rp = W.row_ptr_from_degrees(np.full(100, 3))
    plan = gat.Plan(dev(rp))
    assert plan.info()["n_heavy"] == 0


# ----------------------------------------------------------------------------
# fused layer
# ----------------------------------------------------------------------------
def fused_case(n, seed, H=8, Dh=64, dtype="bf16", deg=None, dmax=4096, mean=16.0):
    d = W.make_fused(seed=seed, n=n, H=H, Dh=Dh, deg=deg, dmax=dmax, mean=mean, dtype=dtype)
    if dtype == "bf16":
        qd, kd, vd = (dev_bf16(d[x]) for x in ("q", "k", "v"))
    else:
        qd, kd, vd = (dev(d[x]) for x in ("q", "k", "v"))
    return d, dev(d["row_ptr"]), dev(d["col_idx"]), qd, kd, vd


def check_fused(d, g, rows=None):
    o, c = oracle.fused_layer(d["row_ptr"], d["col_idx"], d["q"], d["k"], d["v"], d["H"],
                              d["Dh"], d["scale"], rows=rows, want_cond=True)
    if rows is not None:
        g = g[rows]
    if d["dtype"] == "bf16":
        return assert_bf16(g, o, c, name="fused bf16")
    deg = np.diff(d["row_ptr"]).astype(np.float64)
    n = deg if rows is None else deg[rows]
    return assert_fp32(g, o, c, n[:, None, None], name="fused fp32")


@pytest.mark.parametrize("use_plan", [False, True])
def test_fused_small_power_law(gat, use_plan):
    deg = W.zipf_degrees(np.random.default_rng(80), 6000, dmax=2000)
    deg[[5, 17]] = [0, 3000]
    d, rp, ci, q, k, v = fused_case(6000, 81, deg=deg)
    plan = gat.Plan(rp) if use_plan else None
    out = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
    g = host(out)
    assert (g[5] == 0).all()
    check_fused(d, g)


@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "f32"), (4, 64, "bf16"), (2, 64, "bf16"),
                                         (1, 64, "bf16"), (1, 32, "bf16"), (4, 32, "f32"),
                                         (1, 64, "f32"), (3, 24, "f32"), (2, 40, "bf16"),
                                         # head groups: 3 x 4, 2 x 8, 2 x 16, 3 x 2, 2 x 8 heads
                                         (12, 64, "bf16"), (16, 128, "bf16"), (32, 64, "bf16"),
                                         (6, 32, "f32"), (16, 64, "f32")])
def test_fused_shapes(gat, H, Dh, dtype):
    deg = W.zipf_degrees(np.random.default_rng(90 + Dh), 1500, dmax=700)
    d, rp, ci, q, k, v = fused_case(1500, 91 + H, H=H, Dh=Dh, dtype=dtype, deg=deg)
    for plan in (None, gat.Plan(rp, heavy_threshold=48, chunk_edges=40)):
        out = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
        check_fused(d, host(out))


def test_fused_edge_cases(gat):
    # E = 0: every row is zero-degree -> exact zeros
    d, rp, ci, q, k, v = fused_case(50, 100, deg=np.zeros(50, np.int64))
    out = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=gat.Plan(rp, n_edges=0))
    assert (host(out) == 0).all()
    # a single row
    d, rp, ci, q, k, v = fused_case(1, 101, deg=np.array([37]))
    check_fused(d, host(gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=gat.Plan(rp))))
    # one row of degree 100000 (split into ~1563 chunks) among light rows, and
    # degrees at the thresholds +-1
    deg = np.array([3, 100000, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1, 0])
    d, rp, ci, q, k, v = fused_case(deg.size, 102, deg=deg)
    plan = gat.Plan(rp)
    inf = plan.info()
    T, C = inf["heavy_threshold"], inf["chunk_edges"]
    assert inf["n_chunks"] == sum(-(-int(x) // C) for x in deg if x > T)
    assert inf["n_chunks"] > 100  # the 100000-edge row is split
    check_fused(d, host(gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)))


def test_fused_duplicates_unsorted_equal_scores(gat):
    rng = np.random.default_rng(103)
    deg = rng.integers(1, 90, 400)
    d, rp, ci, q, k, v = fused_case(400, 104, deg=deg)
    ci_h = rng.integers(0, 5, d["n_edges"]).astype(np.int32)  # many duplicates, unsorted
    d["col_idx"] = ci_h
    # rows whose queries are zero see equal scores everywhere -> plain averages
    d["q"][:50] = 0
    q = dev_bf16(d["q"])
    out = gat.gat_fused_layer(rp, dev(ci_h), q, k, v, d["scale"], plan=gat.Plan(rp))
    check_fused(d, host(out))


def test_fused_deterministic(gat):
    d, rp, ci, q, k, v = fused_case(20000, 105)
    plan = gat.Plan(rp)
    a = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
    b = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fused_errors(gat):
    d, rp, ci, q, k, v = fused_case(300, 106, deg=np.full(300, 700))
    plan = gat.Plan(rp)
    assert plan.info()["n_chunks"] > 0
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(gat.GatError, match="GAT_ERR_WORKSPACE"):
        gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan, workspace=small)
    other = gat.Plan(dev(W.row_ptr_from_degrees(np.full(10, 3))))
    with pytest.raises(gat.GatError, match="GAT_ERR_PLAN_MISMATCH"):
        gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=other)


def test_validate_graph(gat):
    rp = W.row_ptr_from_degrees(np.array([2, 0, 3]))
    ci = np.array([0, 1, 2, 2, 0], np.int32)
    gat.gat_validate_graph(dev(rp), dev(ci), 3)
    bad = ci.copy()
    bad[3] = 7
    with pytest.raises(gat.GatError, match="GAT_ERR_INDEX_OUT_OF_RANGE"):
        gat.gat_validate_graph(dev(rp), dev(bad), 3)
    bad_rp = rp.copy()
    bad_rp[2] = 1
    with pytest.raises(gat.GatError, match="GAT_ERR_INDEX_OUT_OF_RANGE"):
        gat.gat_validate_graph(dev(bad_rp), dev(ci), 3)


# ----------------------------------------------------------------------------
# full-size fused workload: 1e6 rows, Zipf(2.1) mean 16, H=8, Dh=64, bf16
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "bf16"), (4, 64, "f32"), (16, 64, "bf16"),
                                         (2, 32, "f32")])
def test_sddmm_csr_row_walk_every_edge(gat, H, Dh, dtype):
    """CSR SDDMM on a power-law graph with empty rows and one 3000-edge row,
    every (edge, head) compared: the edge spans of the warps cut rows anywhere."""
    rng = np.random.default_rng(70 + H)
    deg = W.zipf_degrees(rng, 4000, dmax=600)
    deg[[5, 6, 7, 100]] = [0, 0, 3000, 0]
    rp, ci = W.make_csr(rng, deg, 2500, sort_within_rows=True)
    n = deg.size
    k32 = rng.standard_normal((2500, H, Dh)).astype(np.float32)
    q32 = rng.standard_normal((n, H, Dh)).astype(np.float32)
    if dtype == "bf16":
        kb, qb = W.bf16_bits_from_f32(k32), W.bf16_bits_from_f32(q32)
        kd, qd, ko, qo = dev_bf16(kb), dev_bf16(qb), kb, qb
    else:
        kd, qd, ko, qo = dev(k32), dev(q32), k32, q32
    out = gat.gat_sddmm(dev(ci), kd, qd, H, Dh, scale=0.125, row_ptr=dev(rp))
    o, c = oracle.sddmm(ci, ko, qo, H, Dh, scale=0.125, row_ptr=rp, want_cond=True)
    assert_fp32(host(out), o, c, Dh, name=f"sddmm csr {H}x{Dh} {dtype}")


def test_row_shards_through_rebased_row_ptr(gat):
    """The row-sharded layer on one GPU: gat_partition_rows cuts a power-law
    graph (with a heavy row split into chunks) into 3 shards, each shard runs as
    a graph of its own (gat_rebase_row_ptr, its own plan, col_idx / q / out
    slices) and the stitched output matches the oracle; the rebased row
    pointers are bit-exact."""
    deg = W.zipf_degrees(np.random.default_rng(90), 5000, dmax=800)
    deg[[10, 2500]] = [3000, 0]
    d, rp, ci, q, k, v = fused_case(5000, 91, deg=deg)
    rb = gat.gat_partition_rows(d["row_ptr"], 3)
    out = torch.empty_like(q)
    for p in range(3):
        r0, r1 = int(rb[p]), int(rb[p + 1])
        e0, e1 = int(d["row_ptr"][r0]), int(d["row_ptr"][r1])
        lrp = gat.gat_rebase_row_ptr(rp, r0, r1)
        np.testing.assert_array_equal(host(lrp).astype(np.int64),
                                      d["row_ptr"][r0:r1 + 1] - d["row_ptr"][r0])
        plan = gat.Plan(lrp)
        gat.gat_fused_layer(lrp, ci[e0:e1], q[r0:r1], k, v, d["scale"], out=out[r0:r1],
                            plan=plan)
    check_fused(d, host(out))


@pytest.fixture(scope="module")
def full_fused(gat):
    d, rp, ci, q, k, v = fused_case(1_000_000, 3)
    plan = gat.Plan(rp)
    return d, rp, ci, q, k, v, plan


def test_full_size_plan_bit_exact(gat, full_fused):
    d, rp, ci, q, k, v, plan = full_fused
    inf = plan.info()
    hr, cs, cr = (host(t).astype(np.int64) for t in plan.export())
    ohr, ocs, ocr = oracle.plan(d["row_ptr"], inf["heavy_threshold"], inf["chunk_edges"])
    np.testing.assert_array_equal(hr, ohr)
    np.testing.assert_array_equal(cs, ocs)
    np.testing.assert_array_equal(cr, ocr)


def test_full_size_sddmm_csr_sampled_edges(gat, full_fused):
    """The CSR SDDMM of the benchmark's sddmm_csr workload (the fused workload's
    graph and q, k: 1e6 rows, H=8, Dh=64, bf16, scale 1/8): the edges of the
    heaviest rows, of rows around zero-degree... every degree class, and random
    edges against the oracle (COO form of the same edges)."""
    d, rp, ci, q, k, v, _ = full_fused
    out = host(gat.gat_sddmm(ci, k, q, d["H"], d["Dh"], scale=d["scale"], row_ptr=rp))
    deg = np.diff(d["row_ptr"])
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.argsort(deg)[-6:], rng.integers(0, deg.size, 400),
                                     [0, deg.size - 1]]))
    edges = np.concatenate([np.arange(d["row_ptr"][r], d["row_ptr"][r + 1]) for r in rows])
    edges = np.unique(np.concatenate([edges, rng.integers(0, d["n_edges"], 20000)]))
    dst = np.searchsorted(d["row_ptr"], edges, side="right") - 1
    o, c = oracle.sddmm(d["col_idx"][edges], d["k"], d["q"], d["H"], d["Dh"], scale=d["scale"],
                        dst_idx=dst, want_cond=True)
    assert_fp32(out[edges], o, c, d["Dh"], name="sddmm csr 1e6 rows")
    assert np.isfinite(out).all()


def test_full_size_fused_sampled_rows(gat, full_fused):
    d, rp, ci, q, k, v, plan = full_fused
    out = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
    g = host(out)
    deg = np.diff(d["row_ptr"])
    rng = np.random.default_rng(7)
    heaviest = np.argsort(deg)[-12:]
    # rows at the plan's class edges: the light / heavy cut (degree T vs T + 1)
    # and one or two whole chunks (degree C, C + 1, 2C, 2C + 1)
    inf = plan.info()
    T, C = inf["heavy_threshold"], inf["chunk_edges"]
    # (the rescaled Zipf degrees skip some integers: take two rows of every
    # degree present within 4 of each cut, and require rows on both sides)
    edges = []
    for cut in (T, C, 2 * C):
        for dv in range(cut - 3, cut + 5):
            edges.append(np.flatnonzero(deg == dv)[:2])
        near = deg[np.concatenate(edges)] if edges else deg[:0]
        assert (near <= cut).any() and (near > cut).any(), f"no rows on both sides of {cut}"
    rows = np.unique(np.concatenate([heaviest, *edges, rng.integers(0, deg.size, 300),
                                     [0, deg.size - 1]]))
    check_fused(d, g, rows=rows)
    assert np.isfinite(g).all()


# ----------------------------------------------------------------------------
# multi-head weighted aggregation at head_dim 32 (8 heads, fp32) and the
# 8-head softmax, on power-law graphs with the default plan (the launch
# configuration the benchmark times)
# ----------------------------------------------------------------------------
def _sub_csr(row_ptr, col_idx, w, rows):
    """The CSR of the selected rows alone (slicing only, no arithmetic)."""
    deg = (row_ptr[rows + 1] - row_ptr[rows]).astype(np.int64)
    rp = np.zeros(rows.size + 1, dtype=np.int64)
    rp[1:] = np.cumsum(deg)
    take = np.concatenate([np.arange(row_ptr[r], row_ptr[r + 1]) for r in rows]) \
        if rp[-1] else np.zeros(0, dtype=np.int64)
    return rp.astype(np.int32), col_idx[take], w[take], deg


def test_spmm_heads_100k_elementwise(gat):
    d = W.make_spmm_heads(n=100_000)
    H, Dh = d["H"], d["Dh"]
    rp = dev(d["row_ptr"])
    plan = gat.Plan(rp)
    assert plan.info()["n_heavy"] > 0
    out = gat.gat_spmm_weighted(rp, dev(d["col_idx"]), dev(d["w"]), dev(d["feat"]), H, Dh,
                                plan=plan)
    o, c = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], d["w"].astype(np.float64),
                                d["feat"], H, Dh, want_cond=True)
    deg = np.diff(d["row_ptr"]).astype(np.float64)
    rate = assert_fp32(host(out), o, c, deg[:, None, None], name="spmm 8x32 100k")
    assert rate > 0.99


def test_spmm_heads_chunked_equals_block_path_and_is_deterministic(gat):
    d = W.make_spmm_heads(n=50_000, seed=9)
    H, Dh = d["H"], d["Dh"]
    rp, ci, w, f = dev(d["row_ptr"]), dev(d["col_idx"]), dev(d["w"]), dev(d["feat"])
    plan = gat.Plan(rp)
    assert plan.info()["n_chunks"] > 0
    a = gat.gat_spmm_weighted(rp, ci, w, f, H, Dh, plan=plan)
    b = gat.gat_spmm_weighted(rp, ci, w, f, H, Dh, plan=plan)
    assert torch.equal(a, b)
    c = gat.gat_spmm_weighted(rp, ci, w, f, H, Dh, plan=plan, no_workspace=True)
    o, cond = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], d["w"].astype(np.float64),
                                   d["feat"], H, Dh, want_cond=True)
    deg = np.maximum(np.diff(d["row_ptr"]), 1).astype(np.float64)[:, None, None]
    assert_fp32(host(a), o, cond, deg, name="spmm chunked")
    assert_fp32(host(c), o, cond, deg, name="spmm block per heavy row")
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(gat.GatError, match="GAT_ERR_WORKSPACE"):
        gat.gat_spmm_weighted(rp, ci, w, f, H, Dh, plan=plan, workspace=small)


def test_spmm_heads_full_size_sampled_rows(gat):
    d = W.make_spmm_heads()
    H, Dh = d["H"], d["Dh"]
    rp = dev(d["row_ptr"])
    out = gat.gat_spmm_weighted(rp, dev(d["col_idx"]), dev(d["w"]), dev(d["feat"]), H, Dh,
                                plan=gat.Plan(rp))
    g = host(out)
    deg = np.diff(d["row_ptr"])
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.argsort(deg)[-12:], rng.integers(0, deg.size, 400),
                                     [0, deg.size - 1]]))
    srp, sci, sw, sdeg = _sub_csr(d["row_ptr"], d["col_idx"], d["w"], rows)
    o, c = oracle.spmm_weighted(srp, sci, sw.astype(np.float64), d["feat"], H, Dh,
                                want_cond=True)
    assert_fp32(g[rows], o, c, np.maximum(sdeg, 1).astype(np.float64)[:, None, None],
                name="spmm 8x32 1e6 sampled")
    assert np.isfinite(g).all()


def test_edge_softmax_8_heads_power_law_full_size(gat):
    deg = W.zipf_degrees(np.random.default_rng(3), 1_000_000)
    d = W.make_edge_softmax(seed=6, deg=deg, H=8)
    rp = dev(d["row_ptr"])
    out = gat.gat_edge_softmax(rp, dev(d["scores"]), 8, plan=gat.Plan(rp))
    o = oracle.edge_softmax(d["row_ptr"], d["scores"], 8)
    assert_fp32(host(out), o, name="edge_softmax 8 heads 1e6")
