"""GPU parity of the backward pass: the transposed (source-major) view bit for
bit against the oracle's stable counting sort, and the gradients of the fused
layer against the fp64 oracle's chain rule, element by element on graphs that
span several tiles, heavy rows and heavy sources, and on sampled rows and
sources of the 1e6-row power-law graph in the benchmark's configuration."""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def dev_feat(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return dev(a.view(np.int16)).view(torch.bfloat16)
    return dev(a)


def host(t):
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def host_i(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().astype(np.int64)


def graph(seed, n, n_src, deg, hot_share=0.0):
    """CSR with the given degrees, col_idx uniform over [0, n_src) unsorted;
    a share of the edges redirected to source 0 (a heavy source)."""
    rng = np.random.default_rng(seed)
    rp, ci = W.make_csr(rng, deg, n_src, sort_within_rows=False)
    if hot_share:
        ci[rng.random(ci.size) < hot_share] = 0
    return rp, ci


# ----------------------------------------------------------------------------
# transposed view
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("n,n_src,dmax,hot", [(300, 257, 40, 0.0), (1000, 50, 20, 0.3),
                                              (5, 1, 3, 0.0), (64, 4000, 2, 0.0)])
def test_transpose_bit_exact(gat, n, n_src, dmax, hot):
    rng = np.random.default_rng(n + n_src)
    deg = rng.integers(0, dmax + 1, n)
    rp, ci = graph(n, n, n_src, deg, hot)
    t = gat.Transpose(dev(rp), dev(ci), n_src)
    sp, perm, dst = (host_i(x) for x in t.export())
    osp, operm, odst = oracle.transpose(rp, ci, n_src)
    np.testing.assert_array_equal(sp, osp)
    np.testing.assert_array_equal(perm, operm)
    np.testing.assert_array_equal(dst, odst)
    inf = t.info()
    assert inf["max_src_degree"] == int(np.diff(osp).max(initial=0))
    assert (inf["n_heavy_src"] > 0) == (inf["max_src_degree"] > 128)


def test_transpose_empty_and_errors(gat):
    rp = np.zeros(4, np.int32)
    t = gat.Transpose(dev(rp), dev(np.zeros(0, np.int32)), 5)
    sp, perm, dst = t.export()
    assert (host_i(sp) == 0).all() and perm.numel() == 0
    rp = np.array([0, 2, 3], np.int32)
    with pytest.raises(gat.GatError, match="GAT_ERR_INDEX_OUT_OF_RANGE"):
        gat.Transpose(dev(rp), dev(np.array([0, 7, 1], np.int32)), 5)
    with pytest.raises(gat.GatError, match="GAT_ERR_INDEX_OUT_OF_RANGE"):
        gat.Transpose(dev(rp), dev(np.array([0, -1, 1], np.int32)), 5)


def test_transpose_power_law_full_size(gat):
    d = W.make_fused(seed=3, n=1_000_000, H=1, Dh=8, dtype="f32")
    t = gat.Transpose(dev(d["row_ptr"]), dev(d["col_idx"]), d["n_src"])
    sp, perm, dst = (host_i(x) for x in t.export())
    osp, operm, odst = oracle.transpose(d["row_ptr"], d["col_idx"], d["n_src"])
    np.testing.assert_array_equal(sp, osp)
    np.testing.assert_array_equal(perm, operm)
    np.testing.assert_array_equal(dst, odst)


# ----------------------------------------------------------------------------
# gradients
# ----------------------------------------------------------------------------
def check_grads(got, d, n_src, rp, ci, name, rows=None, srcs=None, want=None):
    dq, dk, dv = got
    o = want if want is not None else oracle.fused_backward(
        rp, ci, d["q"], d["k"], d["v"], d["dout"], d["H"], d["Dh"], d["scale"], n_src=n_src,
        want_cond=True)
    odq, odk, odv, cq, ck, cv = o
    deg = np.maximum(np.diff(rp.astype(np.int64)), 1).astype(np.float64)
    sdeg = np.maximum(np.bincount(ci, minlength=n_src), 1).astype(np.float64)
    r = slice(None) if rows is None else rows
    s = slice(None) if srcs is None else srcs
    if d["dtype"] == "bf16":
        assert_bf16(dq[r], odq[r], cq[r], name=f"{name} dq")
        assert_bf16(dk[s], odk[s], ck[s], name=f"{name} dk")
        assert_bf16(dv[s], odv[s], cv[s], name=f"{name} dv")
    else:
        assert_fp32(dq[r], odq[r], cq[r], deg[r][:, None, None], name=f"{name} dq")
        assert_fp32(dk[s], odk[s], ck[s], sdeg[s][:, None, None], name=f"{name} dk")
        assert_fp32(dv[s], odv[s], cv[s], sdeg[s][:, None, None], name=f"{name} dv")


def run_backward(gat, d, rp, ci, n_src, plan_kw=None):
    rpd, cid = dev(rp), dev(ci)
    q, k, v, g = (dev_feat(d[x]) for x in ("q", "k", "v", "dout"))
    plan = gat.Plan(rpd, **plan_kw) if plan_kw is not None else None
    t = gat.Transpose(rpd, cid, n_src)
    dq, dk, dv = gat.gat_fused_layer_backward(rpd, cid, q, k, v, g, d["scale"], t, plan=plan)
    return (host(dq), host(dk), host(dv)), t


def small_case(seed, n, n_src, H, Dh, dtype, deg, hot=0.0):
    rp, ci = graph(seed, n, n_src, deg, hot)
    rng = np.random.default_rng(seed + 1)
    f = lambda m: rng.standard_normal((m, H, Dh)).astype(np.float32)  # noqa: E731
    arrs = {"q": f(n), "k": f(n_src), "v": f(n_src), "dout": f(n)}
    if dtype == "bf16":
        arrs = {x: W.bf16_bits_from_f32(a) for x, a in arrs.items()}
    return dict(arrs, H=H, Dh=Dh, scale=1.0 / np.sqrt(Dh), dtype=dtype), rp, ci


@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "bf16"), (8, 64, "f32"), (4, 32, "f32"),
                                         (2, 16, "bf16"), (16, 16, "f32"), (8, 8, "bf16"),
                                         (3, 5, "f32"), (1, 6, "bf16"), (2, 4, "f32")])
def test_backward_shapes(gat, H, Dh, dtype):
    rng = np.random.default_rng(70 + H * Dh)
    deg = np.concatenate([rng.integers(0, 40, 400), [0, 129, 300, 1000, 64, 65]])
    d, rp, ci = small_case(71 + H, deg.size, 300, H, Dh, dtype, deg, hot=0.08)
    for plan_kw in (None, {"heavy_threshold": 100}):
        got, t = run_backward(gat, d, rp, ci, 300, plan_kw)
        check_grads(got, d, 300, rp, ci, f"{H}x{Dh} {dtype} plan={plan_kw is not None}")
    assert t.info()["n_heavy_src"] == 1  # source 0 collects ~8 % of the edges


def test_backward_power_law_100k_elementwise(gat):
    d = W.make_fused_backward(n=100_000)
    got, t = run_backward(gat, d, d["row_ptr"], d["col_idx"], d["n_src"], {})
    check_grads(got, d, d["n_src"], d["row_ptr"], d["col_idx"], "zipf 1e5 bf16")


def test_backward_deterministic(gat):
    d = W.make_fused_backward(n=20_000, seed=8)
    rpd, cid = dev(d["row_ptr"]), dev(d["col_idx"])
    q, k, v, g = (dev_feat(d[x]) for x in ("q", "k", "v", "dout"))
    plan, t = gat.Plan(rpd), gat.Transpose(rpd, cid, d["n_src"])
    a = gat.gat_fused_layer_backward(rpd, cid, q, k, v, g, d["scale"], t, plan=plan)
    b = gat.gat_fused_layer_backward(rpd, cid, q, k, v, g, d["scale"], t, plan=plan)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_errors(gat):
    d, rp, ci = small_case(80, 50, 40, 2, 8, "f32", np.full(50, 3))
    rpd, cid = dev(rp), dev(ci)
    q, k, v, g = (dev_feat(d[x]) for x in ("q", "k", "v", "dout"))
    t = gat.Transpose(rpd, cid, 40)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gat.GatError, match="GAT_ERR_WORKSPACE"):
        gat.gat_fused_layer_backward(rpd, cid, q, k, v, g, 0.5, t, workspace=small)
    other = gat.Transpose(rpd, cid, 41)
    with pytest.raises(gat.GatError, match="GAT_ERR_PLAN_MISMATCH"):
        gat.gat_fused_layer_backward(rpd, cid, q, k, v, g, 0.5, other)
    lib = gat.library()
    assert lib.gat_fused_layer_backward(None, None, 0, 0, 0, 1, 1, 0.5, None, None, None, None,
                                        0, None, None, None, None, None, None, 0, None) == 1


def _rows_covering(rp, ci, srcs):
    """Every row that has an edge reading one of srcs (so those sources'
    gradients are complete in the sub-graph of these rows)."""
    hit = np.isin(ci, srcs)
    r = np.repeat(np.arange(rp.size - 1), np.diff(rp.astype(np.int64)))
    return np.unique(r[hit])


def _sub_csr(rp, ci, rows):
    deg = (rp[rows + 1] - rp[rows]).astype(np.int64)
    srp = np.zeros(rows.size + 1, np.int64)
    srp[1:] = np.cumsum(deg)
    take = np.concatenate([np.arange(rp[r], rp[r + 1]) for r in rows])
    return srp.astype(np.int32), ci[take]


def test_backward_full_size_sampled(gat):
    d = W.make_fused_backward()
    rp, ci = d["row_ptr"], d["col_idx"]
    got, t = run_backward(gat, d, rp, ci, d["n_src"], {})
    dq, dk, dv = got
    assert all(np.isfinite(x).all() for x in got)
    rng = np.random.default_rng(12)
    deg = np.diff(rp)
    rows = np.unique(np.concatenate([np.argsort(deg)[-6:], rng.integers(0, deg.size, 150)]))
    srcs = np.unique(rng.integers(0, d["n_src"], 60))
    cover = np.unique(np.concatenate([rows, _rows_covering(rp, ci, srcs)]))
    srp, sci = _sub_csr(rp, ci, cover)
    sub = dict(d, q=d["q"][cover], dout=d["dout"][cover])
    want = oracle.fused_backward(srp, sci, sub["q"], d["k"], d["v"], sub["dout"], d["H"], d["Dh"],
                                 d["scale"], n_src=d["n_src"], want_cond=True)
    pos = np.searchsorted(cover, rows)
    odq, odk, odv, cq, ck, cv = want
    assert_bf16(dq[rows], odq[pos], cq[pos], name="1e6 dq sampled rows")
    assert_bf16(dk[srcs], odk[srcs], ck[srcs], name="1e6 dk sampled sources")
    assert_bf16(dv[srcs], odv[srcs], cv[srcs], name="1e6 dv sampled sources")


def test_backward_degenerate_graphs(gat):
    H, Dh = 8, 64
    rng = np.random.default_rng(81)
    f = lambda m: W.bf16_bits_from_f32(rng.standard_normal((m, H, Dh)).astype(np.float32))  # noqa: E731
    # no edges at all: dq = dk = dv = 0
    rp = np.zeros(6, np.int32)
    d = dict(q=f(5), k=f(4), v=f(4), dout=f(5), H=H, Dh=Dh, scale=0.125, dtype="bf16")
    rpd, cid = dev(rp), dev(np.zeros(0, np.int32))
    t = gat.Transpose(rpd, cid, 4)
    dq, dk, dv = gat.gat_fused_layer_backward(rpd, cid, *(dev_feat(d[x]) for x in ("q", "k", "v", "dout")),
                                              d["scale"], t, plan=gat.Plan(rpd, n_edges=0))
    assert all((host(x) == 0).all() for x in (dq, dk, dv))
    # every edge reads one source, one row holds them all (heavy row and heavy source)
    deg = np.array([0, 700, 0, 1], np.int64)
    rp = W.row_ptr_from_degrees(deg)
    ci = np.zeros(int(rp[-1]), np.int32)
    d = dict(q=f(4), k=f(3), v=f(3), dout=f(4), H=H, Dh=Dh, scale=0.125, dtype="bf16")
    got, t = run_backward(gat, d, rp, ci, 3, {})
    assert t.info()["n_heavy_src"] == 1
    check_grads(got, d, 3, rp, ci, "single source")
