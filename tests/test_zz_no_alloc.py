"""gat_fused_layer_no_alloc: the fused layer for callers that cannot allocate
device memory (a framework owning all memory through its own pool, an
allocator callback, a spent allocation budget). Its plan and chunk states live
in the library's static device scratch; this checks, through the C ABI, that
two calls in a row both match the fp64 oracle and gat_fused_layer with an
allocated plan and workspace, and that a graph too large for the scratch is
refused up front.

Kept in its own file, collected last, so a failure here never hides the rest
of the suite; it passes alone in a fresh process as well as after the others.
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


def _case(n, seed, H, Dh, dtype, deg):
    d = W.make_fused(seed=seed, n=n, H=H, Dh=Dh, deg=deg, dtype=dtype)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    if dtype == "bf16":
        qkv = [t(d[x].view(np.int16)).view(torch.bfloat16) for x in ("q", "k", "v")]
    else:
        qkv = [t(d[x]) for x in ("q", "k", "v")]
    return d, t(d["row_ptr"]), t(d["col_idx"]), qkv


@pytest.mark.parametrize("H,Dh,dtype", [(8, 64, "bf16"), (4, 32, "f32")])
def test_no_alloc_matches_allocating_entry_point_twice(gat, H, Dh, dtype):
    deg = W.zipf_degrees(np.random.default_rng(120), 3000, dmax=2000)
    deg[[3, 9]] = [1500, 0]  # a row far above the heavy threshold, and an empty row
    d, rp, ci, (q, k, v) = _case(3000, 121, H, Dh, dtype, deg)
    plan = gat.Plan(rp)
    assert plan.info()["n_chunks"] > 0
    ref = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan)
    torch.cuda.synchronize()
    ref_h = ref.float().cpu().numpy().astype(np.float64)
    o, cond = oracle.fused_layer(d["row_ptr"], d["col_idx"], d["q"], d["k"], d["v"], H, Dh,
                                 d["scale"], want_cond=True)
    deg_n = np.diff(d["row_ptr"]).astype(np.float64)[:, None, None]
    for _ in range(2):  # the scratch keeps the previous call's contents
        out = torch.full_like(q, float("nan"))
        gat.gat_fused_layer_no_alloc(rp, ci, q, k, v, d["scale"], out)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        assert (got[9] == 0).all()
        for want, what in ((o, "oracle"), (ref_h, "gat_fused_layer")):
            if dtype == "bf16":
                assert_bf16(got, want, cond, name=f"no_alloc vs {what}")
            else:
                assert_fp32(got, want, cond, deg_n, name=f"no_alloc vs {what}")


def test_no_alloc_refuses_graphs_beyond_its_scratch(gat):
    # 20 rows of 100000 edges: 31260 chunk states of 2112 bytes > 32 MiB
    d, rp, ci, (q, k, v) = _case(20, 122, 8, 64, "bf16", np.full(20, 100000))
    out = torch.zeros_like(q)
    with pytest.raises(gat.GatError, match="GAT_ERR_WORKSPACE"):
        gat.gat_fused_layer_no_alloc(rp, ci, q, k, v, d["scale"], out)
    torch.cuda.synchronize()
    assert (out.float() == 0).all()  # refused before any layer work
