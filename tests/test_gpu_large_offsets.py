"""Feature tables past 2^31 elements and 2^32 bytes: 4.4 M source rows of
8 heads x 64 bf16 (2.25e9 elements, 4.5 GB per table; the E4M3 code tables
2.25 GB). Edges read sources spread over the whole table and clustered at
its top, so the gather offsets of the fused layer, the CSR SDDMM, the
weighted SpMM, the fp8 layer (and the quantiser's rows) and the backward
(and the dk / dv rows it writes) reach past what 32-bit element or byte
offsets can address.

Only the rows the edges read hold data (host-generated, seeded); the oracle
sees the same rows under a compact renumbering of the sources, so its
inputs are the generator's and its result is compared element by element.
Sources no edge reads must get exactly zero gradient."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_bf16, assert_fp32

pytestmark = pytest.mark.gpu

N_SRC = 4_400_000
H, DH = 8, 64
SCALE = 0.125


@pytest.fixture(scope="module")
def gat():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_graph_attention_head_gb300 as g
    return g


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def dev_bf16(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host(t):
    torch.cuda.synchronize()
    return t.float().cpu().numpy().astype(np.float64)


@pytest.fixture(scope="module")
def big():
    """A 3,000-row graph (Zipf degrees with two heavy rows) over 4.4 M
    sources: half the edges uniform over all sources, half among the top
    300,000 (element offsets past 2^31)."""
    rng = np.random.default_rng(2024)
    n = 3000
    deg = W.zipf_degrees(rng, n, dmax=600)
    deg[[7, 1500]] = [1500, 400]
    rp = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    E = int(rp[-1])
    ci = np.where(rng.random(E) < 0.5, rng.integers(0, N_SRC, E),
                  rng.integers(N_SRC - 300_000, N_SRC, E)).astype(np.int32)
    assert int(ci.max()) * H * DH > 2**31
    touched, compact = np.unique(ci, return_inverse=True)
    compact = compact.astype(np.int32)
    nt = touched.size

    def bf(shape):
        return W.bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32))

    q, dout = bf((n, H, DH)), bf((n, H, DH))
    kc, vc = bf((nt, H, DH)), bf((nt, H, DH))
    return dict(rp=rp, ci=ci, compact=compact, touched=touched, q=q, dout=dout, kc=kc, vc=vc)


def full_table(rows_bits, touched):
    """A [N_SRC, H, DH] bf16 table on the device: the given rows at their
    source ids, zeros elsewhere."""
    t = torch.zeros((N_SRC, H, DH), dtype=torch.bfloat16, device="cuda")
    t[torch.from_numpy(touched.astype(np.int64)).cuda()] = dev_bf16(rows_bits)
    return t


def test_forward_ops_past_32bit_offsets(gat, big):
    rpd, cid = dev(big["rp"]), dev(big["ci"])
    k = full_table(big["kc"], big["touched"])
    v = full_table(big["vc"], big["touched"])
    plan = gat.Plan(rpd)
    assert plan.info()["n_chunks"] > 0
    out = host(gat.gat_fused_layer(rpd, cid, dev_bf16(big["q"]), k, v, SCALE, plan=plan))
    o, c = oracle.fused_layer(big["rp"], big["compact"], big["q"], big["kc"], big["vc"], H, DH,
                              SCALE, want_cond=True)
    assert_bf16(out, o, c, name="fused layer, 4.4M-source tables")
    # weighted SpMM over the same gathers (fp32 weights [E, H])
    E = big["ci"].size
    w = np.random.default_rng(5).standard_normal((E, H)).astype(np.float32)
    g = host(gat.gat_spmm_weighted(rpd, cid, dev(w), v, H, DH, plan=plan))
    os_, cs = oracle.spmm_weighted(big["rp"], big["compact"], w, big["vc"], H, DH, want_cond=True)
    assert_bf16(g, os_, cs, name="spmm, 4.4M-source tables")
    # CSR SDDMM: per-edge scores from the same k rows
    sc = host(gat.gat_sddmm(cid, k, dev_bf16(big["q"]), H, DH, scale=SCALE, row_ptr=rpd))
    osd, csd = oracle.sddmm(big["compact"], big["kc"], big["q"], H, DH, scale=SCALE,
                            row_ptr=big["rp"], want_cond=True)
    assert_fp32(sc, osd, csd, DH, name="sddmm csr, 4.4M-source tables")
    # E4M3 tables quantised on the device (codes of the rows read: bit for bit
    # the oracle's), then the fp8 layer over them
    k8, ks = gat.gat_quantize_fp8(k)
    v8, vs = gat.gat_quantize_fp8(v)
    del k, v
    torch.cuda.empty_cache()
    hk8, hks = oracle.fp8_quantize(big["kc"], H, DH)
    hv8, hvs = oracle.fp8_quantize(big["vc"], H, DH)
    tt = torch.from_numpy(big["touched"].astype(np.int64)).cuda()
    np.testing.assert_array_equal(k8[tt].cpu().numpy(), hk8)
    np.testing.assert_array_equal(vs[tt].cpu().numpy(), hvs)
    o8 = host(gat.gat_fused_layer_fp8(rpd, cid, dev_bf16(big["q"]), k8, ks, v8, vs, SCALE,
                                      plan=plan))
    oo8, co8 = oracle.fused_layer_fp8(big["rp"], big["compact"], big["q"], hk8, hks, hv8, hvs,
                                      H, DH, SCALE, want_cond=True)
    assert_bf16(o8, oo8, co8, name="fp8 layer, 4.4M-source tables")
    del k8, v8, ks, vs
    torch.cuda.empty_cache()


def test_backward_past_32bit_offsets(gat, big):
    rpd, cid = dev(big["rp"]), dev(big["ci"])
    k = full_table(big["kc"], big["touched"])
    v = full_table(big["vc"], big["touched"])
    q, dout = dev_bf16(big["q"]), dev_bf16(big["dout"])
    plan = gat.Plan(rpd)
    tr = gat.Transpose(rpd, cid, N_SRC)
    dq, dk, dv = gat.gat_fused_layer_backward(rpd, cid, q, k, v, dout, SCALE, tr, plan=plan)
    torch.cuda.synchronize()
    tt = torch.from_numpy(big["touched"].astype(np.int64)).cuda()
    dk_t, dv_t = host(dk[tt]), host(dv[tt])
    odq, odk, odv, cdq, cdk, cdv = oracle.fused_backward(
        big["rp"], big["compact"], big["q"], big["kc"], big["vc"], big["dout"], H, DH, SCALE,
        n_src=big["touched"].size, want_cond=True)
    assert_bf16(host(dq), odq, cdq, name="dq, 4.4M-source tables")
    assert_bf16(dk_t, odk, cdk, name="dk, 4.4M-source tables")
    assert_bf16(dv_t, odv, cdv, name="dv, 4.4M-source tables")
    # sources no edge reads: exact zeros, including the top of the table
    # (every nonzero gradient element lies in a row some edge reads)
    for grad in (dk, dv):
        assert int(torch.count_nonzero(grad).item()) == int(torch.count_nonzero(grad[tt]).item())
    del k, v, dk, dv, tr
    torch.cuda.empty_cache()


@pytest.mark.parametrize("use_plan", [True, False])
def test_edge_softmax_scores_past_2_31_elements(gat, use_plan):
    """Scores [E, 8] with E * 8 past 2^31: 290,000 rows of 1,000 edges (the
    heavy-row path with a plan, rows streamed twice through a warp buffer
    without one), then 100,000 light rows of 1..40 edges whose scores all
    lie past the 2^31st element. Sampled row ranges (across the boundary and
    at the end) against the oracle on the same scores."""
    Hs = 8
    deg = np.concatenate([np.full(290_000, 1000),
                          np.random.default_rng(12).integers(1, 41, 100_000)]).astype(np.int64)
    rp = np.concatenate([[0], np.cumsum(deg)]).astype(np.int64)
    assert rp[290_000] * Hs > 2**31 and rp[-1] < 2**31
    rp32 = rp.astype(np.int32)
    E = int(rp[-1])
    g = torch.Generator(device="cuda").manual_seed(77)
    s = torch.randn((E, Hs), device="cuda", generator=g) * 2.0
    out = torch.empty_like(s)
    rpd = dev(rp32)
    plan = gat.Plan(rpd) if use_plan else None
    gat.gat_edge_softmax(rpd, s, Hs, out=out, plan=plan)
    torch.cuda.synchronize()
    boundary = int(np.searchsorted(rp, 2**31 // Hs, side="right")) - 1
    for r0, r1 in ((boundary - 3, boundary + 3), (289_990, 290_010), (389_000, 390_000)):
        e0, e1 = int(rp[r0]), int(rp[r1])
        sub = s[e0:e1].cpu().numpy()
        o = oracle.edge_softmax((rp[r0:r1 + 1] - e0).astype(np.int32), sub, Hs)
        assert_fp32(out[e0:e1].cpu().numpy().astype(np.float64), o,
                    name=f"edge softmax rows {r0}..{r1}, scores past 2^31")
    del s, out
    torch.cuda.empty_cache()
