"""Pins for the fp64 oracle: closed forms, invariants, brute force on tiny
inputs and independent library computations (NumPy / PyTorch CPU float64).

Each test is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a missing max-subtraction, heads
mixed up) fails at least one of them. CPU only.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from tests.golden import fixtures


# ----------------------------------------------------------------------------
# helpers: independent dense formulations (library softmax / matmul)
# ----------------------------------------------------------------------------
def np_softmax(x, axis=-1):
    """Library-style softmax via scipy (independent of the oracle's loops)."""
    from scipy.special import softmax
    return softmax(x, axis=axis)


def tiny_graph(rng, n, n_src, max_deg, allow_dup=False, sort=True):
    deg = rng.integers(0, max_deg + 1, size=n)
    rows, cols = [], []
    for i, d in enumerate(deg):
        if allow_dup:
            c = rng.integers(0, n_src, size=d)
        else:
            d = min(d, n_src)
            c = rng.choice(n_src, size=d, replace=False)
        if sort:
            c = np.sort(c)
        rows.append(np.full(len(c), i))
        cols.append(c)
    deg = np.array([len(c) for c in cols])
    rp = W.row_ptr_from_degrees(deg)
    ci = np.concatenate(cols).astype(np.int32) if cols else np.zeros(0, np.int32)
    return rp, ci


def row_of_edge(rp):
    deg = np.diff(rp.astype(np.int64))
    return np.repeat(np.arange(deg.size), deg)


# ----------------------------------------------------------------------------
# O1 segmented edge softmax
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("case", fixtures.load("softmax_closed_form.txt"))
def test_softmax_closed_forms(case):
    rp = np.array(case["row_ptr"], dtype=np.int32)
    H = int(case["H"][0])
    s = np.array(case["scores"], dtype=np.float64)
    # the fixture's ln values are exact in fp64 but the oracle receives fp32
    # inputs, as the GPU does; compare at fp32-input resolution
    out = oracle.edge_softmax(rp, s.astype(np.float32), H).ravel()
    np.testing.assert_allclose(out, case["expected"], rtol=1e-6, atol=0)


def test_softmax_matches_dense_masked_library_softmax():
    rng = np.random.default_rng(10)
    for H in (1, 3, 4):
        rp, ci = tiny_graph(rng, 9, 7, 6)
        E = int(rp[-1])
        s = (3 * rng.standard_normal((E, H))).astype(np.float32)
        got = oracle.edge_softmax(rp, s, H)
        r = row_of_edge(rp)
        for h in range(H):
            dense = np.full((9, 7), -np.inf)
            dense[r, ci] = s[:, h]
            P = np.zeros_like(dense)
            nz = np.isfinite(dense).any(axis=1)
            P[nz] = np_softmax(dense[nz], axis=1)
            np.testing.assert_allclose(got[:, h], P[r, ci], rtol=1e-13, atol=1e-15)


def test_softmax_invariants():
    rng = np.random.default_rng(11)
    d = W.make_edge_softmax(seed=5)
    rp, s, H = d["row_ptr"], d["scores"], d["H"]
    out = oracle.edge_softmax(rp, s, H)
    r = row_of_edge(rp)
    sums = np.zeros((rp.size - 1, H))
    np.add.at(sums, r, out)
    nonempty = np.diff(rp) > 0
    np.testing.assert_allclose(sums[nonempty], 1.0, rtol=0, atol=1e-13)
    assert (out > 0).all()
    # shift invariance per (row, head); shifts are exact in fp32 (multiples of 1/2)
    shift = (rng.integers(-8, 8, size=(rp.size - 1, H)) / 2.0).astype(np.float32)
    out2 = oracle.edge_softmax(rp, s + shift[r], H)
    np.testing.assert_allclose(out2, out, rtol=1e-6)  # fp32 rounding of s+shift
    # permutation equivariance inside each row
    perm = np.arange(r.size)
    for i in range(rp.size - 1):
        seg = perm[rp[i]:rp[i + 1]]
        perm[rp[i]:rp[i + 1]] = rng.permutation(seg)
    out3 = oracle.edge_softmax(rp, s[perm], H)
    np.testing.assert_allclose(out3, out[perm], rtol=1e-14)  # sum order differs


def test_softmax_large_scores_need_max_subtraction():
    rp = np.array([0, 3], dtype=np.int32)
    s = np.array([[800.0], [799.0], [-800.0]], dtype=np.float32)
    out = oracle.edge_softmax(rp, s, 1).ravel()
    e = math.exp(-1.0)
    np.testing.assert_allclose(out[:2], [1 / (1 + e), e / (1 + e)], rtol=1e-14)
    assert out[2] == 0.0


def test_softmax_heads_with_far_apart_scales():
    """Each head subtracts its own maximum: heads whose scores sit near +700
    and -700 would underflow (or overflow) with another head's maximum."""
    rng = np.random.default_rng(25)
    rp = np.array([0, 5, 9], dtype=np.int32)
    s = np.stack([700 + rng.standard_normal(9), -700 + rng.standard_normal(9)], 1).astype(np.float32)
    out = oracle.edge_softmax(rp, s, 2)
    for h in range(2):
        for i in range(2):
            seg = slice(rp[i], rp[i + 1])
            np.testing.assert_allclose(out[seg, h], np_softmax(s[seg, h].astype(np.float64)),
                                       rtol=1e-12)


def test_softmax_all_minus_inf_row_is_nan_like_library():
    import torch
    rp = np.array([0, 2], dtype=np.int32)
    s = np.full((2, 1), -np.inf, dtype=np.float32)
    out = oracle.edge_softmax(rp, s, 1)
    ref = torch.softmax(torch.tensor(s[:, 0], dtype=torch.float64), 0).numpy()
    assert np.isnan(out).all() and np.isnan(ref).all()


def test_softmax_page_generator_rows():
    # edge-softmax page generator: degrees clamp(18 + (i mod 5) - 2, 1) -> 16..20
    deg = W.page_mod_degrees(384, 18, 5)
    assert deg.min() == 16 and deg.max() == 20
    d = W.make_edge_softmax(seed=6, deg=deg, H=8)
    out = oracle.edge_softmax(d["row_ptr"], d["scores"], 8)
    sums = np.zeros((384, 8))
    np.add.at(sums, row_of_edge(d["row_ptr"]), out)
    np.testing.assert_allclose(sums, 1.0, atol=1e-13)


# ----------------------------------------------------------------------------
# O3 SDDMM
# ----------------------------------------------------------------------------
def test_sddmm_closed_form():
    (c,) = fixtures.load("sddmm_closed_form.txt")
    a = np.array(c["src_feat"], np.float32).reshape(3, 4)
    b = np.array(c["dst_feat"], np.float32).reshape(2, 4)
    out = oracle.sddmm(np.array(c["src_idx"], np.int32), a, b, 1, 4,
                       dst_idx=np.array(c["dst_idx"], np.int32))
    np.testing.assert_array_equal(out.ravel(), c["expected"])


def test_sddmm_equals_library_matmul_sampled_at_edges_full_size():
    d = W.make_sddmm()
    out, cond = oracle.sddmm(d["src_idx"], d["src_feat"], d["dst_feat"], 1, 128,
                             dst_idx=d["dst_idx"], want_cond=True)
    G = d["src_feat"].astype(np.float64) @ d["dst_feat"].astype(np.float64).T
    ref = G[d["src_idx"], d["dst_idx"]]
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)
    assert (cond[:, 0] >= np.abs(out[:, 0]) - 1e-12).all()


def test_sddmm_multihead_scale_and_csr_form():
    rng = np.random.default_rng(12)
    H, Dh, n = 3, 5, 6
    rp, ci = tiny_graph(rng, n, n, 5, allow_dup=True)
    q = rng.standard_normal((n, H, Dh)).astype(np.float32)
    k = rng.standard_normal((n, H, Dh)).astype(np.float32)
    scale = 0.37
    csr = oracle.sddmm(ci, k, q, H, Dh, scale=scale, row_ptr=rp)
    r = row_of_edge(rp)
    coo = oracle.sddmm(ci, k, q, H, Dh, scale=scale, dst_idx=r.astype(np.int32))
    np.testing.assert_array_equal(csr, coo)
    ref = np.stack([(k[:, h].astype(np.float64) @ q[:, h].astype(np.float64).T)[ci, r]
                    for h in range(H)], axis=1) * scale
    np.testing.assert_allclose(csr, ref, rtol=1e-12, atol=1e-13)


def test_sddmm_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(13)
    a = W.bf16_bits_from_f32(rng.standard_normal((7, 16)).astype(np.float32))
    b = W.bf16_bits_from_f32(rng.standard_normal((5, 16)).astype(np.float32))
    si = rng.integers(0, 7, 20).astype(np.int32)
    di = rng.integers(0, 5, 20).astype(np.int32)
    got = oracle.sddmm(si, a, b, 2, 8, dst_idx=di)
    af = W.f32_from_bf16_bits(a).astype(np.float64).reshape(7, 2, 8)
    bf = W.f32_from_bf16_bits(b).astype(np.float64).reshape(5, 2, 8)
    ref = np.einsum("ehd,ehd->eh", af[si], bf[di])
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------
# weighted SpMM and O2 (softmax + aggregation)
# ----------------------------------------------------------------------------
def test_spmm_equals_dense_matmul_with_duplicates_summed():
    rng = np.random.default_rng(14)
    H, Dh, n, n_src = 2, 3, 8, 5
    rp, ci = tiny_graph(rng, n, n_src, 7, allow_dup=True, sort=False)
    E = int(rp[-1])
    w = rng.standard_normal((E, H))
    feat = rng.standard_normal((n_src, H, Dh)).astype(np.float32)
    out, cond = oracle.spmm_weighted(rp, ci, w, feat, H, Dh, want_cond=True)
    r = row_of_edge(rp)
    for h in range(H):
        Wd = np.zeros((n, n_src))
        np.add.at(Wd, (r, ci), w[:, h])
        np.testing.assert_allclose(out[:, h], Wd @ feat[:, h].astype(np.float64),
                                   rtol=1e-12, atol=1e-13)
    assert (cond >= np.abs(out) - 1e-13).all()
    empty = np.diff(rp) == 0
    assert (out[empty] == 0).all()


def test_aggregate_page_semantics_and_zero_rows():
    d = W.make_aggregate(seed=15, n=40)
    w = oracle.edge_softmax(d["row_ptr"], d["scores"], 1)
    out = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], w, d["values"], 1, d["F"])
    # independent: per row, library softmax over the row's scores then a dot
    rp = d["row_ptr"]
    for i in range(40):
        e0, e1 = rp[i], rp[i + 1]
        if e0 == e1:
            assert (out[i] == 0).all()
            continue
        p = np_softmax(d["scores"][e0:e1].astype(np.float64))
        ref = p @ d["values"][d["col_idx"][e0:e1]].astype(np.float64)
        np.testing.assert_allclose(out[i, 0], ref, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# O4 fused layer
# ----------------------------------------------------------------------------
def test_fused_closed_form():
    (c,) = fixtures.load("fused_closed_form.txt")
    rp = np.array(c["row_ptr"], np.int32)
    ci = np.array(c["col_idx"], np.int32)
    q, k, v = (np.array(c[x], np.float64).reshape(3, 1, 2) for x in ("q", "k", "v"))
    # ln 3 is not exact in fp32: feed fp64-exact values through fp32 and
    # compare at fp32-input resolution
    out = oracle.fused_layer(rp, ci, q.astype(np.float32), k.astype(np.float32),
                             v.astype(np.float32), 1, 2, 1.0)
    np.testing.assert_allclose(out.ravel(), c["expected"], rtol=1e-6, atol=1e-6)


def dense_masked_attention(rp, ci, q, k, v, scale):
    """Independent formulation: per head, dense logits Q K^T * scale plus
    log(edge multiplicity) (-inf where no edge), library softmax, times V."""
    n, H, Dh = q.shape
    n_src = k.shape[0]
    r = row_of_edge(rp)
    cnt = np.zeros((n, n_src))
    np.add.at(cnt, (r, ci), 1.0)
    with np.errstate(divide="ignore"):
        logm = np.log(cnt)
    out = np.zeros((n, H, Dh))
    nz = cnt.sum(1) > 0
    for h in range(H):
        S = q[:, h].astype(np.float64) @ k[:, h].astype(np.float64).T * scale + logm
        A = np.zeros_like(S)
        A[nz] = np_softmax(S[nz], axis=1)
        out[:, h] = A @ v[:, h].astype(np.float64)
    return out


@pytest.mark.parametrize("dup", [False, True])
def test_fused_equals_dense_masked_attention(dup):
    rng = np.random.default_rng(16 + dup)
    n, H, Dh = 11, 3, 4
    rp, ci = tiny_graph(rng, n, n, 7, allow_dup=dup, sort=not dup)
    q, k, v = (rng.standard_normal((n, H, Dh)).astype(np.float32) for _ in range(3))
    got = oracle.fused_layer(rp, ci, q, k, v, H, Dh, 0.5)
    ref = dense_masked_attention(rp, ci, q, k, v, 0.5)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_fused_special_cases():
    rng = np.random.default_rng(18)
    n, H, Dh = 5, 2, 3
    k = rng.standard_normal((n, H, Dh)).astype(np.float32)
    v = rng.standard_normal((n, H, Dh)).astype(np.float32)
    q = rng.standard_normal((n, H, Dh)).astype(np.float32)
    # row 0: single edge -> exactly v[src]; row 1: three edges to the same source
    # -> exactly v[src]; row 2: empty -> 0; row 3: q = 0 -> plain average
    rp = np.array([0, 1, 4, 4, 7, 7], np.int32)
    ci = np.array([3, 2, 2, 2, 0, 1, 4], np.int32)
    q[3] = 0
    out = oracle.fused_layer(rp, ci, q, k, v, H, Dh, 0.125)
    np.testing.assert_array_equal(out[0], v[3].astype(np.float64))
    np.testing.assert_allclose(out[1], v[2].astype(np.float64), rtol=1e-15, atol=1e-15)
    assert (out[2] == 0).all() and (out[4] == 0).all()
    np.testing.assert_allclose(out[3], v[[0, 1, 4]].astype(np.float64).mean(0), rtol=1e-14)


def test_fused_composes_from_stages_and_row_selection():
    d = W.make_fused(seed=19, n=300, dmax=64)
    args = (d["row_ptr"], d["col_idx"], d["q"], d["k"], d["v"], d["H"], d["Dh"], d["scale"])
    full = oracle.fused_layer(*args)
    s = oracle.sddmm(d["col_idx"], d["k"], d["q"], d["H"], d["Dh"], scale=d["scale"],
                     row_ptr=d["row_ptr"])
    w = oracle.edge_softmax(d["row_ptr"], s.astype(np.float32), d["H"])
    agg = oracle.spmm_weighted(d["row_ptr"], d["col_idx"], w, d["v"], d["H"], d["Dh"])
    np.testing.assert_allclose(full, agg, rtol=1e-5, atol=1e-6)  # fp32 rounding of s
    rows = np.array([299, 0, 17, 17, 150])
    sel = oracle.fused_layer(*args, rows=rows)
    np.testing.assert_array_equal(sel, full[rows])
    # bf16 bits are widened exactly: same as feeding the widened fp32 values
    f32 = [W.f32_from_bf16_bits(d[x]) for x in ("q", "k", "v")]
    full32 = oracle.fused_layer(d["row_ptr"], d["col_idx"], *f32, d["H"], d["Dh"], d["scale"])
    np.testing.assert_array_equal(full32, full)


def test_fused_matches_dense_on_bf16_zipf_graph():
    d = W.make_fused(seed=20, n=64, dmax=32, mean=6.0)
    f32 = [W.f32_from_bf16_bits(d[x]).reshape(64, 8, 64) for x in ("q", "k", "v")]
    got = oracle.fused_layer(d["row_ptr"], d["col_idx"], d["q"], d["k"], d["v"], 8, 64, 0.125)
    ref = dense_masked_attention(d["row_ptr"], d["col_idx"], *f32, 0.125)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------
# O6 backward of the fused layer: central differences of the (pinned) forward
# oracle, PyTorch float64 autograd of dense masked attention, special cases
# ----------------------------------------------------------------------------
def _grid_values(rng, shape):
    """fp32 values on a coarse binary grid (multiples of 1/64 in [-2, 2)), so
    that x +/- 2^-14 is exact in fp32 and finite differences see exact inputs."""
    return (rng.integers(-128, 128, size=shape) / 64.0).astype(np.float32)


@pytest.mark.parametrize("dup", [False, True])
def test_backward_equals_central_differences_of_forward(dup):
    rng = np.random.default_rng(60 + dup)
    n, n_src, H, Dh, scale = 6, 5, 2, 3, 0.7
    rp, ci = tiny_graph(rng, n, n_src, 4, allow_dup=dup, sort=not dup)
    x = {"q": _grid_values(rng, (n, H, Dh)), "k": _grid_values(rng, (n_src, H, Dh)),
         "v": _grid_values(rng, (n_src, H, Dh))}
    g = _grid_values(rng, (n, H, Dh))
    grads = dict(zip("qkv", oracle.fused_backward(rp, ci, x["q"], x["k"], x["v"], g, H, Dh,
                                                  scale)))

    def loss(**over):
        a = {**x, **over}
        out = oracle.fused_layer(rp, ci, a["q"], a["k"], a["v"], H, Dh, scale)
        return float((out * g.astype(np.float64)).sum())

    step = 2.0 ** -14
    for name in "qkv":
        fd = np.zeros(x[name].shape)
        for idx in np.ndindex(x[name].shape):
            xp, xm = x[name].copy(), x[name].copy()
            xp[idx] += step
            xm[idx] -= step
            fd[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * step)
        np.testing.assert_allclose(grads[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_backward_equals_torch_autograd_of_dense_masked_attention():
    import torch
    rng = np.random.default_rng(62)
    n, n_src, H, Dh, scale = 9, 7, 3, 4, 0.5
    rp, ci = tiny_graph(rng, n, n_src, 6)
    q, g = (rng.standard_normal((n, H, Dh)).astype(np.float32) for _ in range(2))
    k, v = (rng.standard_normal((n_src, H, Dh)).astype(np.float32) for _ in range(2))
    Q, K, V = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    mask = torch.zeros((n, n_src), dtype=torch.bool)
    mask[torch.as_tensor(row_of_edge(rp)), torch.as_tensor(ci.astype(np.int64))] = True
    nz = mask.any(1)
    S = torch.einsum("ihd,jhd->hij", Q, K) * scale
    S = S[:, nz].masked_fill(~mask[nz][None], float("-inf"))
    A = torch.softmax(S, dim=-1)
    out = torch.zeros((n, H, Dh), dtype=torch.float64)
    out[nz] = torch.einsum("hij,jhd->ihd", A, V)
    (out * torch.tensor(g, dtype=torch.float64)).sum().backward()
    dq, dk, dv = oracle.fused_backward(rp, ci, q, k, v, g, H, Dh, scale)
    assert (~nz).any()  # the graph has an empty row
    for got, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-13)


def test_backward_special_cases():
    rng = np.random.default_rng(63)
    n, n_src, H, Dh = 5, 4, 2, 3
    q, g = (rng.standard_normal((n, H, Dh)).astype(np.float32) for _ in range(2))
    k, v = (rng.standard_normal((n_src, H, Dh)).astype(np.float32) for _ in range(2))
    # one edge per row: the softmax weight is 1 whatever the score, so dq = dk = 0
    # exactly and dv[j] is the sum of dout over the rows reading j
    rp = np.arange(n + 1, dtype=np.int32)
    ci = np.array([2, 0, 2, 3, 2], np.int32)
    dq, dk, dv = oracle.fused_backward(rp, ci, q, k, v, g, H, Dh, 0.3)
    assert (dq == 0).all() and (dk == 0).all()
    ref = np.zeros((n_src, H, Dh))
    np.add.at(ref, ci, g.astype(np.float64))
    np.testing.assert_allclose(dv, ref, rtol=1e-15, atol=1e-15)
    assert (dv[1] == 0).all()  # a source no edge reads
    # empty rows contribute nothing; dq of an empty row is zero
    rp2 = np.array([0, 0, 2, 2, 3, 3], np.int32)
    ci2 = np.array([1, 3, 0], np.int32)
    dq2, dk2, dv2, cq, ck, cv = oracle.fused_backward(rp2, ci2, q, k, v, g, H, Dh, 0.3,
                                                      want_cond=True)
    assert (dq2[[0, 2, 3, 4]] == 0).all() and (dk2[2] == 0).all() and (dv2[2] == 0).all()
    assert (cq >= np.abs(dq2)).all() and (ck >= np.abs(dk2)).all() and (cv >= np.abs(dv2)).all()
    # row 3's single edge: no dq/dk, dv[0] = dout[3]
    np.testing.assert_array_equal(dv2[0], g[3].astype(np.float64))


def test_backward_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(64)
    n, H, Dh = 7, 2, 8
    rp, ci = tiny_graph(rng, n, n, 5, allow_dup=True, sort=False)
    f = [rng.standard_normal((n, H, Dh)).astype(np.float32) for _ in range(4)]
    bits = [W.bf16_bits_from_f32(a) for a in f]
    wid = [W.f32_from_bf16_bits(b) for b in bits]
    a = oracle.fused_backward(rp, ci, *bits, H, Dh, 0.25)
    b = oracle.fused_backward(rp, ci, *wid, H, Dh, 0.25)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("n,n_src,max_deg", [(50, 30, 9), (200, 7, 40), (1, 1, 0), (30, 1000, 3)])
def test_transpose_equals_stable_library_argsort(n, n_src, max_deg):
    rng = np.random.default_rng(65 + n)
    rp, ci = tiny_graph(rng, n, n_src, max_deg, allow_dup=True, sort=False)
    sp, perm, dst = oracle.transpose(rp, ci, n_src)
    order = np.argsort(ci, kind="stable")
    np.testing.assert_array_equal(perm, order)
    np.testing.assert_array_equal(dst, row_of_edge(rp)[order])
    np.testing.assert_array_equal(sp, np.concatenate([[0], np.cumsum(np.bincount(ci, minlength=n_src))]))


# ----------------------------------------------------------------------------
# O7 fp8 (E4M3) feature tables: codec against PyTorch's float8_e4m3fn,
# quantiser invariants, the fp8 fused layer against the fused layer
# ----------------------------------------------------------------------------
def test_fp8_decode_all_codes_equal_library():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.fp8_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_fp8_encode_equals_library_rounding_and_saturates():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.fp8_decode(codes)
    fin = np.isfinite(vals)
    grid = np.unique(vals[fin])
    mids = (grid[1:] + grid[:-1]) / 2  # exact ties: nearest-even decides
    rng = np.random.default_rng(66)
    x = np.concatenate([grid, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                        rng.standard_normal(20000) * 60, rng.standard_normal(2000) * 0.01])
    x = x[np.abs(x) <= 448].astype(np.float32)
    got = oracle.fp8_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, ref)
    # every finite code is its own value's encoding
    np.testing.assert_array_equal(oracle.fp8_encode(vals[fin].astype(np.float32)), codes[fin])
    # beyond the largest finite value: saturation
    big = np.array([449, 464, 480, 1e4, 3e38, -500], np.float32)
    np.testing.assert_array_equal(oracle.fp8_encode(big), [0x7E] * 5 + [0xFE])


def test_fp8_quantize_invariants():
    rng = np.random.default_rng(67)
    n, H, Dh = 50, 4, 16
    x = (rng.standard_normal((n, H, Dh)) * rng.uniform(0.01, 100, (n, H, 1))).astype(np.float32)
    x[3, 1] = 0.0  # an all-zero head
    codes, scales = oracle.fp8_quantize(x, H, Dh)
    assert scales[3, 1] == 1.0 and (codes[3, 1] == 0).all()
    amax = np.abs(x).max(-1)
    nz = amax > 0
    np.testing.assert_array_equal(scales[nz], (amax[nz] / np.float32(448)).astype(np.float32))
    # the largest element of each head lands on +-448
    arg = np.abs(x).argmax(-1)
    top = np.take_along_axis(codes, arg[..., None], -1)[..., 0]
    assert np.isin(top[nz], [0x7E, 0xFE]).all()
    # dequantised values within half a grid step (1/16 relative for normals)
    deq = oracle.fp8_decode(codes) * scales[..., None]
    err = np.abs(deq - x)
    tol = np.maximum(np.abs(x) / 16, scales[..., None] * 2.0 ** -10)
    assert (err <= tol * (1 + 1e-6)).all()
    # bf16 inputs widen exactly
    bits = W.bf16_bits_from_f32(x)
    c2, s2 = oracle.fp8_quantize(bits, H, Dh)
    c3, s3 = oracle.fp8_quantize(W.f32_from_bf16_bits(bits), H, Dh)
    np.testing.assert_array_equal(c2, c3)
    np.testing.assert_array_equal(s2, s3)


def test_fused_fp8_equals_fused_layer_on_dequantised_tables():
    rng = np.random.default_rng(68)
    n, H, Dh = 40, 2, 16
    rp, ci = tiny_graph(rng, n, n, 9, allow_dup=True, sort=False)
    q = rng.standard_normal((n, H, Dh)).astype(np.float32)
    k8 = rng.integers(0, 256, (n, H, Dh), dtype=np.uint8)
    v8 = rng.integers(0, 256, (n, H, Dh), dtype=np.uint8)
    for c in (k8, v8):
        c[(c & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    # power-of-two scales: decode * scale is exact in fp32
    ks = (2.0 ** rng.integers(-8, -2, (n, H))).astype(np.float32)
    vs = (2.0 ** rng.integers(-4, 0, (n, H))).astype(np.float32)
    kf = (oracle.fp8_decode(k8) * ks[..., None]).astype(np.float32)
    vf = (oracle.fp8_decode(v8) * vs[..., None]).astype(np.float32)
    got = oracle.fused_layer_fp8(rp, ci, q, k8, ks, v8, vs, H, Dh, 0.25)
    ref = oracle.fused_layer(rp, ci, q, kf, vf, H, Dh, 0.25)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------
# O5 dense-masked block: PyTorch CPU float64 modules
# ----------------------------------------------------------------------------
def torch_block(w, graphs):
    import torch
    from torch import nn
    t = lambda a: torch.tensor(np.asarray(a), dtype=torch.float64)  # noqa: E731
    D, H, P = w["D"], w["H"], w["P"]
    ln = nn.LayerNorm(D, eps=w["ln_eps"]).double()
    q_p, k_p, v_p, o_p = (nn.Linear(D, D, bias=False).double() for _ in range(4))
    mlp = nn.Sequential(nn.Linear(P, P), nn.SiLU(), nn.Linear(P, H)).double()
    with torch.no_grad():
        ln.weight.copy_(t(w["ln_w"]))
        ln.bias.copy_(t(w["ln_b"]))
        q_p.weight.copy_(t(w["Wq"]))
        k_p.weight.copy_(t(w["Wk"]))
        v_p.weight.copy_(t(w["Wv"]))
        o_p.weight.copy_(t(w["Wout"]))
        mlp[0].weight.copy_(t(w["W1"]))
        mlp[0].bias.copy_(t(w["b1"]))
        mlp[2].weight.copy_(t(w["W2"]))
        mlp[2].bias.copy_(t(w["b2"]))
        x = t(w["nodes"][graphs])
        pf = t(w["pair_feats"][graphs])
        m = t(w["edge_mask"][graphs])
        B, N, _ = x.shape
        dh = D // H
        h = ln(x)
        q = q_p(h).view(B, N, H, dh).transpose(1, 2)
        k = k_p(h).view(B, N, H, dh).transpose(1, 2)
        v = v_p(h).view(B, N, H, dh).transpose(1, 2)
        logits = q @ k.transpose(-2, -1) / math.sqrt(dh)
        logits = logits + mlp(pf).permute(0, 3, 1, 2)
        logits = logits.masked_fill(m.unsqueeze(1) < 0.5, float("-inf"))
        a = torch.softmax(logits, dim=-1)
        ctx = (a @ v).transpose(1, 2).reshape(B, N, D)
        return (x + o_p(ctx)).numpy()


@pytest.mark.parametrize("affine", [False, True])
def test_dense_block_equals_torch_modules(affine):
    w = W.make_dense(seed=21, B=6, affine_ln=affine, wstd=0.3)
    g = np.array([0, 3, 5])
    got = oracle.dense_block(w, graphs=g)
    ref = torch_block(w, g)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_dense_block_other_shapes_and_fully_masked_row():
    w = W.make_dense(seed=22, B=3, N=7, D=12, H=3, P=5, wstd=0.5, affine_ln=True)
    w["edge_mask"][1, 4, :] = 0.0  # node 4 of graph 1 attends to nothing
    got = oracle.dense_block(w)
    ref = torch_block(w, np.arange(3))
    assert np.isnan(got[1, 4]).all() and np.isnan(ref[1, 4]).all()
    ok = ~np.isnan(ref)
    np.testing.assert_allclose(got[ok], ref[ok], rtol=1e-12, atol=1e-12)
    assert not np.isnan(got[0]).any()


def test_dense_block_zero_out_proj_is_identity():
    w = W.make_dense(seed=23, B=2)
    w["Wout"][:] = 0
    got = oracle.dense_block(w)
    np.testing.assert_array_equal(got, w["nodes"].astype(np.float64))


# ----------------------------------------------------------------------------
# degree-bucket plan (integers): brute-force re-derivation
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("T,C", [(0, 1), (4, 3), (32, 32), (64, 16)])
def test_plan_brute_force(T, C):
    rng = np.random.default_rng(24)
    deg = np.concatenate([rng.integers(0, 80, 200), [T, T + 1, C, C + 1, 2 * C, 0]])
    rp = W.row_ptr_from_degrees(deg)
    hr, cs, cr = oracle.plan(rp, T, C)
    exp_hr, exp_cs, exp_cr = [], [0], []
    for i, dgr in enumerate(deg):
        if dgr > T:
            nch = -(-int(dgr) // C)
            exp_cr += [len(exp_hr)] * nch
            exp_hr.append(i)
            exp_cs.append(exp_cs[-1] + nch)
    np.testing.assert_array_equal(hr, exp_hr)
    np.testing.assert_array_equal(cs, exp_cs)
    np.testing.assert_array_equal(cr, exp_cr)
    # the chunks tile every heavy row's edge range exactly, each at most C long
    covered = np.zeros(int(rp[-1]), dtype=np.int64)
    for c, r in enumerate(cr):
        row = hr[r]
        j = c - cs[r]
        e0 = rp[row] + j * C
        e1 = min(e0 + C, rp[row + 1])
        assert 0 < e1 - e0 <= C
        covered[e0:e1] += 1
    heavy_edges = np.zeros_like(covered)
    for row in hr:
        heavy_edges[rp[row]:rp[row + 1]] = 1
    np.testing.assert_array_equal(covered, heavy_edges)
