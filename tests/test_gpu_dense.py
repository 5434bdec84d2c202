"""GPU parity of the dense-masked small-graph attention block against the
fp64 oracle (fp32 tolerance: |g - o| <= 1e-6 + 1e-5 |o|)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_fp32

pytestmark = pytest.mark.gpu

NAMES = ("nodes", "pair_feats", "edge_mask", "ln_w", "ln_b")
WEIGHTS = ("Wq", "Wk", "Wv", "W1", "b1", "W2", "b2", "Wout")


@pytest.fixture(scope="module")
def gat():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_graph_attention_head_gb300 as g
    return g


def run(gat, w, workspace=None):
    t = {k: torch.from_numpy(np.ascontiguousarray(w[k])).cuda() for k in NAMES + WEIGHTS}
    out = gat.gat_dense_masked_attention(t["nodes"], t["pair_feats"], t["edge_mask"], t["ln_w"],
                                         t["ln_b"], w["ln_eps"], *[t[k] for k in WEIGHTS],
                                         H=w["H"], workspace=workspace)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def fp32_block(w):
    """The block evaluated in plain float32 on the CPU (PyTorch modules and
    matmuls): the error floor of ordinary fp32 arithmetic on these inputs."""
    f = {k: torch.from_numpy(np.ascontiguousarray(w[k])) for k in NAMES + WEIGHTS}
    B, N, D, H = w["B"], w["N"], w["D"], w["H"]
    dh = D // H
    x = f["nodes"]
    xn = torch.nn.functional.layer_norm(x, (D,), f["ln_w"], f["ln_b"], w["ln_eps"])
    q, k, v = (xn @ f[n].T for n in ("Wq", "Wk", "Wv"))
    hid = f["pair_feats"] @ f["W1"].T + f["b1"]
    r = torch.nn.functional.silu(hid) @ f["W2"].T + f["b2"]
    q, k, v = (a.view(B, N, H, dh).transpose(1, 2) for a in (q, k, v))
    lg = q @ k.transpose(-1, -2) / np.sqrt(dh) + r.permute(0, 3, 1, 2)
    lg = lg.masked_fill((f["edge_mask"] < 0.5)[:, None], float("-inf"))
    ctx = (torch.softmax(lg, -1) @ v).transpose(1, 2).reshape(B, N, D)
    return (x + ctx @ f["Wout"].T).double().numpy()


@pytest.mark.parametrize("wstd,affine", [(0.02, False), (0.05, True)])
def test_dense_block_small_batch(gat, wstd, affine):
    w = W.make_dense(seed=4, B=96, wstd=wstd, affine_ln=affine)
    g = run(gat, w)
    o, c = oracle.dense_block(w, want_cond=True)
    rate = assert_fp32(g, o, c, name="dense block")
    assert rate > 0.999


def test_dense_block_sharp_attention_stress(gat):
    """Weights ~ N(0, 0.3^2) make logits ~ +-10 (sharp softmax). Plain fp32 on
    the CPU lands at ~0.1 of the fp32 tolerance on these inputs (measured
    here), so the kernel is held to the same fp32 tolerance as every other
    case, and also to 10x the measured fp32 error."""
    w = W.make_dense(seed=4, B=32, wstd=0.3, affine_ln=True)
    g = run(gat, w)
    o, c = oracle.dense_block(w, want_cond=True)
    scale = np.maximum(np.abs(o), c)
    floor = float(np.max(np.abs(fp32_block(w) - o) / scale))
    gerr = float(np.max(np.abs(g - o) / scale))
    assert floor < 1e-5  # plain fp32 meets the tolerance here
    assert_fp32(g, o, c, name="dense block stress")
    assert gerr <= 10 * floor + 1e-7, (gerr, floor)


@pytest.mark.parametrize("B,N", [(1, 24), (3, 24), (97, 24), (6, 13), (5, 1), (9, 5)])
def test_dense_block_tensor_core_ragged(gat, B, N):
    """The tensor-core shape (P=16, H=4, D=96) with a partial last tile and
    fewer than 24 nodes; one node that attends to nothing gives NaN."""
    w = W.make_dense(seed=40 + B + N, B=B, N=N, wstd=0.05, affine_ln=True)
    w["edge_mask"][B - 1, N - 1, :] = 0.0
    g = run(gat, w)
    o, c = oracle.dense_block(w, want_cond=True)
    assert np.isnan(g[B - 1, N - 1]).all()
    assert_fp32(g, o, c, name=f"dense block B={B} N={N}")


def test_dense_block_workspace_rules(gat):
    w = W.make_dense(seed=41, B=8)
    need = gat.gat_dense_masked_attention_workspace_size(w["N"], w["D"], w["H"], w["P"])
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(gat.GatError, match="GAT_ERR_WORKSPACE"):
        run(gat, w, workspace=small)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a = run(gat, w, workspace=ws)
    gat.gat_dense_masked_attention_status(ws)  # completed: no bounded wait gave up
    b = run(gat, w, workspace=ws)
    assert np.array_equal(a, b)  # deterministic, workspace reused


def test_dense_block_full_size_sampled_graphs(gat):
    w = W.make_dense(seed=4)  # B=8192, N=24, D=96, H=4, P=16
    g = run(gat, w)
    rng = np.random.default_rng(5)
    sel = np.unique(np.concatenate([[0, 8191], rng.integers(0, 8192, 62)]))
    o, c = oracle.dense_block(w, graphs=sel, want_cond=True)
    assert_fp32(g[sel], o, c, name="dense block full")
    assert np.isfinite(g).all()


@pytest.mark.parametrize("N", [11, 12, 20, 23])
def test_dense_block_tensor_core_several_tiles_per_cta(gat, N):
    """1,301 graphs: 326 tiles of 4 over the 152 resident blocks, 2-3 tiles
    each, so the cross-tile pipeline (the next tile's LayerNorm, mask words,
    pair prefetch and residual rows overlapping this tile's work) runs at
    node counts below 24; N = 11 and 12 sit on either side of the bias row
    stride's step (12 -> 28 floats). Sampled graphs, the last partial tile
    included, against the oracle."""
    B = 1301
    w = W.make_dense(seed=60 + N, B=B, N=N, wstd=0.05, affine_ln=True)
    g = run(gat, w)
    rng = np.random.default_rng(N)
    sel = np.unique(np.concatenate([[0, 1, 607, 608, B - 2, B - 1], rng.integers(0, B, 40)]))
    o, c = oracle.dense_block(w, graphs=sel, want_cond=True)
    assert_fp32(g[sel], o, c, name=f"dense block B={B} N={N}")
    assert np.isfinite(g).all()


def test_dense_block_other_shapes_and_masked_row(gat):
    w = W.make_dense(seed=22, B=5, N=7, D=12, H=3, P=5, wstd=0.1, affine_ln=True)
    w["edge_mask"][1, 4, :] = 0.0  # node 4 of graph 1 attends to nothing -> NaN, as the reference
    g = run(gat, w)
    o, c = oracle.dense_block(w, want_cond=True)
    assert np.isnan(g[1, 4]).all()
    assert_fp32(g, o, c, name="dense block shapes")


def test_dense_block_n32_d128(gat):
    w = W.make_dense(seed=23, B=40, N=32, D=128, H=8, P=32, wstd=0.05)
    o, c = oracle.dense_block(w, want_cond=True)
    assert_fp32(run(gat, w), o, c, name="dense block 32x128")


def test_dense_block_mask_densities_and_unread_masked_pairs(gat):
    """The tensor-core block runs the relation MLP on the unmasked pairs only
    (a masked pair's logit is -inf whatever its bias): masks from all
    unmasked to all masked per graph and per 4-graph tile (a tile with no
    unmasked pair, a tile of 2,304), a partial last tile; every masked pair's
    features are NaN or +inf, so a kernel that read them would show it.
    Rows with every key masked are NaN (as the reference); the rest match
    the oracle."""
    B, N = 37, 24
    w = W.make_dense(seed=51, B=B, wstd=0.05, affine_ln=True)
    rng = np.random.default_rng(52)
    m = w["edge_mask"]
    dens = {0: 1.0, 1: 0.0, 2: 0.05, 3: 0.95, 4: 0.5, 5: 0.3, 6: -1, 7: 0.3}
    for b, d in dens.items():
        if d < 0:  # the diagonal only
            m[b] = np.eye(N, dtype=np.float32)
        else:
            m[b] = (rng.random((N, N)) < d).astype(np.float32)
            if b != 1:
                np.fill_diagonal(m[b], 1.0)
    m[8:12] = 0.0  # a tile without one unmasked pair
    m[12:16] = 1.0  # a tile of unmasked pairs only
    masked = m < 0.5
    pf = w["pair_feats"]
    pf[masked] = np.nan
    pf[masked & (rng.random(masked.shape) < 0.3)] = np.inf
    g = run(gat, w)
    o, c = oracle.dense_block(w, want_cond=True)
    empty = ~(m >= 0.5).any(axis=2)  # [B, N]: queries with every key masked
    assert empty[1].all() and empty[8:12].all() and not empty[12:16].any()
    assert np.isnan(g[empty]).all()
    assert np.isfinite(g[~empty]).all()
    assert_fp32(g[~empty], o[~empty], c[~empty], name="dense block mask densities")
