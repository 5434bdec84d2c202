"""Seeded synthetic inputs for the five graph-attention workloads.

This module is shared by the fp64 oracle's tests and by the CUDA path's tests
and benchmark, so it deliberately holds none of the method's arithmetic: it
only draws random numbers, builds CSR/COO index arrays and rounds fp32 draws to
bf16 bit patterns. Every array is a NumPy array on the host; callers move it to
the device themselves.

Workloads (shapes follow the problem statements on the source pages):

* ``edge_softmax``  - multi-head CSR edge softmax, 384 rows, degrees U{0..36},
  scores [E,4] ~ N(0, 2^2)            (POPCORNBENCH FW-GLM-5-1 l1_p6)
* ``aggregate``     - softmax + neighbourhood aggregation, 384 rows, degrees
  U{0..36}, col_idx U[0,384), scores [E] ~ N(0,1), values [384,64] ~ N(0,1)
                                       (POPCORNBENCH Kimi-K2.6 l2_p37)
* ``sddmm``         - COO gathered dot product, src [1024,128], dst [768,128],
  16384 edges                          (POPCORNBENCH FW-GLM-5-1 l1_p10)
* ``fused``         - fused multi-head GAT layer, 1e6 rows, Zipf(2.1) in-degrees
  clipped to [1,4096] and rescaled to mean 16, col_idx uniform and sorted within
  each row, q/k/v bf16 [N,8,64] ~ N(0,1)
* ``dense``         - dense-masked small-graph attention block, B graphs of 24
  nodes, D=96, H=4, P=16, mask Bernoulli(0.3) with a unit diagonal, all Linear
  weights and biases ~ N(0, 0.02^2)    (POPCORNBENCH Kimi-K2.6 l2_p4)
* ``fused_backward`` - the fused workload plus an upstream gradient
  dout [N,8,64] ~ N(0,1) (bf16), for the backward of the fused layer
* ``spmm_heads``    - multi-head weighted aggregation at head_dim 32, 8 heads,
  fp32, on a power-law graph like ``fused``'s (POPCORNBENCH FW-GLM-5-1 l1_p18)

Draw order inside each generator is fixed and documented, so a seed fully
determines every array.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "f32_from_bf16_bits", "row_ptr_from_degrees",
    "uniform_degrees", "zipf_degrees", "page_mod_degrees",
    "make_edge_softmax", "make_aggregate", "make_sddmm", "make_fused",
    "make_dense", "make_csr", "make_spmm_heads", "make_fused_backward", "WORKLOADS",
]


# ----------------------------------------------------------------------------
# bf16 bit patterns (input quantisation only)
# ----------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); return uint16 bits.

    NaN is kept quiet; no input generated here is NaN or Inf.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


_BLOCK = 1 << 24


def _block_normals(seed_words: list[int], n: int, to_bf16: bool) -> np.ndarray:
    """n standard-normal fp32 draws (as bf16 bits when ``to_bf16``).

    The array is cut into fixed blocks of 2^24 elements; block j is drawn from
    PCG64(SeedSequence(seed_words).spawn(n_blocks)[j]). The result therefore
    depends only on ``seed_words`` and ``n``, not on how many threads fill it.
    """
    nb = max(1, -(-n // _BLOCK))
    kids = np.random.SeedSequence(seed_words).spawn(nb)
    out = np.empty(n, dtype=np.uint16 if to_bf16 else np.float32)

    def fill(j):
        s, e = j * _BLOCK, min(n, (j + 1) * _BLOCK)
        if e <= s:
            return
        g = np.random.Generator(np.random.PCG64(kids[j]))
        x = g.standard_normal(e - s, dtype=np.float32)
        out[s:e] = bf16_bits_from_f32(x) if to_bf16 else x

    if nb == 1:
        fill(0)
    else:
        from concurrent.futures import ThreadPoolExecutor
        import os
        with ThreadPoolExecutor(min(nb, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nb)))
    return out


# ----------------------------------------------------------------------------
# degree distributions and CSR construction
# ----------------------------------------------------------------------------
def row_ptr_from_degrees(deg: np.ndarray) -> np.ndarray:
    """Exclusive prefix sum of per-row degrees: int32 [N+1]."""
    deg = np.asarray(deg, dtype=np.int64)
    rp = np.zeros(deg.size + 1, dtype=np.int64)
    np.cumsum(deg, out=rp[1:])
    if rp[-1] >= 2**31:
        raise ValueError("edge count does not fit int32 row_ptr")
    return rp.astype(np.int32)


def uniform_degrees(rng: np.random.Generator, n: int, lo: int = 0, hi: int = 36) -> np.ndarray:
    """Degrees uniform over the integers [lo, hi] (inclusive)."""
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64)


def zipf_degrees(rng: np.random.Generator, n: int, a: float = 2.1,
                 dmax: int = 4096, mean: float = 16.0) -> np.ndarray:
    """Power-law in-degrees: Zipf(a) draws clipped to [1, dmax], rescaled so the
    sample mean is ``mean``, rounded half-to-even and re-clipped to [1, dmax]."""
    d = np.clip(rng.zipf(a, size=n), 1, dmax).astype(np.float64)
    d = np.rint(d * (mean / d.mean()))
    return np.clip(d, 1, dmax).astype(np.int64)


def page_mod_degrees(n: int, avg: int, k: int) -> np.ndarray:
    """The pages' deterministic degree rule: clamp(avg + (i mod k) - k//2, min=1).

    k=5 is the edge-softmax page's generator (degrees avg-2..avg+2), k=7 the
    aggregation page's (degrees avg-3..avg+3)."""
    i = np.arange(n, dtype=np.int64)
    return np.maximum(avg + (i % k) - (k // 2), 1)


def make_csr(rng: np.random.Generator, deg: np.ndarray, n_src: int,
             sort_within_rows: bool) -> tuple[np.ndarray, np.ndarray]:
    """row_ptr from ``deg`` and col_idx uniform over [0, n_src) with
    replacement (duplicate edges kept), optionally sorted inside each row."""
    rp = row_ptr_from_degrees(deg)
    E = int(rp[-1])
    ci = rng.integers(0, n_src, size=E, dtype=np.int64)
    if sort_within_rows and E:
        row = np.repeat(np.arange(deg.size, dtype=np.int64), np.asarray(deg, dtype=np.int64))
        key = row * np.int64(n_src) + ci
        key.sort(kind="stable")
        ci = key - row * np.int64(n_src)
    return rp, ci.astype(np.int32)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def make_edge_softmax(seed: int = 0, n: int = 384, H: int = 4, dmax: int = 36,
                      sigma: float = 2.0, deg: np.ndarray | None = None) -> dict:
    """Draws: degrees U{0..dmax} (unless ``deg`` is given), then scores."""
    rng = np.random.default_rng(seed)
    if deg is None:
        deg = uniform_degrees(rng, n, 0, dmax)
    rp = row_ptr_from_degrees(deg)
    E = int(rp[-1])
    scores = (sigma * rng.standard_normal((E, H))).astype(np.float32)
    return dict(row_ptr=rp, scores=scores, n_rows=len(deg), n_edges=E, H=H)


def make_aggregate(seed: int = 1, n: int = 384, F: int = 64, dmax: int = 36,
                   deg: np.ndarray | None = None) -> dict:
    """Draws: degrees U{0..dmax}, col_idx U[0,n) (unsorted), scores [E], values [n,F]."""
    rng = np.random.default_rng(seed)
    if deg is None:
        deg = uniform_degrees(rng, n, 0, dmax)
    rp, ci = make_csr(rng, deg, n, sort_within_rows=False)
    E = int(rp[-1])
    scores = rng.standard_normal(E).astype(np.float32)
    values = rng.standard_normal((n, F)).astype(np.float32)
    return dict(row_ptr=rp, col_idx=ci, scores=scores, values=values,
                n_rows=len(deg), n_src=n, n_edges=E, F=F)


def make_sddmm(seed: int = 2, n_src: int = 1024, n_dst: int = 768, E: int = 16384,
               F: int = 128) -> dict:
    """Draws: src_feat, dst_feat, src_idx, dst_idx (in that order)."""
    rng = np.random.default_rng(seed)
    src = rng.standard_normal((n_src, F)).astype(np.float32)
    dst = rng.standard_normal((n_dst, F)).astype(np.float32)
    si = rng.integers(0, n_src, size=E, dtype=np.int64).astype(np.int32)
    di = rng.integers(0, n_dst, size=E, dtype=np.int64).astype(np.int32)
    return dict(src_feat=src, dst_feat=dst, src_idx=si, dst_idx=di,
                n_src=n_src, n_dst=n_dst, n_edges=E, F=F)


def make_fused(seed: int = 3, n: int = 1_000_000, H: int = 8, Dh: int = 64,
               deg: np.ndarray | None = None, dmax: int = 4096, mean: float = 16.0,
               dtype: str = "bf16") -> dict:
    """Draws: Zipf degrees (unless ``deg`` is given) and col_idx from
    default_rng(seed); q, k, v from block streams seeded [seed, 1], [seed, 2],
    [seed, 3] (see ``_block_normals``).

    q/k/v are bf16 bit patterns (uint16) for dtype "bf16", else fp32.
    The score scale is 1/sqrt(Dh)."""
    rng = np.random.default_rng(seed)
    if deg is None:
        deg = zipf_degrees(rng, n, 2.1, dmax, mean)
    rp, ci = make_csr(rng, deg, n, sort_within_rows=True)
    m = n * H * Dh
    q, k, v = (_block_normals([seed, t + 1], m, dtype == "bf16").reshape(n, H, Dh)
               for t in range(3))
    return dict(row_ptr=rp, col_idx=ci, q=q, k=k, v=v, n_rows=n, n_src=n,
                n_edges=int(rp[-1]), H=H, Dh=Dh, scale=1.0 / np.sqrt(Dh), dtype=dtype)


def make_fused_backward(seed: int = 7, n: int = 1_000_000, H: int = 8, Dh: int = 64,
                        deg: np.ndarray | None = None, dmax: int = 4096, mean: float = 16.0,
                        dtype: str = "bf16") -> dict:
    """The fused workload's arrays (``make_fused`` with this seed) plus an
    upstream gradient dout [n,H,Dh] ~ N(0,1) from block stream [seed, 4]."""
    d = make_fused(seed, n, H, Dh, deg, dmax, mean, dtype)
    d["dout"] = _block_normals([seed, 4], n * H * Dh, dtype == "bf16").reshape(n, H, Dh)
    return d


def make_spmm_heads(seed: int = 5, n: int = 1_000_000, H: int = 8, Dh: int = 32,
                    deg: np.ndarray | None = None, dmax: int = 4096, mean: float = 16.0) -> dict:
    """Multi-head weighted aggregation at head_dim 32 on a power-law graph.

    Draws from default_rng(seed): Zipf degrees (unless ``deg``), col_idx
    (sorted within rows), edge weights U[0,1) fp32 [E,H]; then features fp32
    [n,H,Dh] ~ N(0,1) from block stream [seed, 1].
    """
    rng = np.random.default_rng(seed)
    if deg is None:
        deg = zipf_degrees(rng, n, 2.1, dmax, mean)
    rp, ci = make_csr(rng, deg, n, sort_within_rows=True)
    E = int(rp[-1])
    w = rng.random((E, H), dtype=np.float32)
    feat = _block_normals([seed, 1], n * H * Dh, False).reshape(n, H, Dh)
    return dict(row_ptr=rp, col_idx=ci, w=w, feat=feat, n_rows=n, n_src=n, n_edges=E, H=H, Dh=Dh)


def make_dense(seed: int = 4, B: int = 8192, N: int = 24, D: int = 96, H: int = 4,
               P: int = 16, wstd: float = 0.02, p_edge: float = 0.3,
               affine_ln: bool = False) -> dict:
    """Draws: nodes, pair_feats, mask uniforms, then Wq, Wk, Wv, W1, b1, W2, b2,
    Wout (and LayerNorm gamma/beta when ``affine_ln``; else gamma=1, beta=0)."""
    rng = np.random.default_rng(seed)
    nodes = rng.standard_normal((B, N, D)).astype(np.float32)
    pair = rng.standard_normal((B, N, N, P)).astype(np.float32)
    mask = (rng.random((B, N, N)) < p_edge).astype(np.float32)
    idx = np.arange(N)
    mask[:, idx, idx] = 1.0
    w = lambda *s: (wstd * rng.standard_normal(s)).astype(np.float32)  # noqa: E731
    Wq, Wk, Wv = w(D, D), w(D, D), w(D, D)
    W1, b1, W2, b2 = w(P, P), w(P), w(H, P), w(H)
    Wout = w(D, D)
    if affine_ln:
        ln_w = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
        ln_b = (0.1 * rng.standard_normal(D)).astype(np.float32)
    else:
        ln_w = np.ones(D, dtype=np.float32)
        ln_b = np.zeros(D, dtype=np.float32)
    return dict(nodes=nodes, pair_feats=pair, edge_mask=mask, ln_w=ln_w, ln_b=ln_b,
                ln_eps=1e-5, Wq=Wq, Wk=Wk, Wv=Wv, W1=W1, b1=b1, W2=W2, b2=b2,
                Wout=Wout, B=B, N=N, D=D, H=H, P=P)


#: name -> (generator, default seed, one-line description)
WORKLOADS = {
    "edge_softmax": (make_edge_softmax, 0, "multi-head CSR edge softmax, 384 rows, H=4"),
    "aggregate": (make_aggregate, 1, "softmax + aggregation, 384 rows, feat 64"),
    "sddmm": (make_sddmm, 2, "COO SDDMM, 1024x768 nodes, 16384 edges, feat 128"),
    "fused": (make_fused, 3, "fused GAT layer, 1e6 rows, Zipf(2.1) mean 16, H=8, Dh=64, bf16"),
    "dense": (make_dense, 4, "dense-masked small-graph block, B=8192, N=24, D=96, H=4, P=16"),
    "spmm_heads": (make_spmm_heads, 5, "weighted aggregation, 1e6 rows, Zipf(2.1) mean 16, H=8, "
                   "Dh=32, fp32"),
}
