"""fp64 CPU oracle for the graph-attention path (test infrastructure).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product library never
imports this package, and this package never imports the product library: the
two share no code. The arithmetic lives in ``oracle.c`` (plain loops in double
precision); this module builds it with gcc and wraps it with ctypes/NumPy.

Parity pins: every function here is checked against closed forms, invariants
and independent library computations (NumPy / PyTorch CPU float64) in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, -O2, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        # GAT_ORACLE_LIB names another compiled oracle (the mutation tests
        # plant mistakes in a copy of oracle.c and check the pins catch them)
        override = os.environ.get("GAT_ORACLE_LIB")
        if override:
            path = override
        else:
            build()
            path = _LIB
        lib = ctypes.CDLL(path)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.oracle_edge_softmax.argtypes = [P, I64, I32, P, P]
        lib.oracle_spmm_weighted.argtypes = [P, P, I64, I32, I32, P, P, ctypes.c_int, P, P]
        lib.oracle_sddmm.argtypes = [P, P, P, I64, I64, I32, I32, D, P, P, ctypes.c_int, P, P]
        lib.oracle_fused_layer.argtypes = [P, P, I64, I32, I32, D, P, P, P, ctypes.c_int,
                                           P, I64, P, P]
        lib.oracle_dense_block.argtypes = [I32, I32, I32, I32, I32, P, P, P, P, P, D,
                                           P, P, P, P, P, P, P, P, P, I64, P, P]
        lib.oracle_plan.argtypes = [P, I64, I32, I32, P, P, P, P, P]
        lib.oracle_fused_backward.argtypes = [P, P, I64, I64, I32, I32, D, P, P, P, P,
                                              ctypes.c_int, P, P, P, P, P, P]
        lib.oracle_transpose.argtypes = [P, P, I64, I64, P, P, P]
        lib.oracle_fp8_decode.argtypes = [P, I64, P]
        lib.oracle_fp8_encode.argtypes = [P, I64, P]
        lib.oracle_fp8_quantize.argtypes = [P, ctypes.c_int, I64, I32, I32, P, P]
        lib.oracle_fused_layer_fp8.argtypes = [P, P, I64, I32, I32, D, P, ctypes.c_int, P, P, P,
                                               P, P, I64, P, P]
        for f in ("oracle_fp8_decode", "oracle_fp8_encode", "oracle_fp8_quantize",
                  "oracle_fused_layer_fp8","oracle_edge_softmax", "oracle_spmm_weighted", "oracle_sddmm",
                  "oracle_fused_layer", "oracle_dense_block", "oracle_plan",
                  "oracle_fused_backward", "oracle_transpose"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _feat(a):
    """Return (contiguous array, dtype code): uint16 arrays are bf16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    return np.ascontiguousarray(a, dtype=np.float32), F32


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} failed with code {rc}")


def edge_softmax(row_ptr, scores, H):
    """Segmented softmax per row and head. Returns fp64 [E,H] (rows of degree
    0 own no entries)."""
    rp = _c(row_ptr, np.int32)
    s = _c(scores, np.float32).reshape(-1, H)
    out = np.zeros_like(s, dtype=np.float64)
    _check(_load().oracle_edge_softmax(_p(rp), rp.size - 1, H, _p(s), _p(out)),
           "oracle_edge_softmax")
    return out


def spmm_weighted(row_ptr, col_idx, w, feat, H, Dh, want_cond=False):
    """out[i,h,:] = sum_e w[e,h] feat[col_idx[e],h,:]; fp64 [n_rows,H,Dh]."""
    rp, ci = _c(row_ptr, np.int32), _c(col_idx, np.int32)
    w64 = _c(w, np.float64).reshape(-1, H)
    f, dt = _feat(feat)
    n = rp.size - 1
    out = np.empty((n, H, Dh), dtype=np.float64)
    cond = np.empty_like(out) if want_cond else None
    _check(_load().oracle_spmm_weighted(_p(rp), _p(ci), n, H, Dh, _p(w64), _p(f), dt,
                                        _p(out), _p(cond)), "oracle_spmm_weighted")
    return (out, cond) if want_cond else out


def sddmm(src_idx, src_feat, dst_feat, H, Dh, scale=1.0, dst_idx=None, row_ptr=None,
          want_cond=False):
    """Gathered dot products. COO when row_ptr is None, else CSR (dst = row)."""
    si = _c(src_idx, np.int32)
    di = _c(dst_idx, np.int32)
    rp = _c(row_ptr, np.int32)
    a, dt = _feat(src_feat)
    b, dt2 = _feat(dst_feat)
    if dt != dt2:
        raise ValueError("src_feat and dst_feat must share a dtype")
    E = si.size
    out = np.empty((E, H), dtype=np.float64)
    cond = np.empty_like(out) if want_cond else None
    n_rows = 0 if rp is None else rp.size - 1
    _check(_load().oracle_sddmm(_p(rp), _p(si), _p(di), n_rows, E, H, Dh, float(scale),
                                _p(a), _p(b), dt, _p(out), _p(cond)), "oracle_sddmm")
    return (out, cond) if want_cond else out


def fused_layer(row_ptr, col_idx, q, k, v, H, Dh, scale, rows=None, want_cond=False):
    """Fused GAT layer by stages (two-pass softmax). fp64 [n_sel,H,Dh]."""
    rp, ci = _c(row_ptr, np.int32), _c(col_idx, np.int32)
    qa, dt = _feat(q)
    ka, _ = _feat(k)
    va, _ = _feat(v)
    sel = None if rows is None else _c(rows, np.int64)
    n = rp.size - 1
    n_sel = n if sel is None else sel.size
    out = np.empty((n_sel, H, Dh), dtype=np.float64)
    cond = np.empty_like(out) if want_cond else None
    _check(_load().oracle_fused_layer(_p(rp), _p(ci), n, H, Dh, float(scale), _p(qa),
                                      _p(ka), _p(va), dt, _p(sel), n_sel, _p(out),
                                      _p(cond)), "oracle_fused_layer")
    return (out, cond) if want_cond else out


def fused_backward(row_ptr, col_idx, q, k, v, dout, H, Dh, scale, n_src=None,
                   want_cond=False):
    """Gradients of the fused layer for an upstream gradient ``dout``.
    Returns fp64 (dq [n_rows,H,Dh], dk [n_src,H,Dh], dv [n_src,H,Dh]) and,
    with ``want_cond``, their conditioning scales in the same shapes."""
    rp, ci = _c(row_ptr, np.int32), _c(col_idx, np.int32)
    qa, dt = _feat(q)
    ka, _ = _feat(k)
    va, _ = _feat(v)
    ga, _ = _feat(dout)
    n = rp.size - 1
    ns = (va.size // (H * Dh)) if n_src is None else int(n_src)
    dq = np.empty((n, H, Dh))
    dk = np.empty((ns, H, Dh))
    dv = np.empty((ns, H, Dh))
    conds = [np.empty_like(dq), np.empty_like(dk), np.empty_like(dv)] if want_cond else [None] * 3
    _check(_load().oracle_fused_backward(_p(rp), _p(ci), n, ns, H, Dh, float(scale), _p(qa),
                                         _p(ka), _p(va), _p(ga), dt, _p(dq), _p(dk), _p(dv),
                                         *[_p(c) for c in conds]), "oracle_fused_backward")
    return (dq, dk, dv, *conds) if want_cond else (dq, dk, dv)


def dense_block(w: dict, graphs=None, want_cond=False):
    """Dense-masked attention block on the arrays of ``workloads.make_dense``.
    Returns fp64 [n_sel,N,D] (and the conditioning scale when want_cond)."""
    B, N, D, H, P = (int(w[x]) for x in ("B", "N", "D", "H", "P"))
    f = lambda name: _c(w[name], np.float32)  # noqa: E731
    arrs = [f(x) for x in ("nodes", "pair_feats", "edge_mask", "ln_w", "ln_b")]
    wts = [f(x) for x in ("Wq", "Wk", "Wv", "W1", "b1", "W2", "b2", "Wout")]
    sel = None if graphs is None else _c(graphs, np.int64)
    n_sel = B if sel is None else sel.size
    out = np.empty((n_sel, N, D), dtype=np.float64)
    cond = np.empty_like(out) if want_cond else None
    _check(_load().oracle_dense_block(B, N, D, H, P, *[_p(a) for a in arrs],
                                      float(w["ln_eps"]), *[_p(a) for a in wts],
                                      _p(sel), n_sel, _p(out), _p(cond)), "oracle_dense_block")
    return (out, cond) if want_cond else out


def transpose(row_ptr, col_idx, n_src):
    """Edges grouped by source, each group in edge order: (src_ptr [n_src+1],
    perm [E], dst [E]) int32 arrays."""
    rp, ci = _c(row_ptr, np.int32), _c(col_idx, np.int32)
    n = rp.size - 1
    E = int(rp[-1]) if rp.size else 0
    sp = np.empty(int(n_src) + 1, dtype=np.int32)
    perm = np.empty(E, dtype=np.int32)
    dst = np.empty(E, dtype=np.int32)
    _check(_load().oracle_transpose(_p(rp), _p(ci), n, int(n_src), _p(sp), _p(perm), _p(dst)),
           "oracle_transpose")
    return sp, perm, dst


def fp8_decode(codes):
    """E4M3 codes (uint8) -> fp64 values."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _check(_load().oracle_fp8_decode(_p(c), c.size, _p(out)), "oracle_fp8_decode")
    return out


def fp8_encode(x):
    """fp32 values -> nearest E4M3 codes (ties to even, saturating at 448)."""
    a = _c(x, np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _check(_load().oracle_fp8_encode(_p(a), a.size, _p(out)), "oracle_fp8_encode")
    return out


def fp8_quantize(x, H, Dh):
    """Per (row, head) scaled E4M3 quantisation: (codes uint8 [n,H,Dh],
    scales fp32 [n,H])."""
    a, dt = _feat(x)
    n = a.size // (H * Dh)
    codes = np.empty((n, H, Dh), dtype=np.uint8)
    scales = np.empty((n, H), dtype=np.float32)
    _check(_load().oracle_fp8_quantize(_p(a), dt, n, H, Dh, _p(codes), _p(scales)),
           "oracle_fp8_quantize")
    return codes, scales


def fused_layer_fp8(row_ptr, col_idx, q, k8, ks, v8, vs, H, Dh, scale, rows=None,
                    want_cond=False):
    """Fused layer with E4M3 k/v tables and per (node, head) scales. fp64."""
    rp, ci = _c(row_ptr, np.int32), _c(col_idx, np.int32)
    qa, dt = _feat(q)
    k8c, v8c = _c(k8, np.uint8), _c(v8, np.uint8)
    ksc, vsc = _c(ks, np.float32), _c(vs, np.float32)
    sel = None if rows is None else _c(rows, np.int64)
    n = rp.size - 1
    n_sel = n if sel is None else sel.size
    out = np.empty((n_sel, H, Dh), dtype=np.float64)
    cond = np.empty_like(out) if want_cond else None
    _check(_load().oracle_fused_layer_fp8(_p(rp), _p(ci), n, H, Dh, float(scale), _p(qa), dt,
                                          _p(k8c), _p(ksc), _p(v8c), _p(vsc), _p(sel), n_sel,
                                          _p(out), _p(cond)), "oracle_fused_layer_fp8")
    return (out, cond) if want_cond else out


def plan(row_ptr, heavy_threshold, chunk):
    """Degree-bucket plan: (heavy_rows, chunk_start, chunk_row) int32 arrays."""
    rp = _c(row_ptr, np.int32)
    nh, nc = ctypes.c_int64(0), ctypes.c_int64(0)
    lib = _load()
    n = rp.size - 1
    _check(lib.oracle_plan(_p(rp), n, heavy_threshold, chunk, ctypes.byref(nh),
                           ctypes.byref(nc), None, None, None), "oracle_plan")
    hr = np.empty(nh.value, dtype=np.int32)
    cs = np.empty(nh.value + 1, dtype=np.int32)
    cr = np.empty(nc.value, dtype=np.int32)
    _check(lib.oracle_plan(_p(rp), n, heavy_threshold, chunk, ctypes.byref(nh),
                           ctypes.byref(nc), _p(hr), _p(cs), _p(cr)), "oracle_plan")
    return hr, cs, cr
