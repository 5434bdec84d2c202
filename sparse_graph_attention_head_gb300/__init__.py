"""Multi-head graph attention over CSR graphs on GB300 (sm_103a).

Thin ctypes binding over ``libgat.so`` (C ABI declared in ``include/gat.h``).
Each function has the name of its C entry point and only marshals arguments:
torch tensors on the GPU become device pointers, the current torch CUDA stream
becomes the ``stream`` argument, and a non-zero status raises ``GatError``.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU path. PyTorch is used only for device memory and streams.

Importing this package loads ``libgat.so`` and fails loudly when it has not
been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgat.so")

GAT_F32, GAT_BF16 = 0, 1
_STATUS = {0: "GAT_OK", 1: "GAT_ERR_INVALID_ARG", 2: "GAT_ERR_UNSUPPORTED", 3: "GAT_ERR_CUDA",
           4: "GAT_ERR_WORKSPACE", 5: "GAT_ERR_INDEX_OUT_OF_RANGE", 6: "GAT_ERR_PLAN_MISMATCH"}

#: every entry point declared in include/gat.h
EXPORTS = (
    "gat_status_string", "gat_last_error", "gat_version",
    "gat_plan_create", "gat_plan_destroy", "gat_plan_info", "gat_plan_export",
    "gat_validate_graph", "gat_sddmm", "gat_edge_softmax", "gat_spmm_weighted",
    "gat_fused_layer_workspace_size", "gat_fused_layer", "gat_dense_masked_attention",
    "gat_fused_layer_no_alloc",
    "gat_transpose_create", "gat_transpose_destroy", "gat_transpose_info", "gat_transpose_export",
    "gat_fused_layer_backward_workspace_size", "gat_fused_layer_backward",
    "gat_quantize_fp8", "gat_fused_layer_fp8", "gat_spmm_weighted_workspace_size",
    "gat_dense_masked_attention_workspace_size", "gat_dense_masked_attention_status",
    "gat_partition_rows", "gat_rebase_row_ptr", "gat_softmax_aggregate",
)


class GatError(RuntimeError):
    """A libgat entry point returned a non-zero status."""

    def __init__(self, fn: str, code: int, detail: str):
        super().__init__(f"{fn}: {_STATUS.get(code, code)}: {detail}")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libgat.so is not built ({LIB_PATH} missing); build it with "
            "python sparse_graph_attention_head_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, F, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                          ctypes.c_size_t)
    sigs = {
        "gat_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "gat_last_error": ([], ctypes.c_char_p),
        "gat_version": ([], I32),
        "gat_plan_create": ([P, I64, I64, I32, I32, P, P], ctypes.c_int),
        "gat_plan_destroy": ([P], ctypes.c_int),
        "gat_plan_info": ([P, P, P, P, P, P, P], ctypes.c_int),
        "gat_plan_export": ([P, P, P, P, P], ctypes.c_int),
        "gat_validate_graph": ([P, P, I64, I64, I64, P, P], ctypes.c_int),
        "gat_sddmm": ([P, P, P, I64, I64, P, I64, P, I64, I32, I32, F, ctypes.c_int, P, P],
                      ctypes.c_int),
        "gat_edge_softmax": ([P, I64, I64, I32, P, P, P, P], ctypes.c_int),
        "gat_spmm_weighted": ([P, P, I64, I64, I64, I32, I32, P, P, ctypes.c_int, P, P, P, SZ,
                               P], ctypes.c_int),
        "gat_spmm_weighted_workspace_size": ([P, I32, I32, P], ctypes.c_int),
        "gat_fused_layer_workspace_size": ([P, I32, I32, P], ctypes.c_int),
        "gat_fused_layer": ([P, P, I64, I64, I64, I32, I32, F, P, P, P, ctypes.c_int, P, P, P, SZ,
                             P], ctypes.c_int),
        "gat_dense_masked_attention": ([I32] * 5 + [P] * 5 + [F] + [P] * 8 + [P, P, SZ, P],
                                       ctypes.c_int),
        "gat_dense_masked_attention_workspace_size": ([I32, I32, I32, I32, P], ctypes.c_int),
        "gat_dense_masked_attention_status": ([P, P], ctypes.c_int),
        "gat_partition_rows": ([P, I64, I32, P], ctypes.c_int),
        "gat_softmax_aggregate": ([P, P, I64, I64, I64, I32, I32, P, P, ctypes.c_int, P, P, P, SZ,
                                   P], ctypes.c_int),
        "gat_rebase_row_ptr": ([P, I64, I64, P, P], ctypes.c_int),
        "gat_fused_layer_no_alloc": ([P, P, I64, I64, I64, I32, I32, F, P, P, P, ctypes.c_int, P,
                                      P], ctypes.c_int),
        "gat_transpose_create": ([P, P, I64, I64, I64, P, P], ctypes.c_int),
        "gat_transpose_destroy": ([P], ctypes.c_int),
        "gat_transpose_info": ([P, P, P, P, P, P], ctypes.c_int),
        "gat_transpose_export": ([P, P, P, P, P], ctypes.c_int),
        "gat_fused_layer_backward_workspace_size": ([P, I64, I64, I32, I32, P], ctypes.c_int),
        "gat_quantize_fp8": ([P, ctypes.c_int, I64, I32, I32, P, P, P], ctypes.c_int),
        "gat_fused_layer_fp8": ([P, P, I64, I64, I64, I32, I32, F, P, ctypes.c_int, P, P, P, P, P,
                                 P, P, SZ, P], ctypes.c_int),
        "gat_fused_layer_backward": ([P, P, I64, I64, I64, I32, I32, F, P, P, P, P, ctypes.c_int,
                                      P, P, P, P, P, P, SZ, P], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    """The loaded libgat handle."""
    return _lib


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------
def _check(fn: str, code: int) -> None:
    if code != 0:
        raise GatError(fn, code, _lib.gat_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libgat takes device tensors only")
    if not t.is_contiguous():
        raise ValueError("libgat takes contiguous tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GAT_F32
    if t.dtype == torch.bfloat16:
        return GAT_BF16
    raise ValueError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _idx(t, name):
    if t is not None and t.dtype != torch.int32:
        raise ValueError(f"{name} must be int32")
    return t


# ----------------------------------------------------------------------------
# plan
# ----------------------------------------------------------------------------
class Plan:
    """Degree-bucket plan of one graph (``gat_plan_create``). Owns device
    arrays; freed by ``destroy()`` or when garbage-collected."""

    def __init__(self, row_ptr: torch.Tensor, n_edges: int | None = None,
                 heavy_threshold: int = 0, chunk_edges: int = 0, stream=None):
        _idx(row_ptr, "row_ptr")
        n_rows = row_ptr.numel() - 1
        if n_edges is None:
            n_edges = int(row_ptr[-1].item())
        h = ctypes.c_void_p()
        _check("gat_plan_create", _lib.gat_plan_create(
            _ptr(row_ptr), n_rows, n_edges, heavy_threshold, chunk_edges, _stream(stream),
            ctypes.byref(h)))
        self.handle = h.value
        self.device = row_ptr.device

    def info(self) -> dict:
        vals = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32(),
                ctypes.c_int64(), ctypes.c_int64()]
        _check("gat_plan_info", _lib.gat_plan_info(self.handle, *[ctypes.byref(v) for v in vals]))
        keys = ("n_rows", "n_edges", "heavy_threshold", "chunk_edges", "n_heavy", "n_chunks")
        return {k: v.value for k, v in zip(keys, vals)}

    def export(self, stream=None):
        """(heavy_rows, chunk_start, chunk_row) as int32 device tensors."""
        inf = self.info()
        hr = torch.empty(inf["n_heavy"], dtype=torch.int32, device=self.device)
        cs = torch.empty(inf["n_heavy"] + 1, dtype=torch.int32, device=self.device)
        cr = torch.empty(inf["n_chunks"], dtype=torch.int32, device=self.device)
        _check("gat_plan_export", _lib.gat_plan_export(
            self.handle, _ptr(hr) if hr.numel() else None, _ptr(cs),
            _ptr(cr) if cr.numel() else None, _stream(stream)))
        return hr, cs, cr

    def destroy(self):
        if getattr(self, "handle", None):
            _lib.gat_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def gat_plan_create(row_ptr, n_edges=None, heavy_threshold=0, chunk_edges=0, stream=None) -> Plan:
    return Plan(row_ptr, n_edges, heavy_threshold, chunk_edges, stream)


def _plan_handle(plan):
    return None if plan is None else plan.handle


# ----------------------------------------------------------------------------
# operations
# ----------------------------------------------------------------------------
def gat_validate_graph(row_ptr, col_idx, n_src, n_edges=None, flag=None, stream=None) -> None:
    """Raise GatError(GAT_ERR_INDEX_OUT_OF_RANGE) for a malformed graph."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    if n_edges is None:
        n_edges = col_idx.numel() if col_idx is not None else int(row_ptr[-1].item())
    if flag is None:
        flag = torch.empty(1, dtype=torch.int32, device=row_ptr.device)
    _check("gat_validate_graph", _lib.gat_validate_graph(
        _ptr(row_ptr), _ptr(col_idx), row_ptr.numel() - 1, n_src, n_edges, _ptr(flag),
        _stream(stream)))


def gat_sddmm(src_idx, src_feat, dst_feat, H, Dh, scale=1.0, dst_idx=None, row_ptr=None,
              out=None, stream=None):
    """out[e,h] = scale * <src_feat[src(e),h,:], dst_feat[dst(e),h,:]> (fp32 [E,H])."""
    _idx(src_idx, "src_idx")
    _idx(dst_idx, "dst_idx")
    _idx(row_ptr, "row_ptr")
    E = src_idx.numel()
    if out is None:
        out = torch.empty((E, H), dtype=torch.float32, device=src_idx.device)
    n_rows = 0 if row_ptr is None else row_ptr.numel() - 1
    _check("gat_sddmm", _lib.gat_sddmm(
        _ptr(row_ptr), _ptr(src_idx), _ptr(dst_idx), n_rows, E, _ptr(src_feat),
        src_feat.numel() // (H * Dh), _ptr(dst_feat), dst_feat.numel() // (H * Dh), H, Dh,
        float(scale), _dtype(src_feat), _ptr(out) if E else None, _stream(stream)))
    return out


def gat_edge_softmax(row_ptr, scores, H, out=None, plan=None, stream=None):
    """Per-row, per-head softmax of scores [E,H] (fp32); out may be scores."""
    _idx(row_ptr, "row_ptr")
    if out is None:
        out = torch.empty_like(scores)
    E = scores.numel() // H
    _check("gat_edge_softmax", _lib.gat_edge_softmax(
        _ptr(row_ptr), row_ptr.numel() - 1, E, H, _ptr(scores) if E else None,
        _ptr(out) if E else None, _plan_handle(plan), _stream(stream)))
    return out


def gat_spmm_weighted_workspace_size(plan, H, Dh) -> int:
    n = ctypes.c_size_t()
    _check("gat_spmm_weighted_workspace_size",
           _lib.gat_spmm_weighted_workspace_size(_plan_handle(plan), H, Dh, ctypes.byref(n)))
    return n.value


def gat_spmm_weighted(row_ptr, col_idx, w, feat, H, Dh, n_rows=None, out=None, plan=None,
                      workspace=None, no_workspace=False, stream=None):
    """out[i,h,:] = sum_e w[e,h] feat[col_idx[e],h,:]; out has feat's dtype.
    With a plan, heavy rows run as chunks through ``workspace`` (allocated
    here when None); ``no_workspace=True`` passes none (a block per heavy row)."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows = row_ptr.numel() - 1 if n_rows is None else n_rows
    E = col_idx.numel()
    if out is None:
        out = torch.empty((n_rows, H, Dh), dtype=feat.dtype, device=feat.device)
    if no_workspace:
        workspace = None
    elif plan is not None and workspace is None:
        need = gat_spmm_weighted_workspace_size(plan, H, Dh)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=feat.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("gat_spmm_weighted", _lib.gat_spmm_weighted(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, feat.numel() // (H * Dh), E, H, Dh,
        _ptr(w) if E else None, _ptr(feat), _dtype(feat), _ptr(out), _plan_handle(plan),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def gat_softmax_aggregate(row_ptr, col_idx, scores, feat, H, Dh, n_rows=None, out=None,
                          plan=None, workspace=None, stream=None):
    """out[i,h,:] = sum_e softmax_e(scores[:,h]) feat[col_idx[e],h,:], one pass;
    scores fp32 [E,H], feat [n_src,H,Dh], out has feat's dtype."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows = row_ptr.numel() - 1 if n_rows is None else n_rows
    E = col_idx.numel()
    if out is None:
        out = torch.empty((n_rows, H, Dh), dtype=feat.dtype, device=feat.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if plan is not None and workspace is None:
        need = gat_fused_layer_workspace_size(plan, H, Dh)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=feat.device)
            ws_bytes = need
    _check("gat_softmax_aggregate", _lib.gat_softmax_aggregate(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, feat.numel() // (H * Dh), E, H, Dh,
        _ptr(scores) if E else None, _ptr(feat), _dtype(feat), _ptr(out), _plan_handle(plan),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def gat_fused_layer_workspace_size(plan, H, Dh) -> int:
    n = ctypes.c_size_t()
    _check("gat_fused_layer_workspace_size",
           _lib.gat_fused_layer_workspace_size(_plan_handle(plan), H, Dh, ctypes.byref(n)))
    return n.value


def gat_fused_layer(row_ptr, col_idx, q, k, v, scale, out=None, plan=None, workspace=None,
                    stream=None):
    """Fused SDDMM -> edge softmax -> SpMM. q/out [n_rows,H,Dh], k/v [n_src,H,Dh]."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows, H, Dh = q.shape
    E = col_idx.numel()
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if plan is not None and workspace is None:
        need = gat_fused_layer_workspace_size(plan, H, Dh)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            ws_bytes = need
    _check("gat_fused_layer", _lib.gat_fused_layer(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, k.shape[0], E, H, Dh, float(scale),
        _ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(out), _plan_handle(plan),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def gat_fused_layer_no_alloc(row_ptr, col_idx, q, k, v, scale, out, stream=None):
    """gat_fused_layer for callers that cannot allocate device memory: the
    plan and chunk states live in the library's static device scratch, so the
    caller provides only the inputs and the preallocated ``out``. Calls that
    overlap on the GPU race on that scratch; see include/gat.h."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows, H, Dh = q.shape
    E = col_idx.numel()
    _check("gat_fused_layer_no_alloc", _lib.gat_fused_layer_no_alloc(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, k.shape[0], E, H, Dh, float(scale),
        _ptr(q), _ptr(k), _ptr(v), _dtype(q), _ptr(out), _stream(stream)))
    return out


def gat_quantize_fp8(x, codes=None, scales=None, stream=None):
    """Per (node, head) scaled E4M3 quantisation of x [n,H,Dh]: returns
    (codes uint8 [n,H,Dh], scales fp32 [n,H])."""
    n, H, Dh = x.shape
    codes = torch.empty((n, H, Dh), dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty((n, H), dtype=torch.float32, device=x.device) if scales is None else scales
    _check("gat_quantize_fp8", _lib.gat_quantize_fp8(
        _ptr(x), _dtype(x), n, H, Dh, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def gat_fused_layer_fp8(row_ptr, col_idx, q, k8, k_scale, v8, v_scale, scale, out=None,
                        plan=None, workspace=None, stream=None):
    """gat_fused_layer with E4M3 k/v tables and per (node, head) scales."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows, H, Dh = q.shape
    E = col_idx.numel()
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if plan is not None and workspace is None:
        need = gat_fused_layer_workspace_size(plan, H, Dh)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            ws_bytes = need
    _check("gat_fused_layer_fp8", _lib.gat_fused_layer_fp8(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, k8.shape[0], E, H, Dh, float(scale),
        _ptr(q), _dtype(q), _ptr(k8), _ptr(k_scale), _ptr(v8), _ptr(v_scale), _ptr(out),
        _plan_handle(plan), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


class Transpose:
    """Source-major view of one graph (``gat_transpose_create``): for every
    source, the edges that read it, in edge order. Owns device arrays."""

    def __init__(self, row_ptr: torch.Tensor, col_idx: torch.Tensor, n_src: int, stream=None):
        _idx(row_ptr, "row_ptr")
        _idx(col_idx, "col_idx")
        n_rows, E = row_ptr.numel() - 1, col_idx.numel()
        h = ctypes.c_void_p()
        _check("gat_transpose_create", _lib.gat_transpose_create(
            _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, n_src, E, _stream(stream),
            ctypes.byref(h)))
        self.handle = h.value
        self.device = row_ptr.device

    def info(self) -> dict:
        vals = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(),
                ctypes.c_int64()]
        _check("gat_transpose_info",
               _lib.gat_transpose_info(self.handle, *[ctypes.byref(v) for v in vals]))
        keys = ("n_rows", "n_src", "n_edges", "max_src_degree", "n_heavy_src")
        return {k: v.value for k, v in zip(keys, vals)}

    def export(self, stream=None):
        """(src_ptr, perm, dst) as int32 device tensors."""
        inf = self.info()
        sp = torch.empty(inf["n_src"] + 1, dtype=torch.int32, device=self.device)
        perm = torch.empty(inf["n_edges"], dtype=torch.int32, device=self.device)
        dst = torch.empty(inf["n_edges"], dtype=torch.int32, device=self.device)
        e = inf["n_edges"] > 0
        _check("gat_transpose_export", _lib.gat_transpose_export(
            self.handle, _ptr(sp), _ptr(perm) if e else None, _ptr(dst) if e else None,
            _stream(stream)))
        return sp, perm, dst

    def destroy(self):
        if getattr(self, "handle", None):
            _lib.gat_transpose_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def gat_transpose_create(row_ptr, col_idx, n_src, stream=None) -> Transpose:
    return Transpose(row_ptr, col_idx, n_src, stream)


def gat_fused_layer_backward_workspace_size(plan, n_rows, n_edges, H, Dh) -> int:
    n = ctypes.c_size_t()
    _check("gat_fused_layer_backward_workspace_size",
           _lib.gat_fused_layer_backward_workspace_size(_plan_handle(plan), n_rows, n_edges, H, Dh,
                                                        ctypes.byref(n)))
    return n.value


def gat_fused_layer_backward(row_ptr, col_idx, q, k, v, dout, scale, transpose, plan=None,
                             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of gat_fused_layer for the upstream gradient
    ``dout`` [n_rows,H,Dh]; ``transpose`` from gat_transpose_create."""
    _idx(row_ptr, "row_ptr")
    _idx(col_idx, "col_idx")
    n_rows, H, Dh = q.shape
    n_src, E = k.shape[0], col_idx.numel()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        need = gat_fused_layer_backward_workspace_size(plan, n_rows, E, H, Dh)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("gat_fused_layer_backward", _lib.gat_fused_layer_backward(
        _ptr(row_ptr), _ptr(col_idx) if E else None, n_rows, n_src, E, H, Dh, float(scale),
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _dtype(q), _ptr(dq), _ptr(dk), _ptr(dv),
        _plan_handle(plan), transpose.handle, _ptr(workspace), ws_bytes, _stream(stream)))
    return dq, dk, dv


def gat_dense_masked_attention_workspace_size(N, D, H, P) -> int:
    n = ctypes.c_size_t()
    _check("gat_dense_masked_attention_workspace_size",
           _lib.gat_dense_masked_attention_workspace_size(N, D, H, P, ctypes.byref(n)))
    return n.value


def gat_dense_masked_attention(nodes, pair_feats, edge_mask, ln_w, ln_b, ln_eps, Wq, Wk, Wv,
                               W1, b1, W2, b2, Wout, H, out=None, workspace=None, stream=None):
    """Dense-masked small-graph attention block (fp32). nodes [B,N,D]. The
    tensor-core shape needs ``workspace`` (allocated here when None)."""
    B, N, D = nodes.shape
    P = pair_feats.shape[-1]
    if out is None:
        out = torch.empty_like(nodes)
    if workspace is None:
        need = gat_dense_masked_attention_workspace_size(N, D, H, P)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=nodes.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("gat_dense_masked_attention", _lib.gat_dense_masked_attention(
        B, N, D, H, P, _ptr(nodes), _ptr(pair_feats), _ptr(edge_mask), _ptr(ln_w), _ptr(ln_b),
        float(ln_eps), _ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
        _ptr(Wout), _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def gat_dense_masked_attention_status(workspace, stream=None) -> None:
    """Raise GatError when the last tensor-core call with ``workspace`` gave up
    a bounded wait (synchronises the stream)."""
    _check("gat_dense_masked_attention_status",
           _lib.gat_dense_masked_attention_status(_ptr(workspace), _stream(stream)))


def gat_partition_rows(row_ptr, parts: int):
    """Contiguous row ranges of about equal fused-layer traffic (host call on a
    host int32 row_ptr, numpy or CPU tensor); returns row_begin (int64,
    parts + 1 entries)."""
    import numpy as np
    rp = np.ascontiguousarray(row_ptr.numpy() if isinstance(row_ptr, torch.Tensor) else row_ptr,
                              dtype=np.int32)
    out = np.empty(parts + 1, dtype=np.int64)
    _check("gat_partition_rows", _lib.gat_partition_rows(
        rp.ctypes.data, rp.size - 1, parts, out.ctypes.data))
    return out


def gat_rebase_row_ptr(row_ptr, r0: int, r1: int, out=None, stream=None):
    """row_ptr[r0:r1+1] - row_ptr[r0] on the device (rows [r0, r1) as a graph)."""
    _idx(row_ptr, "row_ptr")
    if out is None:
        out = torch.empty(r1 - r0 + 1, dtype=torch.int32, device=row_ptr.device)
    _check("gat_rebase_row_ptr", _lib.gat_rebase_row_ptr(_ptr(row_ptr), r0, r1, _ptr(out),
                                                         _stream(stream)))
    return out


def version() -> int:
    return int(_lib.gat_version())
