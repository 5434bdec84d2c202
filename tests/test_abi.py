"""CPU checks of the C ABI: libgat.so builds, loads, exports every entry point
declared in include/gat.h, and rejects host-checkable bad arguments before
touching the GPU. No compute call runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(gat_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gat_sddmm", "gat_edge_softmax", "gat_spmm_weighted", "gat_fused_layer",
                     "gat_dense_masked_attention", "gat_plan_create", "gat_plan_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_python_binding_covers_every_export(lib):
    import sparse_graph_attention_head_gb300 as gat
    assert sorted(gat.EXPORTS) == declared_functions()


def test_status_strings(lib):
    lib.gat_status_string.restype = ctypes.c_char_p
    assert lib.gat_status_string(0) == b"GAT_OK"
    assert lib.gat_status_string(5) == b"GAT_ERR_INDEX_OUT_OF_RANGE"
    assert lib.gat_version() > 0


def test_host_validation_rejects_bad_arguments(lib):
    """These return before any CUDA call, so they run without a GPU."""
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.gat_last_error.restype = ctypes.c_char_p
    # negative sizes
    lib.gat_fused_layer.argtypes = [P, P, I64, I64, I64, I32, I32, ctypes.c_float, P, P, P,
                                    ctypes.c_int, P, P, P, ctypes.c_size_t, P]
    assert lib.gat_fused_layer(None, None, -1, 0, 0, 8, 64, 0.125, None, None, None, 1, None,
                               None, None, 0, None) == 1
    assert b"bad sizes" in lib.gat_last_error()
    # unknown dtype
    assert lib.gat_fused_layer(None, None, 4, 4, 4, 8, 64, 0.125, None, None, None, 7, None,
                               None, None, 0, None) == 2
    # NULL pointers with work to do
    assert lib.gat_fused_layer(None, None, 4, 4, 4, 8, 64, 0.125, None, None, None, 1, None,
                               None, None, 0, None) == 1
    # empty problem is a no-op
    assert lib.gat_fused_layer(None, None, 0, 0, 0, 8, 64, 0.125, None, None, None, 1, None,
                               None, None, 0, None) == 0
    # unsupported dense shapes
    lib.gat_dense_masked_attention.argtypes = ([I32] * 5 + [P] * 5 + [ctypes.c_float] +
                                               [P] * 10 + [ctypes.c_size_t, P])
    args = [None] * 5 + [1e-5] + [None] * 10 + [0, None]
    assert lib.gat_dense_masked_attention(4, 40, 96, 4, 16, *args) == 2   # N > 32
    assert lib.gat_dense_masked_attention(4, 24, 90, 4, 16, *args) == 2   # D % H
    assert lib.gat_dense_masked_attention(-1, 24, 96, 4, 16, *args) == 1
    # the tensor-core shape needs a workspace; other shapes none
    lib.gat_dense_masked_attention_workspace_size.argtypes = [I32] * 4 + [P]
    n = ctypes.c_size_t(123)
    assert lib.gat_dense_masked_attention_workspace_size(24, 96, 4, 16, ctypes.byref(n)) == 0
    assert n.value >= 8 * 48 * 96 * 4  # the split Q|K|V|out weight images at least
    assert lib.gat_dense_masked_attention_workspace_size(7, 12, 3, 5, ctypes.byref(n)) == 0
    assert n.value == 0
    assert lib.gat_dense_masked_attention_workspace_size(0, 96, 4, 16, ctypes.byref(n)) == 1
    lib.gat_dense_masked_attention_status.argtypes = [P, P]
    assert lib.gat_dense_masked_attention_status(None, None) == 1
    # plan creation without an output handle
    lib.gat_plan_create.argtypes = [P, I64, I64, I32, I32, P, P]
    assert lib.gat_plan_create(None, 4, 4, 0, 0, None, None) == 1
    # sddmm bad head count
    lib.gat_sddmm.argtypes = [P, P, P, I64, I64, P, I64, P, I64, I32, I32, ctypes.c_float,
                              ctypes.c_int, P, P]
    assert lib.gat_sddmm(None, None, None, 0, 10, None, 4, None, 4, 0, 8, 1.0, 0, None,
                         None) == 1
    # softmax empty graph is a no-op
    lib.gat_edge_softmax.argtypes = [P, I64, I64, I32, P, P, P, P]
    assert lib.gat_edge_softmax(None, 0, 0, 4, None, None, None, None) == 0


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    """Importing the binding with libgat.so absent raises instead of falling back."""
    import importlib.util
    src = os.path.join(ROOT, "sparse_graph_attention_head_gb300", "__init__.py")
    pkg = tmp_path / "gatcopy"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("gatcopy", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="libgat.so is not built"):
        spec.loader.exec_module(mod)


def test_oracle_is_not_imported_by_the_product():
    pkg = os.path.join(ROOT, "sparse_graph_attention_head_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.c" not in text, f
