"""The C-ABI library builds, loads and exports every declared entry point (no GPU).

Only host-side argument checks are exercised here: each call below returns
before any CUDA work is issued.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gnn.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_aggregation_dense_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gnn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gnn_graph_create", "gnn_graph_destroy", "gnn_halo_pull", "gnn_halo_push",
                     "gnn_layer_forward", "gnn_layer_backward", "gnn_get_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_export():
    from sparse_aggregation_dense_gb300 import gnn

    assert sorted(gnn.EXPORTS) == declared_functions()


def test_host_side_argument_checks(lib):
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.gnn_graph_create.argtypes = [vp, vp, i64, i64, i64, vp, ctypes.c_int, vp, ctypes.POINTER(vp)]
    out = vp(1234)
    # NULL rowptr, negative sizes, bad aggregation kind: rejected before any CUDA call
    assert lib.gnn_graph_create(None, None, 4, 0, 0, None, 0, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert lib.gnn_graph_create(vp(16), None, -1, 0, 0, None, 0, None, ctypes.byref(out)) == 1
    assert lib.gnn_graph_create(vp(16), vp(16), 4, 0, 4, None, 7, None, ctypes.byref(out)) == 1
    assert lib.gnn_graph_create(vp(16), vp(16), 4, 0, 4, None, 0, None, None) == 1
    assert lib.gnn_graph_create(vp(16), vp(16), 1 << 31, 0, 4, None, 0, None, ctypes.byref(out)) == 4
    lib.gnn_graph_destroy.argtypes = [vp]
    assert lib.gnn_graph_destroy(None) == 1
    lib.gnn_get_error.argtypes = [vp]
    assert lib.gnn_get_error(None) == 1
    lib.gnn_halo_pull.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, ctypes.c_int, vp]
    assert lib.gnn_halo_pull(None, vp(16), 8, 10, vp(16), vp(16), 8, 8, 0, None) == 1
    lib.gnn_layer_forward.argtypes = [vp, vp, i64, i64, vp, i64, ctypes.c_int, vp, i64, vp, i64, ctypes.c_int, vp]
    assert lib.gnn_layer_forward(None, vp(16), 8, 8, vp(16), 8, 1, vp(16), 8, vp(16), 8, 0, None) == 1
    lib.gnn_sage_half_offset.argtypes = [i64, ctypes.c_int]
    lib.gnn_sage_half_offset.restype = i64
    assert lib.gnn_sage_half_offset(100, 1) == 104
    assert lib.gnn_sage_half_offset(100, 0) == 100
    assert lib.gnn_sage_half_offset(41, 0) == 44
    lib.gnn_status_string.restype = ctypes.c_char_p
    assert lib.gnn_status_string(5) == b"bad index data on the device"
    assert lib.gnn_status_string(6) == b"a bounded wait on the device ran out"
    lib.gnn_last_cuda_error.restype = ctypes.c_char_p
    assert isinstance(lib.gnn_last_cuda_error(), bytes) and lib.gnn_last_cuda_error()


def test_binding_reports_cuda_error_text():
    # the Python binding returns the library's static text, not a raw pointer
    from sparse_aggregation_dense_gb300 import gnn
    assert isinstance(gnn.last_cuda_error(), str) and gnn.last_cuda_error()
    err = gnn.GnnError(gnn.GNN_ECUDA, "call")
    assert str(err).startswith("call: CUDA runtime error (status 3): ")
