"""The aggregation entry point that allocates nothing (gnn_aggregate_forward_noalloc).

Some callers cannot allocate device memory where they aggregate (their memory
is reserved by another allocator, or they must not pay for the device-wide
synchronisation cudaMalloc can cause).  For them the library offers a variant
of the forward aggregation whose heavy-row partial sums live in a fixed array
inside the library.  These tests call it through the C ABI and compare it with
the Z of the ordinary forward layer call, on two calls in a row (the second call
reuses the array the first one left behind), and check that a width whose
partials do not fit is rejected before anything runs.

This file is collected last on purpose: a failure here does not hide the rest
of the suite in a run that stops at the first failure.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from synth.configs import WORKLOADS
from sparse_aggregation_dense_gb300 import gnn, padded
from tests._gpu import TOL, assert_ok, close, gen_matrix, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rmat_graph():
    part = WORKLOADS["rmat131k"].make(0)  # hub rows: ~3000 heavy-row chunks
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda(), "gcn")
    return part, g


@pytest.mark.parametrize("dt,f", [("bf16", 128), ("f32", 256)])
def test_noalloc_matches_layer_forward_twice(rmat_graph, dt, f):
    part, g = rmat_graph
    tdt = torch_dtype(dt)
    H = to_device(gen_matrix(part.n_total, f, dt, 0, 123), dt, f)
    W = torch.from_numpy(synth.glorot(f, 16, 0, 7)).cuda()
    Z_ref = padded(part.n_local, f, tdt, "cuda")
    H_out = padded(part.n_local, 16, tdt, "cuda")
    gnn.layer_forward(g, H, W, True, Z_ref, H_out)
    ref = to_host(Z_ref)
    for call in range(2):
        Z = padded(part.n_local, f, tdt, "cuda")
        Z.fill_(float("nan"))
        gnn.aggregate_forward_noalloc(g, H, Z)
        assert_ok(g)
        got = to_host(Z)
        close(got, ref, TOL[dt], f"no-alloc Z, call {call + 1}")
        assert np.array_equal(got, ref)  # same kernels, same order: identical bits


def test_noalloc_rejects_partials_beyond_its_array(rmat_graph):
    _, g = rmat_graph
    lib = gnn._lib()
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    ptr = ctypes.c_void_p(dummy.data_ptr())
    # 2048 bf16 columns: ~3000 chunks x 2048 x 4 bytes > 16 MiB
    st = lib.gnn_aggregate_forward_noalloc(ctypes.c_void_p(g.handle), ptr, 2048, 2048, ptr, 2048, gnn.GNN_BF16,
                                           None)
    assert st == gnn.GNN_EUNSUPPORTED
    assert_ok(g)
