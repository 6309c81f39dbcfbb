"""The aggregation entry point that allocates nothing (gnn_aggregate_forward_noalloc).

Some callers cannot allocate device memory where they aggregate (their memory
is reserved by another allocator, or they must not pay for the device-wide
synchronisation cudaMalloc can cause).  For them the library offers a variant
of the forward aggregation whose heavy-row partial sums live in a fixed array
inside the library.  These tests call it through the C ABI and compare it with
the Z of the ordinary forward layer call and with the oracle, on two calls in a
row (the second call reuses the array the first one left behind), for GCN and
GraphSAGE graphs; check that the calls leave the device's free memory
unchanged; and check that a width whose partials do not fit is rejected before
anything runs.

This file is collected last on purpose: a failure here does not hide the rest
of the suite in a run that stops at the first failure.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.configs import WORKLOADS
from sparse_aggregation_dense_gb300 import gnn, padded
from tests._gpu import TOL, assert_ok, close, gen_matrix, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

HEAVY, CHUNK = 512, 512        # rows longer than HEAVY entries are summed in CHUNK-entry pieces
SCRATCH_BYTES = 16 << 20       # the entry point's fixed array


def _chunks(rowptr: np.ndarray) -> int:
    d = np.diff(rowptr.astype(np.int64))
    heavy = d[d > HEAVY]
    return int(((heavy + CHUNK - 1) // CHUNK).sum())


@pytest.fixture(scope="module", params=["gcn", "sage"])
def graph(request):
    agg = request.param
    if agg == "gcn":
        part = WORKLOADS["rmat131k"].make(0)  # hub rows: a few thousand heavy-row chunks
    else:
        part = synth.chunglu_partition(8000, 200000, 50.0, 2, seed=9, cap_frac=0.25)  # power law: 28 rows past the split
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda(), agg)
    assert _chunks(part.rowptr) > 0  # the fixed array is really used
    return agg, part, g


@pytest.mark.parametrize("dt,f", [("bf16", 128), ("f32", 256), ("bf16", 100)])
def test_noalloc_matches_layer_forward_and_oracle_twice(graph, dt, f):
    agg, part, g = graph
    tdt = torch_dtype(dt)
    sage = agg == "sage"
    half = gnn.sage_half_offset(f, tdt)
    Kp = 2 * half if sage else f
    H_h = gen_matrix(part.n_total, f, dt, 0, 123)
    H = to_device(H_h, dt, f)
    W = torch.from_numpy(synth.glorot(2 * f if sage else f, 16, 0, 7)).cuda()
    Z_ref = padded(part.n_local, Kp, tdt, "cuda")
    H_out = padded(part.n_local, 16, tdt, "cuda")
    gnn.layer_forward(g, H, W, True, Z_ref, H_out)
    assert_ok(g)
    ref = to_host(Z_ref)
    # the oracle's aggregation of the same rows (compact [self | mean] layout for GraphSAGE)
    Zo = oracle.aggregate(part, oracle.widen(H_h[:, :f], dt == "bf16"), f, agg)
    Zo = oracle.round_bf16(Zo) if dt == "bf16" else Zo
    torch.cuda.synchronize()
    for call in range(2):
        Z = padded(part.n_local, Kp, tdt, "cuda")
        Z.fill_(float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        gnn.aggregate_forward_noalloc(g, H, Z)
        assert_ok(g)
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, f"call {call + 1} changed free device memory by {free0 - free1} bytes"
        got = to_host(Z)
        assert np.array_equal(got, ref), f"call {call + 1}"  # same kernels, same order: identical bits
        if sage:
            close(got[:, :f], Zo[:, :f], 0.0, f"self half, call {call + 1}")
            close(got[:, half:half + f], Zo[:, f:], TOL[dt], f"mean half, call {call + 1}")
        else:
            close(got, Zo, TOL[dt], f"no-alloc Z, call {call + 1}")


def test_noalloc_rejects_partials_beyond_its_array(graph):
    agg, part, g = graph
    if agg != "gcn":
        pytest.skip("one graph suffices for the size check")
    f = 2048  # bf16 columns: the partials need chunks x 2048 x 4 bytes
    chunks = _chunks(part.rowptr)
    assert chunks * f * 4 > SCRATCH_BYTES, chunks  # so the call can only be rejected
    # buffers of full valid size all the same: the rejection is about the array, not the arguments
    H = padded(part.n_total, f, torch.bfloat16, "cuda")
    Z = padded(part.n_local, f, torch.bfloat16, "cuda")
    lib = gnn._lib()
    st = lib.gnn_aggregate_forward_noalloc(ctypes.c_void_p(g.handle), ctypes.c_void_p(H.data_ptr()), H.stride(0), f,
                                           ctypes.c_void_p(Z.data_ptr()), Z.stride(0), gnn.GNN_BF16, None)
    assert st == gnn.GNN_EUNSUPPORTED
    assert_ok(g)
