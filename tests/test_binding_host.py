"""Host-side logic of the binding and of the epoch drivers, with no GPU: the
library is replaced by a recorder that accepts every call, so these tests
check (1) that the binding's buffer checks accept the shapes the drivers
really pass and reject undersized or mistyped buffers before any device work,
and (2) the order of the library calls of one epoch for the sequential,
multi-partition "sync" and "stale" schedules."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_aggregation_dense_gb300 import MultiPartitionTrainer, PartitionModel, gnn
from sparse_aggregation_dense_gb300.partition_model import padded
from tests._problems import partition_from_dense, random_sym_adjacency


class _Recorder:
    """Stands in for libgnn: every entry point returns GNN_OK and is logged."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("gnn_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append(name)
            if name == "gnn_graph_create":
                args[-1]._obj.value = 0x1000 + len(self.calls)
            if name == "gnn_sage_half_offset":
                f, dt = int(args[0]), int(args[1])
                m = 8 if dt == gnn.GNN_BF16 else 4
                return (f + m - 1) // m * m
            if name in ("gnn_status_string", "gnn_last_cuda_error"):
                return b"recorded"
            return gnn.GNN_OK

        return fn


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder()
    created = []
    real_create = gnn.graph_create

    def create(*args, **kw):
        g = real_create(*args, **kw)
        created.append(g)
        return g

    monkeypatch.setattr(gnn, "_L", rec)
    monkeypatch.setattr(gnn, "_ptr", lambda t: None if t is None else ctypes.c_void_p(t.data_ptr()))
    monkeypatch.setattr(gnn, "_stream", lambda: 0)
    monkeypatch.setattr(gnn, "graph_create", create)
    yield rec
    for g in created:  # recorded handles must never reach the real library's destroy
        g.handle = None


def _parts(P, N=60, seed=3):
    A = random_sym_adjacency(N, 0.12, seed)
    blocks = np.array_split(np.random.default_rng(seed).permutation(N), P)
    return [partition_from_dense(A, np.sort(b))[0] for b in blocks], N


def _model(agg="gcn", dtype=torch.float32, narrow=False, widths=(12, 16, 6), grad_dtype=torch.float32):
    parts, N = _parts(2)
    part = parts[0]
    assert part.n_halo > 0
    return PartitionModel(part, list(widths), agg, dtype, "cpu", narrow=narrow, grad_dtype=grad_dtype), part


def test_model_rejects_unsupported_precision_pairs():
    with pytest.raises(ValueError):
        _model(dtype=torch.float32, grad_dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _model(dtype=torch.bfloat16, narrow=True, grad_dtype=torch.float32)


@pytest.mark.parametrize("agg,dtype,narrow,grad_dtype", [("gcn", torch.float32, False, torch.float32),
                                                         ("gcn", torch.bfloat16, True, torch.bfloat16),
                                                         ("gcn", torch.bfloat16, False, torch.float32),
                                                         ("sage", torch.bfloat16, False, torch.float32),
                                                         ("sage", torch.bfloat16, False, torch.bfloat16),
                                                         ("sage", torch.float32, False, torch.float32)])
def test_partition_epoch_passes_the_binding_checks(lib, agg, dtype, narrow, grad_dtype):
    m, part = _model(agg, dtype, narrow, widths=(12, 20, 16, 6), grad_dtype=grad_dtype)
    for l in range(m.L):
        m.tables[l] = padded(part.n_table, m.widths[l], dtype, "cpu")
    lib.calls.clear()
    m.step()
    m.check_errors()
    fwd = "gnn_layer_forward_narrow" if narrow else "gnn_layer_forward"
    n_narrow = sum(m.narrow)
    assert lib.calls.count("gnn_layer_forward") + lib.calls.count("gnn_layer_forward_narrow") == m.L
    assert lib.calls.count("gnn_layer_forward_narrow") == n_narrow
    assert lib.calls.count("gnn_halo_push") == m.L - 1
    assert lib.calls.count("gnn_halo_pull") == (m.L if part.n_halo else 0)
    assert lib.calls.count("gnn_softmax_ce") == 1
    assert lib.calls.count("gnn_layer_backward") + lib.calls.count("gnn_layer_backward_narrow") == m.L
    # pull of layer l before its forward, push after it, loss after the last forward, backward last
    first_bwd = min(i for i, c in enumerate(lib.calls) if c.startswith("gnn_layer_backward"))
    assert lib.calls.index("gnn_softmax_ce") < first_bwd
    assert max(i for i, c in enumerate(lib.calls) if c.startswith("gnn_layer_forward")) < lib.calls.index(
        "gnn_softmax_ce")
    assert fwd in lib.calls


@pytest.mark.parametrize("want_halo_grad", [True, False])
def test_reordered_backward_passes_the_binding_checks(lib, want_halo_grad):
    # layers l > 0 take the other product order, layer 0 the textbook backward (it has no input gradient)
    m, part = _model("gcn", torch.bfloat16, widths=(12, 20, 16, 6))
    m.set_reorder(True)
    for l in range(m.L):
        m.tables[l] = padded(part.n_table, m.widths[l], torch.bfloat16, "cpu")
    m.forward()
    m.loss_grad()
    lib.calls.clear()
    m.backward(want_halo_grad)
    assert lib.calls == ["gnn_layer_backward_reordered", "gnn_layer_backward_reordered", "gnn_layer_backward"]
    m.set_reorder(False)
    lib.calls.clear()
    m.backward(want_halo_grad)
    assert lib.calls == ["gnn_layer_backward"] * 3


def test_reordered_backward_needs_gcn_bf16_and_fp32_gradients(lib):
    with pytest.raises(ValueError):
        _model("sage", torch.bfloat16)[0].set_reorder(True)
    with pytest.raises(ValueError):
        _model("gcn", torch.float32)[0].set_reorder(True)
    with pytest.raises(ValueError):
        _model("gcn", torch.bfloat16, grad_dtype=torch.bfloat16)[0].set_reorder(True)
    m, _ = _model("gcn", torch.bfloat16)
    m.set_reorder(True)
    with pytest.raises(ValueError):
        m.set_grad_dtype(torch.bfloat16)


@pytest.mark.parametrize("mode,sync_every", [("sync", 0), ("stale", 0), ("stale", 1)])
def test_multi_partition_epoch_order(lib, mode, sync_every):
    parts, N = _parts(3)
    t = MultiPartitionTrainer(parts, [10, 14, 5], "gcn", torch.float32, N, mode=mode, sync_every=sync_every,
                              device="cpu")
    lib.calls.clear()
    t.epoch()
    c = lib.calls
    assert c.count("gnn_layer_forward") == 3 * 2 and c.count("gnn_layer_backward") == 3 * 2
    assert c.count("gnn_softmax_ce_partial") == 3
    halo_parts = sum(1 for p in parts if p.n_halo)
    assert c.count("gnn_halo_grad_send") == halo_parts  # layer 1 only (layer 0 has no input gradient)
    assert c.count("gnn_halo_grad_recv") == 3
    sync = mode == "sync" or sync_every == 1
    fwd = [i for i, x in enumerate(c) if x == "gnn_layer_forward"]
    if sync:
        # layer by layer across partitions: all layer-0 forwards before any layer-1 forward, every push of
        # layer 0 before the first layer-1 pull
        assert all(c[fwd[i]] == "gnn_layer_forward" for i in range(3))
        pushes = [i for i, x in enumerate(c) if x == "gnn_halo_push"]
        pulls = [i for i, x in enumerate(c) if x == "gnn_halo_pull"]
        assert max(pushes) < max(pulls)
        # every send of the gradient table before the first receive
        sends = [i for i, x in enumerate(c) if x == "gnn_halo_grad_send"]
        recvs = [i for i, x in enumerate(c) if x == "gnn_halo_grad_recv"]
        assert max(sends) < min(recvs)
    else:
        # partition by partition: partition 0's two forwards come before partition 1's first
        pulls = [i for i, x in enumerate(c) if x == "gnn_halo_pull"]
        assert fwd[1] < pulls[2]
        # each partition receives last epoch's gradients before sending this epoch's
        assert c.index("gnn_halo_grad_recv") < c.index("gnn_halo_grad_send")
    assert t.epoch_index == 1


def test_binding_rejects_undersized_or_mistyped_buffers(lib):
    m, part = _model(widths=(12, 16, 6))
    g, nL, nT = m.graph, part.n_local, part.n_local + part.n_halo
    f = 12
    W = torch.zeros((f, 16), dtype=torch.float32)
    Z = padded(nL, f, torch.float32, "cpu")
    Ho = padded(nL, 16, torch.float32, "cpu")
    H = padded(nT, f, torch.float32, "cpu")
    work = lambda: [c for c in lib.calls if c not in ("gnn_status_string", "gnn_last_cuda_error")]  # noqa: E731
    n_calls = len(work())
    bad = [
        lambda: gnn.layer_forward(g, H[:nL], W, True, Z, Ho),                      # H without its halo rows
        lambda: gnn.layer_forward(g, H, W[:8], True, Z, Ho),                       # W with too few rows
        lambda: gnn.layer_forward(g, H, W.double(), True, Z, Ho),                  # W not float32
        lambda: gnn.layer_forward(g, H, W, True, Z[:, :8], Ho),                    # Z narrower than f_in
        lambda: gnn.layer_forward(g, H.bfloat16(), W, True, Z, Ho),                # mixed dtypes
        lambda: gnn.halo_pull(g, padded(part.n_table, 8, torch.float32, "cpu"), m.halo_ids, H),  # narrow table
        lambda: gnn.halo_pull(g, padded(part.n_table, f, torch.float32, "cpu"), m.halo_ids.int(), H),  # int32 ids
        lambda: gnn.halo_push(g, H[:nL - 1], m.local_ids, padded(part.n_table, f, torch.float32, "cpu")),
        lambda: gnn.layer_backward(g, Ho, Ho, Z, W, True, torch.zeros((f, 15)), f),  # dW of the wrong shape
        lambda: gnn.layer_backward(g, Ho, Ho, Z, W, True, torch.zeros((f, 16)), f,
                                   dH=padded(nL, f, torch.float32, "cpu"), want_halo_grad=True),  # no halo rows
        lambda: gnn.softmax_ce(Ho, torch.zeros(nL, dtype=torch.int64), Ho.clone(), torch.zeros(nL),
                               torch.zeros(1)),                                    # int64 labels
        lambda: gnn.layer_backward(g, Ho.bfloat16(), Ho, Z, W, True, torch.zeros((f, 16)), f),  # fp32 acts, bf16 G
        lambda: gnn.layer_backward(g, Ho, Ho.bfloat16(), Z, W, True, torch.zeros((f, 16)), f),  # H_out and Z differ
        lambda: gnn.layer_backward(g, Ho, Ho, Z, W, True, torch.zeros((f, 16)), f, dZ=Z.bfloat16(),
                                   dH=padded(nT, f, torch.float32, "cpu"), want_halo_grad=True),  # dZ not like G
        lambda: gnn.halo_grad_send(g, H[:nL], m.halo_ids, torch.zeros((part.n_table, f))),  # dH without halo rows
        lambda: gnn.halo_push_quantized(g, H[:nL], m.local_ids, torch.zeros((part.n_table, 8), dtype=torch.uint8),
                                        torch.zeros((part.n_table, 2)), 4, 0),      # code rows too short
    ]
    for i, call in enumerate(bad):
        with pytest.raises(gnn.GnnError) as e:
            call()
        assert e.value.status == gnn.GNN_EINVAL, i
    assert len(work()) == n_calls  # nothing but the error text reached the library
    # the same calls with correct buffers go through
    gnn.layer_forward(g, H, W, True, Z, Ho)
    gnn.halo_pull(g, padded(part.n_table, f, torch.float32, "cpu"), m.halo_ids, H)
    assert lib.calls[-2:] == ["gnn_layer_forward", "gnn_halo_pull"]
