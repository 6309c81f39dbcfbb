"""Several partitions trained together on one GPU (MultiPartitionTrainer).

* sync schedule: halo rows exchanged layer by layer through the tables and
  the halo gradients J returned to their owners (Sylvie Alg. 1 / Alg. 2) - the
  epoch must equal the whole-graph layer computed by the oracle on the
  unpartitioned graph (loss, logits, summed dW);
* stale schedule (DIGEST / Sylvie-A): each partition's forward reads the
  previous epoch's tables - its logits must equal the oracle's epoch of that
  partition on those tables; with a forced synchronisation every epoch it
  must equal the sync schedule bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_aggregation_dense_gb300 import MultiPartitionTrainer
from tests._flip import close_bounded, epoch_bounds
from tests._gpu import close
from tests._problems import partition_from_dense, random_sym_adjacency

pytestmark = pytest.mark.gpu

N = 1500
WIDTHS = [24, 40, 32, 6]


def _setup(P, seed, dtype):
    A = random_sym_adjacency(N, 12.0 / N, seed)
    perm = np.random.default_rng(seed).permutation(N)
    blocks = np.array_split(perm, P)
    parts = [partition_from_dense(A, np.sort(b))[0] for b in blocks]
    full, _ = partition_from_dense(A, np.arange(N))
    rng = np.random.default_rng(seed + 1)
    X = rng.standard_normal((N, WIDTHS[0]))
    Ws = [rng.uniform(-1, 1, (WIDTHS[l], WIDTHS[l + 1])) * np.sqrt(6 / (WIDTHS[l] + WIDTHS[l + 1]))
          for l in range(len(WIDTHS) - 1)]
    y = rng.integers(0, WIDTHS[-1], N).astype(np.int32)
    if dtype == torch.bfloat16:  # inputs exactly representable in bf16
        X = oracle.round_bf16(X)
        Ws = [oracle.round_bf16(w) for w in Ws]
    return A, parts, full, X, Ws, y


def _trainer(parts, X, Ws, y, dtype, **kw):
    t = MultiPartitionTrainer(parts, WIDTHS, "gcn", dtype, N, **kw)
    t.set_features(torch.from_numpy(X).to(dtype).cuda())
    t.set_weights([torch.from_numpy(w).float().cuda() for w in Ws])
    t.set_labels(torch.from_numpy(y).cuda())
    return t


# bf16 runs the layers in the textbook order, where its rounding points are the
# oracle's (the multiplication-first order rounds H W instead of A H, and stores
# its gradients in bf16); fp32 runs both orders.  The gradients of the bf16 runs
# are stored in fp32 or in bf16.
@pytest.mark.parametrize("dtype,gdtype,tol,narrow", [(torch.float32, torch.float32, 1e-4, True),
                                                     (torch.float32, torch.float32, 1e-4, False),
                                                     (torch.bfloat16, torch.float32, 2e-2, False),
                                                     (torch.bfloat16, torch.bfloat16, 2e-2, False)])
@pytest.mark.parametrize("P", [2, 3])
def test_sync_epoch_equals_whole_graph(P, dtype, gdtype, tol, narrow):
    A, parts, full, X, Ws, y = _setup(P, 10 + P, dtype)
    t = _trainer(parts, X, Ws, y, dtype, mode="sync", narrow=narrow, grad_dtype=gdtype)
    t.epoch()
    t.check_errors()
    tables = [X] + [np.zeros((N, f)) for f in WIDTHS[1:-1]]
    bf = dtype == torch.bfloat16
    ref = oracle.epoch(full, tables, Ws, y, "gcn", bf16=bf, grad_bf16=gdtype == torch.bfloat16)
    # the multiplication-first layers round other intermediates than the
    # textbook order: their pre-activations get that order's bound
    mf = [narrow and WIDTHS[l + 1] < WIDTHS[l] for l in range(len(Ws))]
    dWb, _, n_amb = epoch_bounds(full, ref, Ws, "gcn", bf, multiply_first=mf)
    assert abs(float(t.loss.item()) - ref["loss"]) <= tol * abs(ref["loss"])
    for m, p in zip(t.models, parts):
        close(m.out_last.float().cpu().numpy().astype(np.float64), ref["Hout"][-1][p.local_ids], tol, "logits")
    for l in range(len(Ws)):
        close_bounded(t.dW[l].cpu().numpy().astype(np.float64), ref["dW"][l], tol, dWb[l],
                      f"dW[{l}] ({n_amb} ambiguous decisions)")


def test_stale_forward_reads_previous_tables():
    dtype = torch.float32
    A, parts, full, X, Ws, y = _setup(3, 7, dtype)
    t = _trainer(parts, X, Ws, y, dtype, mode="stale")
    tables = [X] + [np.zeros((N, f)) for f in WIDTHS[1:-1]]
    for _ in range(2):
        t.epoch()
        t.check_errors()
        nxt = [X] + [np.zeros((N, f)) for f in WIDTHS[1:-1]]
        for m, p in zip(t.models, parts):
            ref = oracle.epoch(p, tables, Ws, y[p.local_ids], "gcn")
            close(m.out_last.cpu().numpy().astype(np.float64), ref["Hout"][-1], 1e-4, "stale logits")
            for l in range(1, len(WIDTHS) - 1):
                nxt[l][p.local_ids] = ref["Hout"][l - 1]
        tables = nxt


def test_forced_sync_every_epoch_equals_sync():
    dtype = torch.float32
    A, parts, full, X, Ws, y = _setup(2, 3, dtype)
    a = _trainer(parts, X, Ws, y, dtype, mode="sync")
    b = _trainer(parts, X, Ws, y, dtype, mode="stale", sync_every=1)
    for _ in range(2):
        a.epoch()
        b.epoch()
    torch.cuda.synchronize()
    assert torch.equal(a.loss, b.loss)
    for da, db in zip(a.dW, b.dW):
        assert torch.equal(da, db)
    for ma, mb in zip(a.models, b.models):
        assert torch.equal(ma.out_last, mb.out_last)
