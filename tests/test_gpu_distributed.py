"""The process-per-partition driver on the GPU (DistributedPartitionTrainer with
libgnn): two processes, one partition each, sharing the one GPU; the halo rows
and the returned halo gradients J travel by gloo all-to-all through host memory
(no kernel waits on the other process: every exchange is a collective between
launches).  The epoch must equal the whole-graph oracle epoch.

Also the two row kernels of the exchange (gnn_gather_rows, gnn_scatter_add_rows)
against numpy, bit for bit.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from sparse_aggregation_dense_gb300 import gnn, padded
from tests._flip import close_bounded, epoch_bounds
from tests._gpu import close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N = 1200
WIDTHS = [24, 40, 32, 6]


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem(world, dtype):
    from tests._problems import partition_from_dense, random_sym_adjacency

    A = random_sym_adjacency(N, 12.0 / N, 21)
    rng = np.random.default_rng(21)
    blocks = [np.sort(b) for b in np.array_split(rng.permutation(N), world)]
    X = rng.standard_normal((N, WIDTHS[0]))
    Ws = [rng.uniform(-1, 1, (WIDTHS[l], WIDTHS[l + 1])) * np.sqrt(6 / (WIDTHS[l] + WIDTHS[l + 1]))
          for l in range(len(WIDTHS) - 1)]
    y = rng.integers(0, WIDTHS[-1], N).astype(np.int32)
    if dtype == "bf16":
        X = oracle.round_bf16(X)
        Ws = [oracle.round_bf16(w) for w in Ws]
    full, _ = partition_from_dense(A, np.arange(N))
    parts = [partition_from_dense(A, b)[0] for b in blocks]
    return parts, full, X, Ws, y


def _worker(rank, world, port, dtype, gdtype, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from sparse_aggregation_dense_gb300 import DistributedPartitionTrainer

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gdt = torch.bfloat16 if gdtype == "bf16" else torch.float32
    parts, full, X, Ws, y = _problem(world, dtype)
    t = DistributedPartitionTrainer(parts[rank], WIDTHS, "gcn", tdt, device="cuda", grad_dtype=gdt)
    m = t.model
    lid = torch.from_numpy(t.part.local_ids)
    m.H[0][:m.n_local] = torch.from_numpy(X)[lid].to(tdt).cuda()
    for w, src in zip(m.W, Ws):
        w.copy_(torch.from_numpy(src).float())
    m.labels.copy_(torch.from_numpy(y)[lid])
    t.epoch()
    t.check_errors()
    torch.cuda.synchronize()
    q.put((rank, t.part.local_ids.copy(), m.out_last.float().cpu().numpy().astype(np.float64), float(m.loss.item()),
           [d.cpu().numpy().astype(np.float64) for d in m.dW]))
    dist.destroy_process_group()


@pytest.mark.parametrize("dtype,gdtype,tol", [("f32", "f32", 1e-4), ("bf16", "f32", 2e-2)])
def test_two_processes_on_one_gpu_equal_the_whole_graph(dtype, gdtype, tol):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, dtype, gdtype, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=600) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    parts, full, X, Ws, y = _problem(world, dtype)
    bf = dtype == "bf16"
    ref = oracle.epoch(full, [X] + [np.zeros((N, f)) for f in WIDTHS[1:-1]], Ws, y, "gcn", bf16=bf,
                       grad_bf16=gdtype == "bf16")
    dWb, _, n_amb = epoch_bounds(full, ref, Ws, "gcn", bf)
    for rank, lid, logits, loss, dW in res:
        close(logits, ref["Hout"][-1][lid], tol, f"rank {rank} logits")
        assert abs(loss - ref["loss"]) <= tol * abs(ref["loss"])
        for l in range(len(Ws)):
            close_bounded(dW[l], ref["dW"][l], tol, dWb[l], f"rank {rank} dW[{l}] ({n_amb} ambiguous decisions)")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("f", [1, 5, 40, 256, 300])
def test_exchange_row_kernels_bit_exact(dt, f):
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    rng = np.random.default_rng(f)
    n_src, n = 5000, 3000
    src = padded(n_src, f, tdt, "cuda")
    src.copy_(torch.from_numpy(rng.standard_normal((n_src, f))).to(tdt))
    ids = torch.from_numpy(rng.integers(0, n_src, n)).cuda()
    dst = padded(n, f, tdt, "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gnn.gather_rows(src, ids, dst, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(dst, src[ids])
    # scatter-add of distinct ids, in two calls (the second adds onto the first)
    tgt = padded(n_src, f, tdt, "cuda")
    tgt.copy_(torch.from_numpy(rng.standard_normal((n_src, f))).to(tdt))
    perm = torch.from_numpy(rng.permutation(n_src)[:n]).cuda()
    before = tgt.float().cpu().numpy().astype(np.float64)
    gnn.scatter_add_rows(dst, perm, tgt, err)
    gnn.scatter_add_rows(dst[:100], perm[:100], tgt, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = before.copy()
    add = dst.float().cpu().numpy().astype(np.float64)
    p = perm.cpu().numpy()
    ref[p] = (torch.from_numpy(ref[p] + add).float().to(tdt).double()).numpy()  # one rounding per call
    ref[p[:100]] = (torch.from_numpy(ref[p[:100]] + add[:100]).float().to(tdt).double()).numpy()
    np.testing.assert_array_equal(tgt.float().cpu().numpy().astype(np.float64), ref)
    # an id outside the matrix is reported and its row left alone
    bad = ids.clone()
    bad[7] = n_src
    dst2 = padded(n, f, tdt, "cuda")
    dst2.fill_(3.0)
    gnn.gather_rows(src, bad, dst2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert bool(torch.all(dst2[7] == 3.0))
