"""Multi-process paths on the CPU (gloo, world size 2), no GPU needed.

1. bench.py's rank logic: max / sum over ranks, and the reference arm under
   torchrun (rank 0 prints one JSON line, rank 1 exits 0 without work).
2. The multi-partition exchange the pages describe (Sylvie HALO exchange,
   DIGEST pull/push through a shared table): two ranks, one partition each,
   exchange pushed rows through a table assembled with an all-gather, and
   together reproduce the full-graph two-layer forward and dW of the oracle.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _reduce_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench

    _init(rank, world, port)
    mx = bench.max_over_ranks(dist, float(rank + 1) * 10.0, False)
    sm = bench.sum_over_ranks(dist, float(rank + 1), False)
    bench.barrier(dist, False)
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_bench_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reduce_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 20.0, 3.0), (1, 20.0, 3.0)]


def test_bench_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "er5k-tiny", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-seconds", "0.05"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def _partition_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import oracle
    from tests._problems import dense_gcn_block, partition_from_dense, random_sym_adjacency

    _init(rank, world, port)
    import torch

    N, f, hid = 40, 5, 4
    A = random_sym_adjacency(N, 0.15, 77)
    rng = np.random.default_rng(77)
    X = rng.standard_normal((N, f))
    W0 = rng.standard_normal((f, hid))
    W1 = rng.standard_normal((hid, 3))
    blocks = [np.arange(0, 23), np.arange(23, N)]
    part, _ = partition_from_dense(A, blocks[rank])
    # layer 0: halo rows pulled from the feature table
    H = np.zeros((part.n_total, f))
    H[:part.n_local] = X[part.local_ids]
    oracle.halo_pull(X, part.halo_ids, H, part.n_local, f)
    _, h1 = oracle.layer_forward(part, H, W0, "gcn", relu=True)
    # push: every rank contributes its fresh rows to the shared table
    mine = np.zeros((N, hid))
    oracle.halo_push(h1, part.n_local, hid, part.local_ids, mine)
    table = torch.from_numpy(mine)
    dist.all_reduce(table)  # rows are disjoint: the sum assembles the table
    table1 = table.numpy()
    # layer 1 pulls its halo from the assembled table
    H1 = np.zeros((part.n_total, hid))
    H1[:part.n_local] = h1
    oracle.halo_pull(table1, part.halo_ids, H1, part.n_local, hid)
    Z1, h2 = oracle.layer_forward(part, H1, W1, "gcn", relu=False)
    R = np.random.default_rng(5).standard_normal((N, 3))
    dW1, _, _ = oracle.layer_backward(part, oracle.transpose(part), R[part.local_ids], h2, Z1, W1, "gcn",
                                      relu=False)
    dw = torch.from_numpy(dW1)
    dist.all_reduce(dw)  # parameter sync of the partitions' gradients
    Ad = dense_gcn_block(A, np.arange(N), np.arange(N))
    full_h2 = Ad @ np.maximum(Ad @ X @ W0, 0) @ W1
    full_dw1 = (Ad @ np.maximum(Ad @ X @ W0, 0)).T @ R
    q.put((rank, float(np.max(np.abs(h2 - full_h2[part.local_ids]))), float(np.max(np.abs(dw.numpy() - full_dw1)))))
    dist.destroy_process_group()


def test_two_partitions_exchange_through_table_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, e_h, e_dw in res:
        assert e_h < 1e-12 and e_dw < 1e-10
