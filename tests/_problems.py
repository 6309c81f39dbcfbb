"""Tiny hand-built problems for the oracle pins (dense numpy, independent of oracle.c)."""
from __future__ import annotations

import numpy as np

from synth import Partition


def random_sym_adjacency(N: int, p: float, seed: int) -> np.ndarray:
    """Symmetric 0/1 adjacency without self loops."""
    rng = np.random.default_rng(seed)
    A = rng.random((N, N)) < p
    A = np.triu(A, 1)
    return (A | A.T).astype(np.int64)


def partition_from_dense(A: np.ndarray, local: np.ndarray, halo_all: bool = False, pass_deg: bool = True):
    """Partition of the undirected graph A (no self loops) for the local vertex list.

    Columns are the local vertices (in the given order) followed by the halo
    vertices (ascending global id).  Returns (Partition, cols) where cols[c] is the
    global vertex of block column c.
    """
    N = A.shape[0]
    local = np.asarray(local, dtype=np.int64)
    is_local = np.zeros(N, dtype=bool)
    is_local[local] = True
    if halo_all:
        halo = np.array([u for u in range(N) if not is_local[u]], dtype=np.int64)
    else:
        touched = A[local].sum(axis=0) > 0
        halo = np.array([u for u in range(N) if touched[u] and not is_local[u]], dtype=np.int64)
    cols = np.concatenate([local, halo])
    pos = -np.ones(N, dtype=np.int64)
    pos[cols] = np.arange(cols.shape[0])
    AI = A + np.eye(N, dtype=np.int64)
    rowptr = [0]
    colidx = []
    for v in local:
        cs = sorted(int(pos[u]) for u in np.nonzero(AI[v])[0])
        colidx.extend(cs)
        rowptr.append(len(colidx))
    deg = AI.sum(axis=1).astype(np.float32)[cols] if pass_deg else None
    part = Partition(rowptr=np.array(rowptr, dtype=np.int32), colidx=np.array(colidx, dtype=np.int32),
                     n_local=int(local.shape[0]), n_halo=int(halo.shape[0]), deg=deg, local_ids=local.copy(),
                     halo_ids=halo.copy(), n_table=N)
    return part, cols


def dense_gcn_block(A: np.ndarray, local: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Rows `local`, columns `cols` of D^-1/2 (A + I) D^-1/2 (D: degrees of A + I)."""
    N = A.shape[0]
    AI = A + np.eye(N)
    d = AI.sum(axis=1)
    Dm = np.diag(1.0 / np.sqrt(d))
    Ahat = Dm @ AI @ Dm
    return Ahat[np.ix_(local, cols)]


def dense_mean_block(A: np.ndarray, local: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Rows `local`, columns `cols` of the neighbour-mean operator (self excluded)."""
    M = A[np.ix_(local, cols)].astype(np.float64)
    cnt = M.sum(axis=1, keepdims=True)
    return np.divide(M, cnt, out=np.zeros_like(M), where=cnt > 0)


def circulant(N: int, half_k: int) -> np.ndarray:
    """k-regular ring lattice: v ~ v +- 1 .. half_k (mod N)."""
    A = np.zeros((N, N), dtype=np.int64)
    for v in range(N):
        for s in range(1, half_k + 1):
            A[v, (v + s) % N] = 1
            A[(v + s) % N, v] = 1
    return A
