"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This package builds graphs, partitions, features, weights and labels and nothing
else: it holds none of the layer's arithmetic.  The heavy lifting is a small C
library (``csrc/synth.c``) compiled with gcc; every random value is a counter-based
draw, so results are identical on any machine and for any thread count.

Workload shapes follow the source pages (Sylvie, DIGEST, CAGNET, DistDGL): an
Erdos-Renyi toy partition, R-MAT graphs, Chung-Lu power-law graphs shaped like
the Reddit / Amazon / products datasets by size, and one partition of a
billion-edge R-MAT graph with stale-representation tables.  See ``configs.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None

# seed streams (fixed numbers so every consumer draws the same values)
STREAM_FEATURES = 1
STREAM_TABLE = 10  # + layer index: stale-representation table contents
STREAM_WEIGHT = 20  # + layer index
STREAM_LABELS = 30
STREAM_GRAD = 40  # + layer index: synthetic upstream gradients for per-call tests
STREAM_SAMPLE = 50


def build(force: bool = False) -> str:
    """Compile ``csrc/synth.c`` into ``_synth.so`` next to this file."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=gnu11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Part(ctypes.Structure):
    _fields_ = [
        ("n_local", ctypes.c_int64),
        ("n_halo", ctypes.c_int64),
        ("nnz", ctypes.c_int64),
        ("n_table", ctypes.c_int64),
        ("rowptr", ctypes.POINTER(ctypes.c_int32)),
        ("colidx", ctypes.POINTER(ctypes.c_int32)),
        ("deg", ctypes.POINTER(ctypes.c_float)),
        ("local_ids", ctypes.POINTER(ctypes.c_int64)),
        ("halo_ids", ctypes.POINTER(ctypes.c_int64)),
    ]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(_Part)
        i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        L.synth_make_er.argtypes = [i64, i64, dbl, u64]
        L.synth_make_er.restype = P
        L.synth_make_rmat_sym.argtypes = [ctypes.c_int, dbl, dbl, dbl, i64, i64, ctypes.c_int, u64]
        L.synth_make_rmat_sym.restype = P
        L.synth_make_chunglu.argtypes = [i64, dbl, dbl, dbl, i64, i64, u64]
        L.synth_make_chunglu.restype = P
        L.synth_make_rmat_block.argtypes = [ctypes.c_int, dbl, dbl, dbl, dbl, i64, i64, u64]
        L.synth_make_rmat_block.restype = P
        L.synth_part_free.argtypes = [P]
        L.synth_part_free.restype = None
        L.synth_features.argtypes = [vp, i64, i64, i64, u64, u64, ctypes.c_int, ctypes.c_int, vp]
        L.synth_features.restype = None
        L.synth_glorot.argtypes = [i64, i64, u64, u64, vp]
        L.synth_glorot.restype = None
        L.synth_labels.argtypes = [vp, i64, i64, u64, u64, vp]
        L.synth_labels.restype = None
        L.synth_uniform.argtypes = [i64, u64, u64, vp]
        L.synth_uniform.restype = None
        L.synth_num_threads.argtypes = []
        L.synth_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


@dataclass
class Partition:
    """One partition: block CSR of A+I over local rows and local+halo columns.

    rowptr  int32[n_local+1]; colidx int32[nnz] (sorted per row, self loops included)
    deg     float32[n_local+n_halo] global degrees of A+I, or None (not passed)
    local_ids / halo_ids int64 table rows of the local / halo vertices
    n_table number of rows of the stale-representation tables
    """

    rowptr: np.ndarray
    colidx: np.ndarray
    n_local: int
    n_halo: int
    deg: Optional[np.ndarray]
    local_ids: np.ndarray
    halo_ids: np.ndarray
    n_table: int

    @property
    def nnz(self) -> int:
        return int(self.colidx.shape[0])

    @property
    def n_total(self) -> int:
        return self.n_local + self.n_halo


def _take(ptr) -> Partition:
    if not ptr:
        raise MemoryError("synthetic graph generation failed")
    p = ptr.contents
    nL, nH, nnz = p.n_local, p.n_halo, p.nnz

    def arr(field, n, dtype):
        if n == 0:
            return np.zeros(0, dtype=dtype)
        return np.ctypeslib.as_array(field, shape=(n,)).astype(dtype, copy=True)

    out = Partition(
        rowptr=arr(p.rowptr, nL + 1, np.int32),
        colidx=arr(p.colidx, nnz, np.int32),
        n_local=int(nL),
        n_halo=int(nH),
        deg=arr(p.deg, nL + nH, np.float32) if bool(p.deg) else None,
        local_ids=arr(p.local_ids, nL, np.int64),
        halo_ids=arr(p.halo_ids, nH, np.int64),
        n_table=int(p.n_table),
    )
    lib().synth_part_free(ptr)
    return out


def er_partition(n: int, n_local: int, p: float, seed: int = 0) -> Partition:
    """Undirected G(n, p); local = [0, n_local), halo = every other vertex."""
    return _take(lib().synth_make_er(n, n_local, p, seed))


def rmat_sym_partition(scale: int, n_unique: int, n_local: int, seed: int = 0, abc=(0.57, 0.19, 0.19),
                       halo_all: bool = True) -> Partition:
    """Undirected R-MAT, first n_unique unique edges, random vertex permutation."""
    a, b, c = abc
    return _take(lib().synth_make_rmat_sym(scale, a, b, c, n_unique, n_local, int(halo_all), seed))


def chunglu_partition(n: int, n_unique: int, mean_deg: float, nparts: int, seed: int = 0, gamma: float = 2.5,
                      cap_frac: float = 1.0 / 8.0) -> Partition:
    """Chung-Lu power-law graph; partition 0 of nparts contiguous blocks."""
    return _take(lib().synth_make_chunglu(n, gamma, mean_deg, cap_frac * n, n_unique, nparts, seed))


def rmat_block_partition(scale: int, n_local: int, n_halo: int, samples: float, seed: int = 0,
                         abc=(0.57, 0.19, 0.19)) -> Partition:
    """Directed R-MAT block of one partition of a 2^scale-vertex graph (deg not passed)."""
    a, b, c = abc
    return _take(lib().synth_make_rmat_block(scale, a, b, c, samples, n_local, n_halo, seed))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def features(n_rows: int, f: int, ld: int, seed: int, stream: int, dist: str = "normal", bf16: bool = False,
             ids: Optional[np.ndarray] = None) -> np.ndarray:
    """Dense rows (n_rows x ld); row i holds id ids[i] (or i); columns >= f are zero.

    dist: "uniform" -> U[-1, 1], "normal" -> N(0, 1).  bf16=True returns uint16 bf16
    bit patterns (round to nearest even), else float32.
    """
    if ids is not None:
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        n_rows = ids.shape[0]
    out = np.empty((n_rows, ld), dtype=np.uint16 if bf16 else np.float32)
    if n_rows:
        lib().synth_features(_ptr(ids), n_rows, f, ld, seed, stream, 0 if dist == "uniform" else 1, int(bf16),
                             _ptr(out))
    return out


def glorot(fi: int, fo: int, seed: int, stream: int) -> np.ndarray:
    """Glorot-uniform fi x fo float32 weight matrix."""
    out = np.empty((fi, fo), dtype=np.float32)
    lib().synth_glorot(fi, fo, seed, stream, _ptr(out))
    return out


def labels(n: int, n_classes: int, seed: int, stream: int = STREAM_LABELS,
           ids: Optional[np.ndarray] = None) -> np.ndarray:
    if ids is not None:
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        n = ids.shape[0]
    out = np.empty(n, dtype=np.int32)
    if n:
        lib().synth_labels(_ptr(ids), n, n_classes, seed, stream, _ptr(out))
    return out


def uniform(n: int, seed: int, stream: int = STREAM_SAMPLE) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        lib().synth_uniform(n, seed, stream, _ptr(out))
    return out


def sample_rows(n: int, k: int, seed: int, stream: int = STREAM_SAMPLE) -> np.ndarray:
    """k distinct sorted row indices in [0, n) (all rows if k >= n)."""
    if k >= n:
        return np.arange(n, dtype=np.int64)
    u = uniform(n, seed, stream)
    return np.sort(np.argsort(u, kind="stable")[:k]).astype(np.int64)


def num_threads() -> int:
    return int(lib().synth_num_threads())


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m
