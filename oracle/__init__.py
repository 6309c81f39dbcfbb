"""CPU oracle for one partition's GCN / GraphSAGE layer, forward and backward.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain loops, double precision, one output
row per loop iteration); this module only widens inputs to float64, calls the C
functions and composes them in the order the pages give:

  pull halo rows from the stale table   (DIGEST page, system design, Fig. 1c)
  Z  = A_block H            aggregation (CAGNET page, GNN section; Sylvie Alg. 1)
  H' = sigma(Z W)           update      (CAGNET page, GNN section)
  push local rows to the table          (DIGEST page, Fig. 1c)
  backward by the chain rule            (CAGNET page, GNN section: the backward
                                         reuses the forward's SpMM and GEMM;
                                         the derivation is not in the text)

Every function here is pinned by a ``-m "not gpu"`` test against facts fixed
outside the oracle (``tests/test_oracle_pins.py``, ``tests/test_codec_pins.py``);
none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None

OK = 0
ERR_INDEX = 5


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``_oracle.so`` next to this file."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O3", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=gnu11", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_halo_pull.argtypes = [vp, i64, i64, vp, i64, vp, i64, i64, i64, i32]
        L.oracle_halo_pull.restype = i32
        L.oracle_halo_push.argtypes = [vp, i64, i64, i64, vp, vp, i64, i64, i32]
        L.oracle_halo_push.restype = i32
        L.oracle_gcn_dinv.argtypes = [vp, vp, i64, i64, vp, vp]
        L.oracle_gcn_dinv.restype = None
        L.oracle_sage_invcnt.argtypes = [vp, vp, i64, vp]
        L.oracle_sage_invcnt.restype = None
        L.oracle_gcn_aggregate.argtypes = [vp, vp, vp, vp, i64, vp, i64, vp, i64, vp, i64]
        L.oracle_gcn_aggregate.restype = None
        L.oracle_sage_aggregate.argtypes = [vp, vp, vp, vp, i64, vp, i64, vp, i64, vp, i64, i64]
        L.oracle_sage_aggregate.restype = None
        L.oracle_update.argtypes = [vp, i64, i64, i64, vp, i64, i32, vp, i64]
        L.oracle_update.restype = None
        L.oracle_update_backward_dz.argtypes = [vp, i64, vp, i64, i64, i64, i32, vp, i64, vp, i64]
        L.oracle_update_backward_dz.restype = None
        L.oracle_update_backward_dw.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, i32, vp]
        L.oracle_update_backward_dw.restype = None
        L.oracle_transpose.argtypes = [vp, vp, i64, i64, vp, vp, vp]
        L.oracle_transpose.restype = i32
        L.oracle_gcn_aggregate_backward.argtypes = [vp, vp, vp, vp, i64, vp, i64, vp, i64, vp, i64]
        L.oracle_gcn_aggregate_backward.restype = None
        L.oracle_sage_aggregate_backward.argtypes = [vp, vp, vp, i64, vp, i64, vp, i64, i64, vp, i64, vp, i64]
        L.oracle_sage_aggregate_backward.restype = None
        L.oracle_softmax_ce.argtypes = [vp, i64, i64, i64, vp, vp, i64]
        L.oracle_softmax_ce.restype = ctypes.c_double
        L.oracle_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.oracle_splitmix64.restype = ctypes.c_uint64
        L.oracle_codec_quantize.argtypes = [vp, i64, i64, i64, vp, i32, ctypes.c_uint64, vp, i64, vp]
        L.oracle_codec_quantize.restype = None
        L.oracle_codec_dequantize.argtypes = [vp, i64, vp, i64, i64, i32, vp, i64]
        L.oracle_codec_dequantize.restype = None
        L.oracle_gat_attend.argtypes = [vp, vp, i64, vp, vp, vp, i64, i64, ctypes.c_double, vp, vp, i64]
        L.oracle_gat_attend.restype = None
        L.oracle_gat_attend_backward.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i64, ctypes.c_double, vp, vp, i64,
                                                 vp, i64, vp, vp]
        L.oracle_gat_attend_backward.restype = None
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_set_num_threads.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i64(a) -> Optional[np.ndarray]:
    return None if a is None else np.ascontiguousarray(a, dtype=np.int64)


def num_threads() -> int:
    return int(_L().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads of the oracle's parallel loops from now on (n > 0)."""
    _L().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------
# value decoding (inputs are stored fp32 or bf16; the oracle works in double)
# --------------------------------------------------------------------------

def widen(a: np.ndarray, bf16: bool) -> np.ndarray:
    """Exact float64 copy of stored values (bf16 given as uint16 bit patterns)."""
    if bf16:
        return (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (through float32, nearest even); returns float64."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# stale-representation table
# --------------------------------------------------------------------------

def halo_pull(table: np.ndarray, halo_ids: np.ndarray, H: np.ndarray, n_local: int, f: int) -> int:
    """H[n_local + i, :f] = table[halo_ids[i], :f] (in place, bit-exact copy)."""
    assert table.dtype == H.dtype and table.flags.c_contiguous and H.flags.c_contiguous
    ids = _i64(halo_ids)
    return int(_L().oracle_halo_pull(_p(table), table.shape[1], table.shape[0], _p(ids), ids.shape[0], _p(H),
                                     H.shape[1], n_local, f, table.dtype.itemsize))


def halo_push(H: np.ndarray, n_local: int, f: int, local_ids: np.ndarray, table: np.ndarray) -> int:
    """table[local_ids[v], :f] = H[v, :f] (in place); repeated or bad ids -> ERR_INDEX."""
    assert table.dtype == H.dtype and table.flags.c_contiguous and H.flags.c_contiguous
    ids = _i64(local_ids)
    return int(_L().oracle_halo_push(_p(H), H.shape[1], n_local, f, _p(ids), _p(table), table.shape[1],
                                     table.shape[0], table.dtype.itemsize))


# --------------------------------------------------------------------------
# degrees and aggregation
# --------------------------------------------------------------------------

def _csr(part):
    return (np.ascontiguousarray(part.rowptr, dtype=np.int32), np.ascontiguousarray(part.colidx, dtype=np.int32))


def gcn_dinv(part) -> np.ndarray:
    rp, ci = _csr(part)
    out = np.empty(part.n_local + part.n_halo, dtype=np.float64)
    deg = None if part.deg is None else np.ascontiguousarray(part.deg, dtype=np.float32)
    _L().oracle_gcn_dinv(_p(rp), _p(ci), part.n_local, part.n_halo, _p(deg), _p(out))
    return out


def sage_invcnt(part) -> np.ndarray:
    rp, ci = _csr(part)
    out = np.empty(part.n_local, dtype=np.float64)
    _L().oracle_sage_invcnt(_p(rp), _p(ci), part.n_local, _p(out))
    return out


def aggregate(part, H: np.ndarray, f: int, agg: str, rows=None, hmap=None, weights=None) -> np.ndarray:
    """Forward aggregation for local rows `rows` (default: all).

    H: float64 input rows; column c of the block reads H[hmap[c]] (hmap None: H[c]).
    GCN returns n_rows x f; SAGE returns n_rows x 2f = [self | mean].
    weights: precomputed gcn_dinv / sage_invcnt (computed when None).
    """
    rp, ci = _csr(part)
    H = _f64(H)
    rows = _i64(rows)
    hmap = _i64(hmap)
    n_rows = part.n_local if rows is None else rows.shape[0]
    if agg == "gcn":
        w = gcn_dinv(part) if weights is None else _f64(weights)
        Z = np.empty((n_rows, f), dtype=np.float64)
        _L().oracle_gcn_aggregate(_p(rp), _p(ci), _p(w), _p(H), H.shape[1], _p(hmap), f, _p(rows), n_rows, _p(Z), f)
    elif agg == "sage":
        w = sage_invcnt(part) if weights is None else _f64(weights)
        Z = np.empty((n_rows, 2 * f), dtype=np.float64)
        _L().oracle_sage_aggregate(_p(rp), _p(ci), _p(w), _p(H), H.shape[1], _p(hmap), f, _p(rows), n_rows, _p(Z),
                                   2 * f, f)
    else:
        raise ValueError(agg)
    return Z


def update(Z: np.ndarray, W: np.ndarray, relu: bool) -> np.ndarray:
    """H' = relu(Z W) or Z W."""
    Z, W = _f64(Z), _f64(W)
    n, K = Z.shape
    N = W.shape[1]
    assert W.shape[0] == K
    out = np.empty((n, N), dtype=np.float64)
    _L().oracle_update(_p(Z), K, n, K, _p(W), N, int(relu), _p(out), N)
    return out


def update_backward(G: np.ndarray, Hout: np.ndarray, Z: np.ndarray, W: np.ndarray, relu: bool,
                    want_dz: bool = True, dy_bf16: bool = False):
    """Returns (dW, dZ): dY = G * 1[Hout > 0] (relu) or G; dW = Z^T dY; dZ = dY W^T.

    dy_bf16=True rounds dY to bf16 before the products: with bf16 activations
    every operand of the update's products is bf16 (Z, W and dY alike)."""
    G, Hout, Z, W = _f64(G), _f64(Hout), _f64(Z), _f64(W)
    if dy_bf16:
        G = round_bf16(G * (Hout > 0) if relu else G)
        relu = False
    n, N = G.shape
    K = W.shape[0]
    dW = np.empty((K, N), dtype=np.float64)
    _L().oracle_update_backward_dw(_p(G), N, _p(Hout), Hout.shape[1], _p(Z), Z.shape[1], n, K, N, int(relu), _p(dW))
    dZ = None
    if want_dz:
        dZ = np.empty((n, K), dtype=np.float64)
        _L().oracle_update_backward_dz(_p(G), N, _p(Hout), Hout.shape[1], n, N, int(relu), _p(W), K, _p(dZ), K)
    return dW, dZ


def update_backward_dw_entries(G, Hout, Z, relu: bool, entries: Sequence[tuple]) -> np.ndarray:
    """Selected entries (k, j) of dW = Z^T dY, each summed over all rows in order."""
    out = np.empty(len(entries), dtype=np.float64)
    for t, (k, j) in enumerate(entries):
        zk = _f64(np.ascontiguousarray(Z[:, k:k + 1]))
        gj = _f64(np.ascontiguousarray(G[:, j:j + 1]))
        hj = _f64(np.ascontiguousarray(Hout[:, j:j + 1]))
        dw = np.empty((1, 1), dtype=np.float64)
        _L().oracle_update_backward_dw(_p(gj), 1, _p(hj), 1, _p(zk), 1, zk.shape[0], 1, 1, int(relu), _p(dw))
        out[t] = dw[0, 0]
    return out


def update_backward_dw_columns(G, Hout, Z, relu: bool, cols: Sequence[int], bf16_act: bool, bf16_grad: bool,
                               block_rows: int = 1 << 20) -> np.ndarray:
    """Whole columns `cols` of dW = Z^T dY (K x len(cols)) from stored matrices.

    G, Hout, Z are the stored arrays (uint16 bf16 bit patterns or float32; rows of
    any leading dimension, the first K / N columns used).  With bf16 activations
    dY is rounded to bf16 (an operand of the bf16 products, as in
    update_backward).  Rows are taken in blocks of block_rows, each block
    widened to float64 and its products summed by the C routine; the block sums
    are added in row order in double, so the host never holds a widened copy of
    the whole matrix."""
    cols = [int(c) for c in cols]
    n, K = Z.shape[0], Z.shape[1]
    out = np.zeros((K, len(cols)), dtype=np.float64)
    part = np.empty((K, len(cols)), dtype=np.float64)
    for r0 in range(0, n, block_rows):
        r1 = min(n, r0 + block_rows)
        g = _f64(widen(G[r0:r1][:, cols], bf16_grad))
        h = _f64(widen(Hout[r0:r1][:, cols], bf16_act))
        z = _f64(widen(Z[r0:r1], bf16_act))
        rl = relu
        if bf16_act:
            g = _f64(round_bf16(g * (h > 0) if relu else g))
            rl = False
        _L().oracle_update_backward_dw(_p(g), len(cols), _p(h), len(cols), _p(z), K, r1 - r0, K, len(cols),
                                       int(rl), _p(part))
        out += part
    return out


def transpose(part):
    """(rowptrT int32[nT+1], colidxT int32[nnz], permT int32[nnz]) of the block."""
    rp, ci = _csr(part)
    nT = part.n_local + part.n_halo
    rT = np.empty(nT + 1, dtype=np.int32)
    cT = np.empty(max(part.nnz, 1), dtype=np.int32)
    pT = np.empty(max(part.nnz, 1), dtype=np.int32)
    if _L().oracle_transpose(_p(rp), _p(ci), part.n_local, nT, _p(rT), _p(cT), _p(pT)) != 0:
        raise MemoryError("oracle transpose")
    return rT, cT[:part.nnz], pT[:part.nnz]


def aggregate_backward(part, T, dZ: np.ndarray, f: int, agg: str, rows=None, dmap=None, weights=None) -> np.ndarray:
    """Backward aggregation dH for output rows `rows` of [0, n_local + n_halo) (default all).

    T: transpose(part).  GCN: dZ is n_local x f.  SAGE: dZ = [dZ_self | dZ_mean]
    (n_local x 2f).  dZ row v is dZ[dmap[v]] (dmap None: dZ[v])."""
    rT, cT, _ = T
    rT = np.ascontiguousarray(rT, dtype=np.int32)
    cT = np.ascontiguousarray(cT, dtype=np.int32)
    dZ = _f64(dZ)
    rows = _i64(rows)
    dmap = _i64(dmap)
    nT = part.n_local + part.n_halo
    n_rows = nT if rows is None else rows.shape[0]
    dH = np.empty((n_rows, f), dtype=np.float64)
    if agg == "gcn":
        w = gcn_dinv(part) if weights is None else _f64(weights)
        _L().oracle_gcn_aggregate_backward(_p(rT), _p(cT), _p(w), _p(dZ), dZ.shape[1], _p(dmap), f, _p(rows), n_rows,
                                           _p(dH), f)
    elif agg == "sage":
        w = sage_invcnt(part) if weights is None else _f64(weights)
        _L().oracle_sage_aggregate_backward(_p(rT), _p(cT), _p(w), part.n_local, _p(dZ), dZ.shape[1], _p(dmap), f, f,
                                            _p(rows), n_rows, _p(dH), f)
    else:
        raise ValueError(agg)
    return dH


def softmax_ce(logits: np.ndarray, labels: np.ndarray):
    """(mean loss, G = (softmax - onehot) / n)."""
    x = _f64(logits)
    n, C = x.shape
    lab = np.ascontiguousarray(labels, dtype=np.int32)
    G = np.empty((n, C), dtype=np.float64)
    loss = _L().oracle_softmax_ce(_p(x), C, n, C, _p(lab), _p(G), C)
    return float(loss), G



# --------------------------------------------------------------------------
# graph attention (GAT; named by the Sylvie and DIGEST pages, formula from the
# textbook single-head layer)
# --------------------------------------------------------------------------

GAT_SLOPE = 0.2  # LeakyReLU slope of the attention scores


def gat_attend(part, T: np.ndarray, s_src: np.ndarray, s_dst: np.ndarray):
    """(alpha per entry, Y = sum_u alpha_vu T[u] for the local rows)."""
    rp, ci = _csr(part)
    T = _f64(T)
    f = T.shape[1]
    alpha = np.empty(max(part.nnz, 1), dtype=np.float64)
    Y = np.empty((part.n_local, f), dtype=np.float64)
    _L().oracle_gat_attend(_p(rp), _p(ci), part.n_local, _p(_f64(s_src)), _p(_f64(s_dst)), _p(T), f, f, GAT_SLOPE,
                           _p(alpha), _p(Y), f)
    return alpha[:part.nnz], Y


def gat_attend_backward(part, T, s_src, s_dst, alpha, dY):
    """(dT over every row, ds_src over every row, ds_dst over the local rows)."""
    rp, ci = _csr(part)
    T, dY = _f64(T), _f64(dY)
    f = T.shape[1]
    nT = part.n_local + part.n_halo
    dT = np.empty((nT, f), dtype=np.float64)
    ds_src = np.empty(nT, dtype=np.float64)
    ds_dst = np.empty(max(part.n_local, 1), dtype=np.float64)
    a = _f64(alpha) if part.nnz else np.zeros(1)
    _L().oracle_gat_attend_backward(_p(rp), _p(ci), part.n_local, nT, _p(_f64(s_src)), _p(_f64(s_dst)), _p(T), f, f,
                                    GAT_SLOPE, _p(a), _p(dY), f, _p(dT), f, _p(ds_src), _p(ds_dst))
    return dT, ds_src, ds_dst[:part.n_local]


def gat_layer_forward(part, H: np.ndarray, W: np.ndarray, a_src: np.ndarray, a_dst: np.ndarray, relu: bool,
                      bf16: bool = False):
    """One GAT layer: T = H W (every row), scores s_src = T a_src (every row),
    s_dst = T a_dst (local rows), attention and Y; H' = relu(Y) or Y.  bf16=True
    stores T and H' in bf16 (the scores and alpha stay unrounded).
    Returns dict(T, s_src, s_dst, alpha, Hout)."""
    T = update(H, W, relu=False)
    if bf16:
        T = round_bf16(T)
    s_src = T @ _f64(a_src)
    s_dst = T[:part.n_local] @ _f64(a_dst)
    alpha, Y = gat_attend(part, T, s_src, s_dst)
    Hout = np.maximum(Y, 0.0) if relu else Y
    if bf16:
        Hout = round_bf16(Hout)
    return dict(T=T, s_src=s_src, s_dst=s_dst, alpha=alpha, Hout=Hout)


def gat_layer_backward(part, fwd: dict, H: np.ndarray, G: np.ndarray, W: np.ndarray, a_src: np.ndarray,
                       a_dst: np.ndarray, relu: bool, bf16: bool = False, grad_bf16: bool = False):
    """Chain rule of gat_layer_forward: dY = G * 1[H' > 0] (relu) or G; the
    attention's backward gives dT, ds_src, ds_dst; dT += ds_src a_src^T (every
    row) + ds_dst a_dst^T (local rows); da_src = T^T ds_src, da_dst = T_local^T
    ds_dst; dW = H^T dT, dH = dT W^T (every row: the halo rows are J).  With
    bf16 activations dT enters the products dW, dH as bf16 (their operands are
    bf16); grad_bf16 rounds the stored dH.  Returns dict(dW, da_src, da_dst, dT, dH)."""
    nL = part.n_local
    G = _f64(G)
    dY = G * (fwd["Hout"] > 0) if relu else G
    dT, ds_src, ds_dst = gat_attend_backward(part, fwd["T"], fwd["s_src"], fwd["s_dst"], fwd["alpha"], dY)
    if grad_bf16:
        dT = round_bf16(dT)  # stored after the attention-weighted sum, then after the score terms
    dT = dT + ds_src[:, None] * _f64(a_src)[None, :]
    dT[:nL] += ds_dst[:, None] * _f64(a_dst)[None, :]
    da_src = fwd["T"].T @ ds_src
    da_dst = fwd["T"][:nL].T @ ds_dst
    dTp = round_bf16(dT) if (bf16 or grad_bf16) else dT
    dW, dH = update_backward(dTp, dTp, _f64(H), _f64(W), relu=False, want_dz=True)
    if grad_bf16:
        dH = round_bf16(dH)
    return dict(dW=dW, da_src=da_src, da_dst=da_dst, dT=dT, dH=dH)


def gat_epoch(part, tables: Sequence[np.ndarray], Ws: Sequence[np.ndarray], a_srcs: Sequence[np.ndarray],
              a_dsts: Sequence[np.ndarray], labels_local: np.ndarray, bf16: bool = False, grad_bf16: bool = False,
              hidden_relu: bool = True):
    """One epoch of an L-layer GAT on one partition, composed like epoch():
    layer l pulls its halo rows from tables[l] (its local rows: the features,
    then the previous layer's output), ReLU on all layers but the last (none
    with hidden_relu=False), mean
    softmax cross-entropy over the local rows, then the backward layer by layer
    (G of layer l - 1 = the local rows of layer l's dH).  Returns a dict with
    the forward intermediates (fwd), Hout, loss, dW, da_src, da_dst, dH."""
    L = len(Ws)
    nL = part.n_local
    h_local = tables[0][part.local_ids]
    Hs, fwds = [], []
    for l in range(L):
        f = Ws[l].shape[0]
        H = np.zeros((part.n_local + part.n_halo, f), dtype=np.float64)
        H[:nL] = h_local[:, :f]
        if part.n_halo:
            H[nL:] = tables[l][part.halo_ids, :f]
        fw = gat_layer_forward(part, H, Ws[l], a_srcs[l], a_dsts[l], relu=hidden_relu and l < L - 1, bf16=bf16)
        Hs.append(H)
        fwds.append(fw)
        h_local = fw["Hout"]
    loss, G = softmax_ce(fwds[-1]["Hout"], labels_local)
    if grad_bf16:
        G = round_bf16(G)
    out = dict(fwd=fwds, H=Hs, Hout=[fw["Hout"] for fw in fwds], loss=loss, dW=[None] * L, da_src=[None] * L,
               da_dst=[None] * L, dH=[None] * L)
    for l in reversed(range(L)):
        bw = gat_layer_backward(part, fwds[l], Hs[l], G, Ws[l], a_srcs[l], a_dsts[l], relu=hidden_relu and l < L - 1,
                                bf16=bf16, grad_bf16=grad_bf16)
        out["dW"][l], out["da_src"][l], out["da_dst"][l] = bw["dW"], bw["da_src"], bw["da_dst"]
        out["dH"][l] = bw["dH"]
        G = bw["dH"][:nL]
    return out


# --------------------------------------------------------------------------
# Sylvie low-bit halo codec (Sylvie page, Quantizer / Dequantizer)
# --------------------------------------------------------------------------

def splitmix64(seed: int, k: int) -> int:
    """k-th output of the SplitMix64 stream seeded with `seed` (k >= 1)."""
    return int(_L().oracle_splitmix64(seed & (2**64 - 1), k & (2**64 - 1)))


def codec_row_bytes(f: int, bits: int) -> int:
    """Bytes of one packed row of f b-bit codes, padded to 16."""
    return (f * bits + 127) // 128 * 16


def quantize_rows(x: np.ndarray, ids: np.ndarray, bits: int, seed: int, ld_codes: Optional[int] = None):
    """(codes uint8 n x ld_codes, scale_zero float32 n x 2) of the rows of x.

    x holds values exactly representable in fp32 (fp32 or bf16 inputs); ids are
    the rows' table ids (they select the stochastic-rounding draws)."""
    xf = np.ascontiguousarray(x, dtype=np.float32)
    n, f = xf.shape
    ids64 = np.ascontiguousarray(ids, dtype=np.int64)
    assert ids64.shape[0] == n and bits in (1, 2, 4, 8)
    ldc = codec_row_bytes(f, bits) if ld_codes is None else ld_codes
    codes = np.zeros((n, ldc), dtype=np.uint8)
    sz = np.zeros((n, 2), dtype=np.float32)
    if n:
        _L().oracle_codec_quantize(_p(xf), f, n, f, _p(ids64), bits, seed & (2**64 - 1), _p(codes), ldc, _p(sz))
    return codes, sz


def dequantize_rows(codes: np.ndarray, scale_zero: np.ndarray, f: int, bits: int) -> np.ndarray:
    """float32 n x f: code * scale + zero, row by row."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    sz = np.ascontiguousarray(scale_zero, dtype=np.float32)
    n = c.shape[0]
    y = np.zeros((n, f), dtype=np.float32)
    if n:
        _L().oracle_codec_dequantize(_p(c), c.shape[1], _p(sz), n, f, bits, _p(y), f)
    return y

# --------------------------------------------------------------------------
# one layer and one epoch, composed step by step
# --------------------------------------------------------------------------

def layer_forward(part, H: np.ndarray, W: np.ndarray, agg: str, relu: bool, bf16: bool = False):
    """(Z, H') for all local rows.  H: float64 (n_local + n_halo) x f.

    bf16=True rounds the stored Z and H' to bf16, as the bf16 path stores them."""
    f = H.shape[1]
    Z = aggregate(part, H, f, agg)
    if bf16:
        Z = round_bf16(Z)
    Hout = update(Z, W, relu)
    if bf16:
        Hout = round_bf16(Hout)
    return Z, Hout


def layer_backward(part, T, G: np.ndarray, Hout: np.ndarray, Z: np.ndarray, W: np.ndarray, agg: str, relu: bool,
                   want_dh: bool = True, bf16: bool = False, grad_bf16: bool = False):
    """(dW, dZ, dH) with dH over all n_local + n_halo rows (None when not wanted).

    bf16=True: the activations are bf16, so dY enters the update's products as
    bf16 (like Z and W).  grad_bf16=True rounds the stored dZ and dH to bf16, as
    a path that stores activation gradients in bf16 does; with False they stay
    unrounded (the fp32 gradient storage of the bf16 workloads)."""
    dW, dZ = update_backward(G, Hout, Z, W, relu, want_dz=want_dh, dy_bf16=bf16)
    dH = None
    if want_dh:
        if grad_bf16:
            dZ = round_bf16(dZ)
        f = Z.shape[1] if agg == "gcn" else Z.shape[1] // 2
        dH = aggregate_backward(part, T, dZ, f, agg)
        if grad_bf16:
            dH = round_bf16(dH)
    return dW, dZ, dH


def layer_backward_reordered(part, T, G: np.ndarray, Hout: np.ndarray, Z: np.ndarray, W: np.ndarray, relu: bool,
                             bf16: bool = False, rows=None):
    """(dW, P, dH) of a GCN layer with the backward products in the other order
    (associativity of the chain rule of H = sigma(A^T H W), CAGNET page, GNN
    section): dY = G * 1[Hout > 0] (or G); dW = Z^T dY; P = A_hat^T dY over the
    output rows `rows` (default all n_local + n_halo); dH = P W^T.

    bf16=True: bf16 activations with fp32 gradients as the library's path takes
    them: dY rounded to bf16 (an operand of the products, as in layer_backward)
    and P rounded to bf16 once (the operand of dH = P W^T); dH itself is not
    rounded (fp32 gradient storage).  With bf16=False it equals layer_backward's
    dH exactly up to the order of the sums."""
    G, Hout, Z, W = _f64(G), _f64(Hout), _f64(Z), _f64(W)
    dY = G * (Hout > 0) if relu else G
    if bf16:
        dY = round_bf16(dY)
    dW, _ = update_backward(dY, Hout, Z, W, False, want_dz=False)
    P = aggregate_backward(part, T, dY, dY.shape[1], "gcn", rows=rows)
    if bf16:
        P = round_bf16(P)
    return dW, P, P @ W.T


def epoch(part, tables: Sequence[np.ndarray], Ws: Sequence[np.ndarray], labels_local: np.ndarray, agg: str,
          bf16: bool = False, grad_bf16: bool = False):
    """One full-graph epoch of an L-layer model on one partition.

    tables[l] (float64, n_table x f_l) hold the stale representations of layer l
    (tables[0]: the input features of every vertex).  Layer l pulls its halo
    rows from tables[l]; the local rows of layer 0 are the partition's own
    features (tables[0][local_ids]); the local rows of layer l > 0 are the
    previous layer's output, which is pushed into tables[l] (push of a copy).
    ReLU on every layer but the last.

    Precision: bf16=True rounds the activations (Z, H') to bf16, and the
    backward's products take dY in bf16 (their operands are bf16 like Z and W);
    grad_bf16=True also rounds the stored activation gradients (G, dZ, dH).
    Everything else is double.

    Returns a dict of every intermediate; G[l] is the gradient with respect to
    layer l's output that layer l's backward consumed.
    """
    L = len(Ws)
    nL = part.n_local
    T = transpose(part)
    Hs, Zs, Houts = [], [], []
    new_tables = [t.copy() for t in tables]
    h_local = tables[0][part.local_ids]
    for l in range(L):
        f = Ws[l].shape[0] if agg == "gcn" else Ws[l].shape[0] // 2
        H = np.zeros((part.n_local + part.n_halo, f), dtype=np.float64)
        H[:nL] = h_local[:, :f]
        if part.n_halo:
            H[nL:] = tables[l][part.halo_ids, :f]
        Z, Hout = layer_forward(part, H, Ws[l], agg, relu=l < L - 1, bf16=bf16)
        Hs.append(H)
        Zs.append(Z)
        Houts.append(Hout)
        if l + 1 < L:
            new_tables[l + 1][part.local_ids, :Hout.shape[1]] = Hout
        h_local = Hout
    loss, G = softmax_ce(Houts[-1], labels_local)
    if grad_bf16:
        G = round_bf16(G)
    dWs = [None] * L
    dHs = [None] * L
    Gs = [None] * L
    for l in reversed(range(L)):
        Gs[l] = G
        dW, _, dH = layer_backward(part, T, G, Houts[l], Zs[l], Ws[l], agg, relu=l < L - 1, want_dh=l > 0,
                                   bf16=bf16, grad_bf16=grad_bf16)
        dWs[l] = dW
        dHs[l] = dH
        if l > 0:
            G = dH[:nL]
    return dict(H=Hs, Z=Zs, Hout=Houts, loss=loss, dW=dWs, dH=dHs, G=Gs, tables=new_tables, T=T)
