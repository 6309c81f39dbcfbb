"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Index work (transpose, pull, push) must match bit for bit; floating point must
satisfy |x - r| <= tol * (|r| + rms(r)) with tol 1e-4 (fp32) or 2e-2 (bf16
storage, fp32 accumulation).  Small workloads are compared on every row; the
full-size ones on sampled rows (random rows plus the heaviest rows and rows just
past the heavy-row split), which the oracle computes one by one, and the
transpose at full size through properties that fix it uniquely.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.configs import TINY, WORKLOADS
from sparse_aggregation_dense_gb300 import PartitionModel, gnn, ld_for, padded
from tests._flip import close_bounded, epoch_bounds
from tests._gpu import (TOL, assert_ok, close, column_subset, gen_matrix, maybe_round, sample_with_heavy, to_device,
                        to_host, torch_dtype, widen)

pytestmark = pytest.mark.gpu

SMALL_FULL = ["er5k", "rmat131k"]
BIG_FULL = ["powerlaw233k", "sage2m", "rmat16m"]
ALL = list(WORKLOADS)
SEED = 0

_cache = {}


def problem(name: str, size: str):
    """(workload, partition, graph) with the graph built once per session."""
    key = (name, size)
    if key not in _cache:
        w = (TINY if size == "tiny" else WORKLOADS)[name]
        part = w.make(SEED)
        rp = torch.from_numpy(part.rowptr).cuda()
        ci = torch.from_numpy(part.colidx).cuda()
        deg = None if part.deg is None else torch.from_numpy(part.deg).cuda()
        g = gnn.graph_create(rp, ci, part.n_local, part.n_halo, deg, w.agg)
        _cache[key] = (w, part, g)
    return _cache[key]


def is_sampled(size: str, name: str) -> bool:
    return size == "full" and name in BIG_FULL


CASES = [(n, "tiny") for n in ALL] + [(n, "full") for n in ALL]


def case_id(c):
    return f"{c[0]}-{c[1]}"


# ---------------------------------------------------------------------------
# transpose (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_transpose_bit_exact(case):
    name, size = case
    w, part, g = problem(name, size)
    rT, cT, pT = (t.cpu().numpy() for t in gnn.graph_copy_transpose(g))
    if not is_sampled(size, name):
        orT, ocT, opT = oracle.transpose(part)
        np.testing.assert_array_equal(rT, orT)
        np.testing.assert_array_equal(cT, ocT)
        np.testing.assert_array_equal(pT, opT)
        return
    # full size: properties that determine the stable transpose uniquely
    nT = part.n_total
    cnt = np.bincount(part.colidx, minlength=nT)
    np.testing.assert_array_equal(rT, np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32))
    assert np.all(np.bincount(pT, minlength=part.nnz) == 1)  # a permutation of the entries
    row_of = np.repeat(np.arange(part.n_local, dtype=np.int32), np.diff(part.rowptr))
    np.testing.assert_array_equal(cT, row_of[pT])  # entry k came from row colidxT[k]
    trow = np.repeat(np.arange(nT, dtype=np.int32), cnt)
    np.testing.assert_array_equal(part.colidx[pT], trow)  # ... and carries column (transpose row) of k
    same_row = trow[1:] == trow[:-1]
    assert np.all(cT[1:][same_row] > cT[:-1][same_row])  # ascending source rows within a transpose row


# ---------------------------------------------------------------------------
# pull / push (bit-exact)
# ---------------------------------------------------------------------------

def _bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy()
    return t.contiguous().view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_pull_push_bit_exact(case):
    name, size = case
    w, part, g = problem(name, size)
    dt = w.dtype
    f = w.widths[0]
    tdt = torch_dtype(dt)
    table_h = gen_matrix(part.n_table, f, dt, SEED, synth.STREAM_FEATURES, w.feat_dist)
    table = to_device(table_h, dt, f)
    H = padded(part.n_total, f, tdt, "cuda")
    gnn.halo_pull(g, table, torch.from_numpy(part.halo_ids).cuda(), H)
    assert_ok(g)
    H_ref = np.zeros((part.n_total, table_h.shape[1]), dtype=table_h.dtype)
    assert oracle.halo_pull(table_h, part.halo_ids, H_ref, part.n_local, f) == oracle.OK
    np.testing.assert_array_equal(_bits(H[part.n_local:]), H_ref[part.n_local:, :f].view(
        np.int16 if dt == "bf16" else np.int32))
    # push fresh local rows into the table
    out_h = gen_matrix(part.n_local, f, dt, SEED, 77, "normal")
    out = to_device(out_h, dt, f)
    gnn.halo_push(g, out, torch.from_numpy(part.local_ids).cuda(), table)
    assert_ok(g)
    ref = table_h.copy()
    assert oracle.halo_push(out_h, part.n_local, f, part.local_ids, ref) == oracle.OK
    np.testing.assert_array_equal(_bits(table), ref[:, :f].view(np.int16 if dt == "bf16" else np.int32))


# ---------------------------------------------------------------------------
# forward layer
# ---------------------------------------------------------------------------

FWD_CASES = [(n, s, l) for (n, s) in CASES for l in range(WORKLOADS[n].layers)]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: f"{c[0]}-{c[1]}-L{c[2]}")
def test_forward_layer(case):
    name, size, l = case
    w, part, g = problem(name, size)
    dt, agg = w.dtype, w.agg
    tdt = torch_dtype(dt)
    f_in, f_out = w.widths[l], w.widths[l + 1]
    relu = l < w.layers - 1
    sage = agg == "sage"
    K = 2 * f_in if sage else f_in
    half = gnn.sage_half_offset(f_in, tdt)
    Kp = 2 * half if sage else f_in
    H_h = gen_matrix(part.n_total, f_in, dt, SEED, 100 + l)
    W = synth.glorot(K, f_out, SEED, synth.STREAM_WEIGHT + l)
    H = to_device(H_h, dt, f_in)
    Z = padded(part.n_local, Kp, tdt, "cuda", fill=None)
    Z.as_strided((part.n_local, Z.stride(0)), (Z.stride(0), 1)).fill_(7.0)  # padding must come back zero
    Hout = padded(part.n_local, f_out, tdt, "cuda")
    gnn.layer_forward(g, H, torch.from_numpy(W).cuda(), relu, Z, Hout)
    assert_ok(g)
    if is_sampled(size, name):
        rows = sample_with_heavy(part.rowptr, 1500, SEED)
        cols, cmap = column_subset(part.rowptr, part.colidx, rows, part.n_total)
        cols = np.union1d(cols, rows)
        cmap = -np.ones(part.n_total, np.int64)
        cmap[cols] = np.arange(cols.shape[0])
        Hsub = oracle.widen(gen_matrix(0, f_in, dt, SEED, 100 + l, ids=cols)[:, :f_in], dt == "bf16")
        hmap = cmap
    else:
        rows = np.arange(part.n_local, dtype=np.int64)
        Hsub = widen(H_h, dt, f_in)
        hmap = None
    wts = oracle.gcn_dinv(part) if not sage else oracle.sage_invcnt(part)
    Zr = oracle.aggregate(part, Hsub, f_in, agg, rows=rows, hmap=hmap, weights=wts)
    Zr = maybe_round(Zr, dt)
    Hr = oracle.update(Zr, maybe_round(W.astype(np.float64), dt), relu)
    rows_t = torch.from_numpy(rows).cuda()
    Zg = to_host(Z.index_select(0, rows_t))
    Hg = to_host(Hout.index_select(0, rows_t))
    tol = TOL[dt]
    if sage:
        close(Zg[:, :f_in], Zr[:, :f_in], 0.0, "Z self half (a copy)")
        close(Zg[:, half:half + f_in], Zr[:, f_in:], tol, "Z mean half")
        assert np.all(Zg[:, f_in:half] == 0) and np.all(Zg[:, half + f_in:] == 0)
    else:
        close(Zg, Zr, tol, "Z")
    close(Hg, Hr, tol, "H_out")
    # padding columns of the written rows (up to the 16-byte boundary) are zero
    ldz = Z.stride(0)
    buf = Z.as_strided((part.n_local, ldz), (ldz, 1)).index_select(0, rows_t).float().cpu().numpy()
    assert np.all(buf[:, (2 * half if sage else f_in):] == 0)


# ---------------------------------------------------------------------------
# backward layer
# ---------------------------------------------------------------------------

def _grad_dtypes(name: str, size: str, l: int):
    """Gradient storage of a backward case: fp32 always (bf16 workloads: bf16
    activations with fp32 gradients); bf16 gradients too for the bf16 workloads
    (every layer of the small graphs, one layer at full size)."""
    if WORKLOADS[name].dtype != "bf16":
        return ["f32"]
    return ["f32", "bf16"] if (size == "tiny" or l == 1) else ["f32"]


BWD_CASES = [(n, s, l, gd) for (n, s) in CASES for l in range(WORKLOADS[n].layers) for gd in _grad_dtypes(n, s, l)]


def _z_input(part, f_in, dt, sage, half, Kp, l):
    """Saved-aggregation input in the library's layout (stored values, rows of ld)."""
    tdt = torch_dtype(dt)
    ld = ld_for(Kp, tdt)
    a = gen_matrix(part.n_local, f_in, dt, SEED, 400 + l)
    if not sage:
        return a
    b = gen_matrix(part.n_local, f_in, dt, SEED, 500 + l)
    z = np.zeros((part.n_local, ld), dtype=a.dtype)
    z[:, :f_in] = a[:, :f_in]
    z[:, half:half + f_in] = b[:, :f_in]
    return z


def _compact(z_rows: np.ndarray, f_in: int, half: int, sage: bool) -> np.ndarray:
    """Widened rows of Z in the oracle's layout ([self | mean] without padding)."""
    if not sage:
        return z_rows[:, :f_in]
    return np.concatenate([z_rows[:, :f_in], z_rows[:, half:half + f_in]], axis=1)


def _sampled_transpose(part, n_rows, seed):
    """Output rows U of the transposed aggregation (random local and halo rows
    and the heaviest transpose rows), the transpose of the entries that reach
    them, and the input rows V those entries read."""
    nL, nT = part.n_local, part.n_total
    rowptrT = np.concatenate([[0], np.cumsum(np.bincount(part.colidx, minlength=nT))])
    U = sample_with_heavy(rowptrT, n_rows, seed)
    sel = np.zeros(nT, bool)
    sel[U] = True
    keep = sel[part.colidx]
    cnt = np.zeros(nL, np.int64)
    row_of = np.repeat(np.arange(nL), np.diff(part.rowptr))
    np.add.at(cnt, row_of[keep], 1)
    sub_rowptr = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
    sub = synth.Partition(sub_rowptr, part.colidx[keep], nL, part.n_halo, part.deg, part.local_ids,
                          part.halo_ids, part.n_table)
    T = oracle.transpose(sub)
    return U, T, np.unique(T[1]).astype(np.int64)


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"{c[0]}-{c[1]}-L{c[2]}-grad_{c[3]}")
def test_backward_layer(case):
    name, size, l, gd = case
    w, part, g = problem(name, size)
    dt, agg = w.dtype, w.agg
    tdt, gdt = torch_dtype(dt), torch_dtype(gd)
    f_in, f_out = w.widths[l], w.widths[l + 1]
    relu = l < w.layers - 1
    sage = agg == "sage"
    K = 2 * f_in if sage else f_in
    half = gnn.sage_half_offset(f_in, tdt)
    Kp = 2 * half if sage else f_in
    nL, nT = part.n_local, part.n_total
    G_h = gen_matrix(nL, f_out, gd, SEED, 200 + l)
    Ho_h = gen_matrix(nL, f_out, dt, SEED, 300 + l)
    Z_h = _z_input(part, f_in, dt, sage, half, Kp, l)
    W = synth.glorot(K, f_out, SEED, synth.STREAM_WEIGHT + l)
    G = to_device(G_h, gd, f_out)
    Ho = to_device(Ho_h, dt, f_out)
    Z = to_device(Z_h, dt, Kp)
    dW = torch.zeros((K, f_out), dtype=torch.float32, device="cuda")
    dZ = padded(nL, Kp, gdt, "cuda")
    dH = padded(nT, f_in, gdt, "cuda")
    gnn.layer_backward(g, G, Ho, Z, torch.from_numpy(W).cuda(), relu, dW, f_in, dZ=dZ, dH=dH, want_halo_grad=True)
    assert_ok(g)
    tol = TOL[dt]
    Wr = maybe_round(W.astype(np.float64), dt)
    dWg = dW.cpu().numpy()
    bf_a, bf_g = dt == "bf16", gd == "bf16"
    # dW: whole columns (every row summed) at full size, all of it otherwise
    cols = sorted({0, f_out // 2, f_out - 1}) if is_sampled(size, name) else list(range(f_out))
    if sage:  # the stored Z's two halves, in the oracle's compact order
        zc = np.concatenate([Z_h[:, :f_in], Z_h[:, half:half + f_in]], axis=1)
    else:
        zc = Z_h[:, :f_in]
    dWr = oracle.update_backward_dw_columns(G_h[:, :f_out], Ho_h[:, :f_out], zc, relu, cols, bf_a, bf_g)
    close(dWg[:, cols], dWr, tol, f"dW columns {cols}")
    # dH on output rows U (random local + halo rows and the heaviest transpose rows)
    if is_sampled(size, name):
        U, T, V = _sampled_transpose(part, 600, SEED + 1)
    else:
        U = np.arange(nT, dtype=np.int64)
        T = oracle.transpose(part)
        V = np.arange(nL, dtype=np.int64)
    vmap = -np.ones(nL, np.int64)
    vmap[V] = np.arange(V.shape[0])
    Gw, How = oracle.widen(G_h[V][:, :f_out], bf_g), oracle.widen(Ho_h[V][:, :f_out], bf_a)
    Zw = _compact(oracle.widen(Z_h[V], bf_a), f_in, half, sage)
    _, dZr = oracle.update_backward(Gw, How, Zw, Wr, relu, want_dz=True, dy_bf16=bf_a)
    dZr = maybe_round(dZr, gd)
    wts = oracle.gcn_dinv(part) if not sage else oracle.sage_invcnt(part)
    dHr = oracle.aggregate_backward(part, T, dZr, f_in, agg, rows=U, dmap=vmap, weights=wts)
    dHg = to_host(dH.index_select(0, torch.from_numpy(U).cuda()))
    close(dHg, dHr, tol, "dH")
    # the intermediate dZ rows as well (compact layout)
    dZg = to_host(dZ.index_select(0, torch.from_numpy(V[:2000]).cuda()))
    dZr_rows = dZr[:min(2000, V.shape[0])]
    if sage:
        close(dZg[:, :f_in], dZr_rows[:, :f_in], tol, "dZ self")
        close(dZg[:, half:half + f_in], dZr_rows[:, f_in:], tol, "dZ mean")
    else:
        close(dZg, dZr_rows, tol, "dZ")


# ---------------------------------------------------------------------------
# whole epoch: pulls, forwards, pushes, loss, backwards with halo gradients
# ---------------------------------------------------------------------------

EPOCH_CASES = ([(n, "tiny", gd) for n in ALL for gd in (["f32", "bf16"] if WORKLOADS[n].dtype == "bf16" else ["f32"])]
               + [(n, "full", "f32") for n in SMALL_FULL + ["sage2m"]])


def _load_model(w, part, gd="f32", **kw):
    dt = w.dtype
    tdt = torch_dtype(dt)
    m = PartitionModel(part, w.widths, w.agg, tdt, "cuda", grad_dtype=torch_dtype(gd), **kw)
    tables_h = []
    for l in range(w.layers):
        stream = synth.STREAM_FEATURES if l == 0 else synth.STREAM_TABLE + l
        t = gen_matrix(part.n_table, w.widths[l], dt, SEED, stream, w.feat_dist if l == 0 else "normal")
        tables_h.append(t)
        m.tables[l] = to_device(t, dt, w.widths[l])
    m.H[0][:part.n_local] = m.tables[0][torch.from_numpy(part.local_ids).cuda()]
    Ws = []
    for l in range(w.layers):
        K = (2 if w.agg == "sage" else 1) * w.widths[l]
        Ws.append(synth.glorot(K, w.widths[l + 1], SEED, synth.STREAM_WEIGHT + l))
        m.W[l].copy_(torch.from_numpy(Ws[l]))
    y = synth.labels(part.n_local, w.widths[-1], SEED, ids=part.local_ids)
    m.labels.copy_(torch.from_numpy(y))
    return m, tables_h, Ws, y


@pytest.mark.parametrize("case", EPOCH_CASES, ids=lambda c: f"{c[0]}-{c[1]}-grad_{c[2]}")
def test_epoch(case):
    name, size, gd = case
    w, part, _ = problem(name, size)
    dt = w.dtype
    m, tables_h, Ws, y = _load_model(w, part, gd)
    m.step()
    m.check_errors()
    bf = dt == "bf16"
    Wr = [maybe_round(x.astype(np.float64), dt) for x in Ws]
    ref = oracle.epoch(part, [widen(t, dt, f) for t, f in zip(tables_h, w.widths)], Wr, y, w.agg, bf16=bf,
                       grad_bf16=gd == "bf16")
    tol = TOL[dt]
    # Chained layers: a pre-activation closer to zero than the two sides can
    # differ may take the other ReLU branch; every gradient entry downstream of
    # such a decision is allowed its bound (tests/_flip.py), every other entry
    # is compared strictly elementwise.
    dWb, dHb, n_amb = epoch_bounds(part, ref, Wr, w.agg, bf)
    close(to_host(m.out_last), ref["Hout"][-1], tol, "logits")
    assert abs(float(m.loss.item()) - ref["loss"]) <= tol * abs(ref["loss"])
    for l in range(w.layers):
        close_bounded(m.dW[l].cpu().numpy(), ref["dW"][l], tol, dWb[l], f"dW[{l}] ({n_amb} ambiguous decisions)")
    for l in range(1, w.layers):
        close_bounded(to_host(m.dH[l]), ref["dH"][l], tol, dHb[l], f"dH[{l}] (local + halo)")
        pushed = to_host(m.tables[l].index_select(0, torch.from_numpy(part.local_ids).cuda()))
        close(pushed, ref["Hout"][l - 1], tol, f"pushed table {l}")


def test_epoch_reordered_backward():
    # the epoch with layers l > 0 differentiated in the other product order agrees with the oracle's epoch to the
    # bf16 tolerance: the two orders differ by the rounding of P = A_hat^T dY to bf16 (|error| <= 2^-9 |P| per
    # element, a few 1e-3 of dH's scale after the product with W^T)
    w, part, _ = problem("rmat16m", "tiny")
    m, tables_h, Ws, y = _load_model(w, part, "f32", reorder=True)
    m.step()
    m.check_errors()
    Wr = [maybe_round(x.astype(np.float64), "bf16") for x in Ws]
    ref = oracle.epoch(part, [widen(t, "bf16", f) for t, f in zip(tables_h, w.widths)], Wr, y, w.agg, bf16=True)
    dWb, dHb, n_amb = epoch_bounds(part, ref, Wr, w.agg, True)
    tol = TOL["bf16"]
    for l in range(w.layers):
        close_bounded(m.dW[l].cpu().numpy(), ref["dW"][l], tol, dWb[l], f"dW[{l}] ({n_amb} ambiguous decisions)")
    for l in range(1, w.layers):
        close_bounded(to_host(m.dH[l]), ref["dH"][l], tol, dHb[l], f"dH[{l}] (local + halo)")
    with pytest.raises(ValueError):
        m.set_grad_dtype(torch.bfloat16)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _custom_graph(rows, n_halo, agg="gcn", deg=None):
    """Graph from a list of column lists (rows of the block)."""
    rowptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    colidx = np.array([c for r in rows for c in r], dtype=np.int32)
    n_local = len(rows)
    part = synth.Partition(rowptr, colidx, n_local, n_halo, deg, np.arange(n_local, dtype=np.int64),
                           np.arange(n_local, n_local + n_halo, dtype=np.int64), n_local + n_halo)
    g = gnn.graph_create(torch.from_numpy(rowptr).cuda(), torch.from_numpy(colidx).cuda(), n_local, n_halo,
                         None if deg is None else torch.from_numpy(deg).cuda(), agg)
    return part, g


def _run_layer_pair(part, g, agg, dt, f_in, f_out, relu, seed=3, gd=None):
    """Forward + backward on generator inputs; compare every row with the oracle.
    gd: the gradients' dtype (default: the activations')."""
    gd = gd or dt
    tdt, gdt = torch_dtype(dt), torch_dtype(gd)
    sage = agg == "sage"
    K = 2 * f_in if sage else f_in
    half = gnn.sage_half_offset(f_in, tdt)
    Kp = 2 * half if sage else f_in
    nL, nT = part.n_local, part.n_total
    H_h = gen_matrix(nT, f_in, dt, seed, 1)
    W = synth.glorot(K, f_out, seed, 2)
    Z = padded(nL, Kp, tdt, "cuda")
    Ho = padded(nL, f_out, tdt, "cuda")
    Wd = torch.from_numpy(W).cuda()
    gnn.layer_forward(g, to_device(H_h, dt, f_in), Wd, relu, Z, Ho)
    tol = TOL[dt]
    Zr = maybe_round(oracle.aggregate(part, widen(H_h, dt, f_in), f_in, agg), dt)
    Hr = oracle.update(Zr, maybe_round(W.astype(np.float64), dt), relu)
    Zg = to_host(Z)
    if sage:
        close(Zg[:, :f_in], Zr[:, :f_in], tol, "Z self")
        close(Zg[:, half:half + f_in], Zr[:, f_in:], tol, "Z mean")
    else:
        close(Zg, Zr, tol, "Z")
    close(to_host(Ho), Hr, tol, "H_out")
    G_h = gen_matrix(nL, f_out, gd, seed, 4)
    dW = torch.zeros((K, f_out), dtype=torch.float32, device="cuda")
    dZ = padded(nL, Kp, gdt, "cuda")
    dH = padded(nT, f_in, gdt, "cuda")
    gnn.layer_backward(g, to_device(G_h, gd, f_out), Ho, Z, Wd, relu, dW, f_in, dZ=dZ, dH=dH, want_halo_grad=True)
    assert_ok(g)
    Zc = np.concatenate([Zg[:, :f_in], Zg[:, half:half + f_in]], axis=1) if sage else Zg
    dWr, dZr = oracle.update_backward(widen(G_h, gd, f_out), to_host(Ho), Zc, maybe_round(W.astype(np.float64), dt),
                                      relu, dy_bf16=dt == "bf16")
    close(dW.cpu().numpy(), dWr, tol, "dW")
    dHr = oracle.aggregate_backward(part, oracle.transpose(part), maybe_round(dZr, gd), f_in, agg)
    close(to_host(dH), dHr, tol, "dH")
    return Z, Ho, dW, dH


PRECISIONS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]  # (activations, gradients)


@pytest.mark.parametrize("dt,gd", PRECISIONS)
@pytest.mark.parametrize("agg", ["gcn", "sage"])
@pytest.mark.parametrize("f_in,f_out", [(1, 3), (5, 41), (47, 172), (100, 47), (602, 41), (256, 256)])
def test_ragged_widths(dt, gd, agg, f_in, f_out):
    part = synth.chunglu_partition(1500, 12000, 16.0, 3, seed=5)
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda(), agg)
    _run_layer_pair(part, g, agg, dt, f_in, f_out, relu=True, gd=gd)


@pytest.mark.parametrize("dt,gd,f_in", [("f32", "f32", 1024), ("bf16", "bf16", 2048), ("bf16", "f32", 1024)])
def test_maximum_widths(dt, gd, f_in):
    # rows of 4096 bytes, the widest the aggregation takes (in the activations' and the gradients' types); a
    # bf16 update with K = 2048 runs its backward in eight 256-column slices
    part = synth.chunglu_partition(1500, 12000, 16.0, 3, seed=7)
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda(), "gcn")
    _run_layer_pair(part, g, "gcn", dt, f_in, 16, relu=True, gd=gd)
    # eight columns wider are refused before anything runs: the forward's rows (same dtype), or with fp32
    # gradients the backward's fp32 rows
    tdt, gdt = torch_dtype(dt), torch_dtype(gd)
    fw = f_in + 8
    H = padded(part.n_total, fw, tdt, "cuda")
    Z = padded(part.n_local, fw, tdt, "cuda")
    Ho = padded(part.n_local, 16, tdt, "cuda")
    W = torch.zeros((fw, 16), device="cuda")
    with pytest.raises(gnn.GnnError) as e:
        if dt == gd:
            gnn.layer_forward(g, H, W, True, Z, Ho)
        else:
            gnn.layer_backward(g, padded(part.n_local, 16, gdt, "cuda"), Ho, Z, W, True,
                               torch.zeros((fw, 16), device="cuda"), fw, dZ=padded(part.n_local, fw, gdt, "cuda"),
                               dH=padded(part.n_total, fw, gdt, "cuda"), want_halo_grad=True)
    assert e.value.status == gnn.GNN_EUNSUPPORTED


@pytest.mark.parametrize("dt,gd", PRECISIONS)
@pytest.mark.parametrize("agg", ["gcn", "sage"])
def test_heavy_rows_and_columns(dt, gd, agg):
    # one hub row with 3000 entries (several chunks and a partial one) and one hub
    # column referenced by 2500 rows; rows of exactly 512 and 513 entries
    rng = np.random.default_rng(11)
    nL, nH = 3000, 700
    nT = nL + nH
    hub = nL + 5
    sizes = {7: 2999, 11: 511, 13: 512}  # entries besides the self loop
    rows = []
    for v in range(nL):
        pool = np.setdiff1d(np.arange(nT), [v, hub])
        if v in sizes:
            cols = set(rng.choice(pool, sizes[v], replace=False).tolist())
        else:
            cols = set(rng.choice(pool, int(rng.integers(0, 12)), replace=False).tolist())
            if v < 2500:
                cols.add(hub)  # hub halo column: a heavy transpose row
        rows.append(sorted(cols | {v}))
    part, g = _custom_graph(rows, nH, agg)
    deg = np.diff(part.rowptr)
    assert deg[7] == 3000 and deg[11] == 512 and deg[13] == 513
    assert np.sum(part.colidx == hub) > 2000
    a = _run_layer_pair(part, g, agg, dt, 96, 40, relu=True, gd=gd)
    b = _run_layer_pair(part, g, agg, dt, 96, 40, relu=True, gd=gd)
    for x, y in zip(a, b):  # bitwise reproducible
        assert torch.equal(x, y)


def test_no_halo_empty_rows_and_single_row():
    # no halo, a row with no entries at all (no self loop), a row with only itself
    rows = [[0, 1], [], [2], [0, 1, 3], [3, 4]]
    deg = np.array([3, 2, 1, 2, 2], dtype=np.float32)
    part, g = _custom_graph(rows, 0, "gcn", deg)
    Z, Ho, dW, dH = _run_layer_pair(part, g, "gcn", "f32", 8, 4, relu=False)
    assert float(Z[1].abs().max()) == 0.0
    part1, g1 = _custom_graph([[0, 1]], 1, "gcn")
    _run_layer_pair(part1, g1, "gcn", "f32", 16, 8, relu=True)
    part2, g2 = _custom_graph([[0, 1]], 1, "sage")
    _run_layer_pair(part2, g2, "sage", "bf16", 16, 8, relu=True)


def test_bad_ids_are_reported_and_rows_left_alone():
    part = synth.er_partition(300, 200, 0.05, seed=1)
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda(), "gcn")
    f = 12
    table_h = gen_matrix(part.n_table, f, "f32", 0, 1)
    table = to_device(table_h, "f32", f)
    ids = part.halo_ids.copy()
    ids[5] = part.n_table  # out of range
    ids[6] = -1
    H = padded(part.n_total, f, torch.float32, "cuda")
    H.fill_(-3.0)
    gnn.halo_pull(g, table, torch.from_numpy(ids).cuda(), H)
    assert gnn.get_error(g) == gnn.GNN_EINDEX
    assert_ok(g)  # cleared
    Hh = H.cpu().numpy()
    assert np.all(Hh[part.n_local + 5] == -3.0) and np.all(Hh[part.n_local + 6] == -3.0)
    good = [i for i in range(part.n_halo) if i not in (5, 6)]
    np.testing.assert_array_equal(Hh[part.n_local + np.array(good)], table_h[ids[good], :f])
    # push with a repeated id: neither copy is written, the others are
    lids = part.local_ids.copy()
    lids[9] = lids[3]
    before = table.cpu().numpy().copy()
    out_h = gen_matrix(part.n_local, f, "f32", 0, 9)
    gnn.halo_push(g, to_device(out_h, "f32", f), torch.from_numpy(lids).cuda(), table)
    assert gnn.get_error(g) == gnn.GNN_EINDEX
    after = table.cpu().numpy()
    np.testing.assert_array_equal(after[lids[3]], before[lids[3]])
    ok = [v for v in range(part.n_local) if v not in (3, 9)]
    np.testing.assert_array_equal(after[lids[ok]], out_h[ok, :f])
    # a second, clean push after the failed one works (claim generations advance)
    gnn.halo_push(g, to_device(out_h, "f32", f), torch.from_numpy(part.local_ids).cuda(), table)
    assert_ok(g)
    np.testing.assert_array_equal(table.cpu().numpy()[part.local_ids], out_h[:, :f])


def test_bad_csr_is_rejected():
    rowptr = torch.tensor([0, 2, 3], dtype=torch.int32, device="cuda")
    colidx = torch.tensor([0, 5, 1], dtype=torch.int32, device="cuda")  # 5 >= n_local + n_halo = 4
    with pytest.raises(gnn.GnnError) as e:
        gnn.graph_create(rowptr, colidx, 2, 2, None, "gcn")
    assert e.value.status == gnn.GNN_EINDEX
    rowptr2 = torch.tensor([0, 3, 2], dtype=torch.int32, device="cuda")  # not monotone
    with pytest.raises(gnn.GnnError):
        gnn.graph_create(rowptr2, colidx[:2], 2, 2, None, "gcn")


# ---------------------------------------------------------------------------
# softmax cross-entropy (training-harness helper): G elementwise, the mean loss,
# the padding of G left alone, a bad label giving a NaN loss
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt,gd", PRECISIONS)
@pytest.mark.parametrize("n,C", [(1, 1), (37, 7), (1000, 41), (33333, 172), (5000, 256), (3000, 300), (700, 520)])
def test_softmax_ce(dt, gd, n, C):
    tdt, gdt = torch_dtype(dt), torch_dtype(gd)
    X_h = gen_matrix(n, C, dt, SEED, 55)
    X = to_device(X_h, dt, C)
    y = synth.labels(n, C, SEED)
    G = padded(n, C, gdt, "cuda", fill=None)
    G.as_strided((n, G.stride(0)), (G.stride(0), 1)).fill_(7.0)
    row_loss = torch.empty(n, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    gnn.softmax_ce(X, torch.from_numpy(y).cuda(), G, row_loss, loss)
    ref_loss, ref_G = oracle.softmax_ce(widen(X_h, dt, C), y)
    close(to_host(G), maybe_round(ref_G, gd), TOL[dt], "G")
    assert abs(float(loss.item()) - ref_loss) <= 1e-5 * abs(ref_loss)  # fp32 sums of exact-input rows
    pad = G.as_strided((n, G.stride(0)), (G.stride(0), 1))[:, C:]
    assert bool(torch.all(pad == 7.0))


def test_softmax_ce_bad_label_gives_nan():
    n, C = 100, 16
    X = to_device(gen_matrix(n, C, "f32", SEED, 56), "f32", C)
    y = synth.labels(n, C, SEED)
    y[17] = C  # out of range
    G = padded(n, C, torch.float32, "cuda")
    row_loss = torch.empty(n, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    gnn.softmax_ce(X, torch.from_numpy(y).cuda(), G, row_loss, loss)
    assert np.isnan(float(loss.item()))


# ---------------------------------------------------------------------------
# overlapped schedule: pulls and pushes on a second stream give the same epoch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", [(n, "tiny") for n in ALL] + [("rmat131k", "full")], ids=case_id)
def test_overlapped_epoch_matches_sequential(case):
    name, size = case
    w, part, _ = problem(name, size)
    results = []
    for overlap in (False, True):
        m, _, _, _ = _load_model(w, part)
        if overlap:
            m.overlap, m.side = True, torch.cuda.Stream()
        for _ in range(2):  # the second epoch reads the tables the first one pushed
            m.step()
        m.check_errors()
        torch.cuda.synchronize()
        results.append([m.loss.cpu(), m.out_last.float().cpu()] + [d.cpu() for d in m.dW] +
                       [t.float().cpu() for t in m.tables[1:]])
    for a, b in zip(*results):
        assert torch.equal(a, b)


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("name", ["rmat131k", "sage2m", "rmat16m"])
def test_staged_inputs_match_synchronous_copies(name, overlap):
    # three epochs whose inputs change every epoch: copied before each step on
    # the compute stream, or staged during the previous step on the copy stream
    w = TINY[name]
    part = w.make(0)
    dt = w.dtype
    xs = []
    for e in range(3):
        x = gen_matrix(part.n_local, w.widths[0], dt, SEED, 900 + e)  # n_local x the row stride of H[0]
        x = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(x)
        xs.append(x.pin_memory())
    ys = [torch.from_numpy(synth.labels(part.n_local, w.widths[-1], SEED, 910 + e)).pin_memory() for e in range(3)]
    results = []
    for staged in (False, True):
        m, _, _, _ = _load_model(w, part)
        if overlap:
            m.overlap, m.side = True, torch.cuda.Stream()
        h0 = m._h0_local(xs[0].shape[1])
        if staged:
            h0.copy_(xs[0], non_blocking=True)
            m.labels.copy_(ys[0], non_blocking=True)
        for e in range(3):
            if staged:
                if e + 1 < 3:
                    m.stage_inputs(xs[e + 1], ys[e + 1])
            else:
                h0.copy_(xs[e], non_blocking=True)
                m.labels.copy_(ys[e], non_blocking=True)
            m.step()
        m.check_errors()
        torch.cuda.synchronize()
        results.append([m.loss.cpu(), m.out_last.float().cpu()] + [d.cpu() for d in m.dW] +
                       [t.float().cpu() for t in m.tables[1:]])
    for a, b in zip(*results):
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# narrow layers (multiplication first: A (H W)) against the textbook order
# ---------------------------------------------------------------------------

NARROW_CASES = [(n, "tiny", l) for n in ["er5k", "rmat131k", "powerlaw233k", "rmat16m"]
                for l in range(TINY[n].layers) if TINY[n].widths[l + 1] < TINY[n].widths[l]]


@pytest.mark.parametrize("case", NARROW_CASES, ids=lambda c: f"{c[0]}-{c[1]}-L{c[2]}")
def test_narrow_layer_matches_oracle(case):
    name, size, l = case
    w, part, g = problem(name, size)
    dt = w.dtype
    tdt = torch_dtype(dt)
    f_in, f_out = w.widths[l], w.widths[l + 1]
    relu = l < w.layers - 1
    nL, nT = part.n_local, part.n_total
    H_h = gen_matrix(nT, f_in, dt, SEED, 500 + l)
    W = synth.glorot(f_in, f_out, SEED, synth.STREAM_WEIGHT + l)
    Wr = maybe_round(W.astype(np.float64), dt)
    H = to_device(H_h, dt, f_in)
    T = padded(nT, f_out, tdt, "cuda")
    Hout = padded(nL, f_out, tdt, "cuda")
    gnn.layer_forward_narrow(g, H, torch.from_numpy(W).cuda(), relu, T, Hout)
    assert_ok(g)
    Hw = widen(H_h, dt, f_in)
    Zr, Hr = oracle.layer_forward(part, Hw, Wr, "gcn", relu)
    close(to_host(Hout), Hr, TOL[dt], "H_out")
    close(to_host(T), Hw @ Wr, TOL[dt], "T = H W")
    # backward with the GPU's H_out on both sides (the same ReLU mask)
    G_h = gen_matrix(nL, f_out, dt, SEED, 600 + l)
    G = to_device(G_h, dt, f_out)
    P = padded(nT, f_out, tdt, "cuda")
    dH = padded(nT, f_in, tdt, "cuda")
    dW = torch.zeros((f_in, f_out), dtype=torch.float32, device="cuda")
    gnn.layer_backward_narrow(g, G, Hout, H, torch.from_numpy(W).cuda(), relu, dW, P, dH)
    assert_ok(g)
    dWr, _, dHr = oracle.layer_backward(part, oracle.transpose(part), widen(G_h, dt, f_out), to_host(Hout), Zr, Wr,
                                        "gcn", relu, want_dh=True)
    close(dW.cpu().numpy().astype(np.float64), dWr, TOL[dt], "dW")
    close(to_host(dH), dHr, TOL[dt], "dH (local and halo rows)")


# ---------------------------------------------------------------------------
# failure detection: a bounded device wait that runs out is reported, and the
# context stays usable (no fault, no hang)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_expired_wait_is_reported_and_the_next_call_is_exact(dt):
    w, part, g = problem("rmat131k", "tiny")
    tdt = torch_dtype(dt)
    f_in, f_out = 64, 16
    H_h = gen_matrix(part.n_total, f_in, dt, SEED, 31)
    W = torch.from_numpy(synth.glorot(f_in, f_out, SEED, 32)).cuda()
    H = to_device(H_h, dt, f_in)
    Z = padded(part.n_local, f_in, tdt, "cuda")
    Hout = padded(part.n_local, f_out, tdt, "cuda")
    assert_ok(g)
    gnn.debug_expire_next_wait(200_000_000)  # 0.2 s
    gnn.layer_forward(g, H, W, True, Z, Hout)
    assert gnn.get_error(g) == gnn.GNN_ETIMEOUT
    assert_ok(g)  # the word was cleared; the context answers
    # the hook was one-shot: the same call now runs to completion and is exact
    gnn.layer_forward(g, H, W, True, Z, Hout)
    assert_ok(g)
    Zr = maybe_round(oracle.aggregate(part, widen(H_h, dt, f_in), f_in, "gcn"), dt)
    close(to_host(Z), Zr, TOL[dt], "Z after the expired wait")


@pytest.mark.parametrize("f_in,f_out,relu,halo", [(256, 256, True, True), (128, 256, False, True),
                                                  (256, 64, True, False), (200, 40, True, True)])
def test_reordered_backward_matches_oracle(f_in, f_out, relu, halo):
    # the GCN backward in the other product order (P = A_hat^T dY in bf16, dH = P W^T) against the oracle's
    # own reading of that order: R-MAT partition, bf16 activations, fp32 gradients, ragged widths included
    part = TINY["rmat16m"].make(0)
    nL, nT = part.n_local, part.n_total
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), nL,
                         part.n_halo, None, "gcn")
    bf = torch.bfloat16
    Zh = synth.features(nL, f_in, ld_for(f_in, bf), SEED, 61, "normal", bf16=True)
    Oh = synth.features(nL, f_out, ld_for(f_out, bf), SEED, 62, "normal", bf16=True)
    Gh = synth.features(nL, f_out, ld_for(f_out, torch.float32), SEED, 63, "normal")
    W = synth.glorot(f_in, f_out, SEED, 64)
    Z = torch.from_numpy(Zh.view(np.int16)).cuda().view(bf)[:, :f_in]
    Hout = torch.from_numpy(Oh.view(np.int16)).cuda().view(bf)[:, :f_out]
    G = torch.from_numpy(Gh).cuda()[:, :f_out]
    rows = nT if halo else nL
    dW = torch.full((f_in, f_out), float("nan"), dtype=torch.float32, device="cuda")
    P = padded(rows, f_out, bf, "cuda")
    dH = padded(rows, f_in, torch.float32, "cuda")
    gnn.layer_backward_reordered(g, G, Hout, Z, torch.from_numpy(W).cuda(), relu, dW, P, dH, want_halo_grad=halo)
    torch.cuda.synchronize()
    assert gnn.get_error(g) == gnn.GNN_OK
    Wr = oracle.round_bf16(W.astype(np.float64))
    dWr, Pr, dHr = oracle.layer_backward_reordered(
        part, oracle.transpose(part), Gh[:, :f_out], oracle.widen(Oh[:, :f_out], True),
        oracle.widen(Zh[:, :f_in], True), Wr, relu, bf16=True, rows=None if halo else np.arange(nL))
    close(dW.cpu().numpy(), dWr, TOL["bf16"], "dW")
    close(P.float().cpu().numpy(), Pr[:rows], TOL["bf16"], "P")
    close(dH.cpu().numpy(), dHr[:rows], TOL["bf16"], "dH")
    gnn.graph_destroy(g)


@pytest.mark.parametrize("l", [1, 2])
def test_reordered_backward_full_size_sampled(l):
    # the bench partition's layers 2 and 1 in the other product order, in the launch configuration the bench's
    # other_order step uses: dW on whole columns, P and dH on sampled output rows (local, halo, heaviest)
    w, part, g = problem("rmat16m", "full")
    f_in, f_out = w.widths[l], w.widths[l + 1]
    relu = l < w.layers - 1
    nL, nT = part.n_local, part.n_total
    G_h = gen_matrix(nL, f_out, "f32", SEED, 200 + l)
    Ho_h = gen_matrix(nL, f_out, "bf16", SEED, 300 + l)
    Z_h = gen_matrix(nL, f_in, "bf16", SEED, 400 + l)
    W = synth.glorot(f_in, f_out, SEED, synth.STREAM_WEIGHT + l)
    dW = torch.full((f_in, f_out), float("nan"), dtype=torch.float32, device="cuda")
    P = padded(nT, f_out, torch.bfloat16, "cuda")
    dH = padded(nT, f_in, torch.float32, "cuda")
    gnn.layer_backward_reordered(g, to_device(G_h, "f32", f_out), to_device(Ho_h, "bf16", f_out),
                                 to_device(Z_h, "bf16", f_in), torch.from_numpy(W).cuda(), relu, dW, P, dH)
    assert_ok(g)
    tol = TOL["bf16"]
    cols = sorted({0, f_out // 2, f_out - 1})
    dWr = oracle.update_backward_dw_columns(G_h[:, :f_out], Ho_h[:, :f_out], Z_h[:, :f_in], relu, cols, True, False)
    close(dW.cpu().numpy()[:, cols], dWr, tol, f"dW columns {cols}")
    U, T, V = _sampled_transpose(part, 600, SEED + 2)
    vmap = -np.ones(nL, np.int64)
    vmap[V] = np.arange(V.shape[0])
    Gw, How = oracle.widen(G_h[V][:, :f_out], False), oracle.widen(Ho_h[V][:, :f_out], True)
    dY = oracle.round_bf16(Gw * (How > 0) if relu else Gw)  # the product operand dY, as the layer rounds it
    Pr = oracle.round_bf16(oracle.aggregate_backward(part, T, dY, f_out, "gcn", rows=U, dmap=vmap,
                                                     weights=oracle.gcn_dinv(part)))
    Uc = torch.from_numpy(U).cuda()
    close(P.index_select(0, Uc).float().cpu().numpy(), Pr, tol, "P")
    close(to_host(dH.index_select(0, Uc)), Pr @ oracle.round_bf16(W.astype(np.float64)).T, tol, "dH")


def test_reordered_backward_refuses_other_aggregations():
    # GraphSAGE graphs (and any precision but bf16 activations with fp32 gradients) are not taken
    part = TINY["sage2m"].make(0)
    g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(), part.n_local,
                         part.n_halo, torch.from_numpy(part.deg).cuda() if part.deg is not None else None, "sage")
    f = 64
    bf = torch.bfloat16
    Z = padded(part.n_local, f, bf, "cuda")
    G = padded(part.n_local, f, torch.float32, "cuda")
    W = torch.zeros((f, f), dtype=torch.float32, device="cuda")
    with pytest.raises(gnn.GnnError) as e:
        gnn.layer_backward_reordered(g, G, Z, Z, W, False, W.clone(), padded(part.n_total, f, bf, "cuda"),
                                     padded(part.n_total, f, torch.float32, "cuda"))
    assert e.value.status == gnn.GNN_EUNSUPPORTED
    gnn.graph_destroy(g)
