"""Pins of the CPU oracle against facts fixed outside it (no GPU needed).

Each test checks the oracle against something it does not compute itself: a dense
matrix formulation evaluated with numpy matmul, a closed form, an invariant of
the normalised adjacency, central finite differences, an independent library
routine (scipy.sparse, torch CPU casts) or a hand-derived fixture.
"""
import json
import os

import numpy as np
import pytest
import scipy.sparse as sp

import oracle
import synth
from tests._problems import (circulant, dense_gcn_block, dense_mean_block, partition_from_dense,
                             random_sym_adjacency)

HERE = os.path.dirname(os.path.abspath(__file__))


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


def _tiny(seed, N=40, nL=24, p=0.15, halo_all=False, pass_deg=True):
    A = random_sym_adjacency(N, p, seed)
    local = np.arange(nL)
    part, cols = partition_from_dense(A, local, halo_all=halo_all, pass_deg=pass_deg)
    return A, local, part, cols


# ---------------------------------------------------------------------------
# T1: dense brute force (CAGNET GNN section: H = sigma(A^T H W), A normalised)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gcn_forward_matches_dense(seed):
    A, local, part, cols = _tiny(seed)
    rng = np.random.default_rng(100 + seed)
    f = 7
    H = rng.standard_normal((part.n_total, f))
    Z = oracle.aggregate(part, H, f, "gcn")
    Zd = dense_gcn_block(A, local, cols) @ H
    assert _rel(Z, Zd) < 1e-13


@pytest.mark.parametrize("seed", [0, 1])
def test_gcn_backward_matches_dense(seed):
    A, local, part, cols = _tiny(seed)
    rng = np.random.default_rng(200 + seed)
    f = 5
    dZ = rng.standard_normal((part.n_local, f))
    T = oracle.transpose(part)
    dH = oracle.aggregate_backward(part, T, dZ, f, "gcn")
    dHd = dense_gcn_block(A, local, cols).T @ dZ
    assert dH.shape == (part.n_total, f)
    assert _rel(dH, dHd) < 1e-13


@pytest.mark.parametrize("seed", [0, 1])
def test_reordered_backward_is_the_dense_chain_rule(seed):
    # dH = (A_hat^T dY) W^T, the other order of the same products: against the dense
    # A_hat_block^T (dY W^T) and the textbook-order oracle; with bf16 rounding, P is
    # rounded once (dense: the same rounding applied to A_hat^T dY)
    A, local, part, cols = _tiny(seed)
    rng = np.random.default_rng(300 + seed)
    f_in, f_out = 6, 4
    Z = rng.standard_normal((part.n_local, f_in))
    W = rng.standard_normal((f_in, f_out))
    G = rng.standard_normal((part.n_local, f_out))
    Hout = rng.standard_normal((part.n_local, f_out))
    T = oracle.transpose(part)
    Ad = dense_gcn_block(A, local, cols)
    dY = G * (Hout > 0)
    dW, P, dH = oracle.layer_backward_reordered(part, T, G, Hout, Z, W, relu=True)
    assert _rel(dW, Z.T @ dY) < 1e-13
    assert _rel(P, Ad.T @ dY) < 1e-13
    assert _rel(dH, Ad.T @ (dY @ W.T)) < 1e-12
    dW_t, _, dH_t = oracle.layer_backward(part, T, G, Hout, Z, W, "gcn", relu=True)
    assert _rel(dW, dW_t) < 1e-13 and _rel(dH, dH_t) < 1e-12
    dWb, Pb, dHb = oracle.layer_backward_reordered(part, T, G, Hout, Z, W, relu=True, bf16=True)
    dYb = oracle.round_bf16(dY)
    assert np.array_equal(Pb, oracle.round_bf16(Pb)) and _rel(Pb, oracle.round_bf16(Ad.T @ dYb)) < 1e-13
    assert _rel(dHb, oracle.round_bf16(Ad.T @ dYb) @ W.T) < 1e-12 and _rel(dWb, Z.T @ dYb) < 1e-13
    # only the halo-free rows
    rows = np.arange(part.n_local)
    _, Pr, dHr = oracle.layer_backward_reordered(part, T, G, Hout, Z, W, relu=True, rows=rows)
    assert _rel(dHr, dH[:part.n_local]) < 1e-13


@pytest.mark.parametrize("seed", [0, 3])
def test_sage_forward_backward_match_dense(seed):
    A, local, part, cols = _tiny(seed, N=36, nL=20, p=0.2)
    rng = np.random.default_rng(300 + seed)
    f = 6
    H = rng.standard_normal((part.n_total, f))
    Z = oracle.aggregate(part, H, f, "sage")
    M = dense_mean_block(A, local, cols)
    assert _rel(Z[:, :f], H[:part.n_local]) == 0.0
    assert _rel(Z[:, f:], M @ H) < 1e-13
    dZ = rng.standard_normal((part.n_local, 2 * f))
    dH = oracle.aggregate_backward(part, oracle.transpose(part), dZ, f, "sage")
    ref = M.T @ dZ[:, f:]
    ref[:part.n_local] += dZ[:, :f]
    assert _rel(dH, ref) < 1e-13


def test_update_forward_backward_match_dense():
    rng = np.random.default_rng(7)
    n, K, N = 23, 9, 5  # K != N so a transposed operand cannot pass
    Z = rng.standard_normal((n, K))
    W = rng.standard_normal((K, N))
    for relu in (False, True):
        Hout = oracle.update(Z, W, relu)
        Y = Z @ W
        assert _rel(Hout, np.maximum(Y, 0.0) if relu else Y) < 1e-14
        G = rng.standard_normal((n, N))
        dW, dZ = oracle.update_backward(G, Hout, Z, W, relu)
        dY = G * (Hout > 0) if relu else G
        assert dW.shape == (K, N) and dZ.shape == (n, K)
        assert _rel(dW, Z.T @ dY) < 1e-13
        assert _rel(dZ, dY @ W.T) < 1e-13
        sel = [(0, 0), (K - 1, N - 1), (3, 2)]
        ent = oracle.update_backward_dw_entries(G, Hout, Z, relu, sel)
        assert _rel(ent, np.array([dW[k, j] for k, j in sel])) < 1e-14


@pytest.mark.parametrize("bf16", [False, True])
def test_dw_columns_streamed_over_row_blocks_match_dense(bf16):
    # the full-size dW check streams rows in blocks; on a small case it equals
    # the dense product (ragged last block, strided stored rows, bf16 bits)
    rng = np.random.default_rng(17)
    n, K, N = 1037, 12, 9
    Zf = rng.standard_normal((n, K + 4)).astype(np.float32)
    Gf = rng.standard_normal((n, N + 3)).astype(np.float32)
    Hf = rng.standard_normal((n, N + 3)).astype(np.float32)
    if bf16:
        torch = pytest.importorskip("torch")
        bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        Zs, Gs, Hs = bits(Zf), bits(Gf), bits(Hf)
    else:
        Zs, Gs, Hs = Zf, Gf, Hf
    Zw, Gw, Hw = (oracle.widen(a, bf16) for a in (Zs, Gs, Hs))
    cols = [0, 4, N - 1]
    for relu in (False, True):
        got = oracle.update_backward_dw_columns(Gs, Hs, Zs[:, :K], relu, cols, bf16, bf16, block_rows=100)
        dY = Gw[:, cols] * (Hw[:, cols] > 0) if relu else Gw[:, cols]
        assert _rel(got, Zw[:, :K].T @ dY) < 1e-13


def test_relu_derivative_at_zero_is_zero():
    # ReLU'(0) = 0: a pre-activation of exactly zero passes no gradient.
    Z = np.array([[1.0, -1.0]])
    W = np.array([[1.0], [1.0]])
    Hout = oracle.update(Z, W, True)
    assert Hout[0, 0] == 0.0
    dW, dZ = oracle.update_backward(np.array([[1.0]]), Hout, Z, W, True)
    assert np.all(dW == 0.0) and np.all(dZ == 0.0)


# ---------------------------------------------------------------------------
# T2: A_hat 1 = 1 on a regular graph with self loops; the mean of constants
# ---------------------------------------------------------------------------

def test_normalised_adjacency_preserves_constants_on_regular_graph():
    A = circulant(60, 3)  # 6-regular, degree of A + I is 7 everywhere
    part, _ = partition_from_dense(A, np.arange(30))
    assert part.n_halo == 6
    H = np.full((part.n_total, 4), 2.5)
    Z = oracle.aggregate(part, H, 4, "gcn")
    np.testing.assert_allclose(Z, 2.5, rtol=4e-16 * 8, atol=0)
    Zs = oracle.aggregate(part, H, 4, "sage")
    np.testing.assert_allclose(Zs, 2.5, rtol=4e-16 * 8, atol=0)


# ---------------------------------------------------------------------------
# T3: P = P_in + P_out (DIGEST matrix form of the stale-representation layer)
# ---------------------------------------------------------------------------

def test_in_plus_out_propagation_equals_full():
    A, local, part, cols = _tiny(11, N=50, nL=25, p=0.12)
    rng = np.random.default_rng(11)
    f = 4
    H = rng.standard_normal((part.n_total, f))
    w = oracle.gcn_dinv(part)

    def restricted(keep):
        rp, ci = [0], []
        for v in range(part.n_local):
            row = part.colidx[part.rowptr[v]:part.rowptr[v + 1]]
            ci.extend(int(c) for c in row if keep(int(c)))
            rp.append(len(ci))
        return synth.Partition(np.array(rp, np.int32), np.array(ci, np.int32), part.n_local, part.n_halo, part.deg,
                               part.local_ids, part.halo_ids, part.n_table)

    p_in = restricted(lambda c: c < part.n_local)
    p_out = restricted(lambda c: c >= part.n_local)
    Z = oracle.aggregate(part, H, f, "gcn", weights=w)
    Zi = oracle.aggregate(p_in, H, f, "gcn", weights=w)
    Zo = oracle.aggregate(p_out, H, f, "gcn", weights=w)
    assert np.abs(Zo).max() > 0.1  # the halo really contributes
    assert _rel(Zi + Zo, Z) < 1e-14


# ---------------------------------------------------------------------------
# T4: central finite differences of L = <R, layer(H, W)>
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("agg", ["gcn", "sage"])
def test_layer_gradients_match_finite_differences(agg):
    A, local, part, cols = _tiny(21, N=20, nL=12, p=0.25)
    rng = np.random.default_rng(21)
    f, fo = 5, 4
    K = f if agg == "gcn" else 2 * f
    H = rng.standard_normal((part.n_total, f))
    W = rng.standard_normal((K, fo))
    R = rng.standard_normal((part.n_local, fo))
    Z, Hout = oracle.layer_forward(part, H, W, agg, relu=True)
    pre = oracle.update(Z, W, relu=False)
    assert np.min(np.abs(pre)) > 1e-4  # away from ReLU kinks

    def loss(Hx, Wx):
        return float(np.sum(R * oracle.layer_forward(part, Hx, Wx, agg, relu=True)[1]))

    T = oracle.transpose(part)
    dW, _, dH = oracle.layer_backward(part, T, R, Hout, Z, W, agg, relu=True)
    eps = 1e-6
    num_dW = np.zeros_like(W)
    for idx in np.ndindex(*W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += eps
        Wm[idx] -= eps
        num_dW[idx] = (loss(H, Wp) - loss(H, Wm)) / (2 * eps)
    num_dH = np.zeros_like(H)
    for idx in np.ndindex(*H.shape):
        Hp, Hm = H.copy(), H.copy()
        Hp[idx] += eps
        Hm[idx] -= eps
        num_dH[idx] = (loss(Hp, W) - loss(Hm, W)) / (2 * eps)
    assert _rel(dW, num_dW) < 1e-6
    assert _rel(dH, num_dH) < 1e-6
    assert np.abs(dH[part.n_local:]).max() > 0  # halo rows receive gradient (Sylvie's J)


def test_softmax_ce_gradient_matches_finite_differences():
    rng = np.random.default_rng(5)
    n, C = 6, 4
    x = rng.standard_normal((n, C))
    y = rng.integers(0, C, size=n).astype(np.int32)
    loss, G = oracle.softmax_ce(x, y)
    p = np.exp(x - x.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert abs(loss - float(np.mean(-np.log(p[np.arange(n), y])))) < 1e-13
    np.testing.assert_allclose(G.sum(axis=1), 0.0, atol=1e-15)
    eps = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        num[idx] = (oracle.softmax_ce(xp, y)[0] - oracle.softmax_ce(xm, y)[0]) / (2 * eps)
    assert _rel(G, num) < 1e-7


# ---------------------------------------------------------------------------
# T5: special cases - no halo is the textbook full-graph GCN; partitions with
# fresh tables stitch into the full-graph result (forward and backward)
# ---------------------------------------------------------------------------

def test_degree_rule_without_deg_matches_true_degree_when_visible():
    # Halo vertices whose neighbours all lie in the block: counting the block's
    # columns (plus the self loop) recovers their true degree of A + I.
    rng = np.random.default_rng(9)
    N, nL = 30, 20
    A = np.zeros((N, N), dtype=np.int64)
    for v in range(nL):
        for u in range(v + 1, N):
            if rng.random() < 0.2:
                A[v, u] = A[u, v] = 1
    part_deg, _ = partition_from_dense(A, np.arange(nL), pass_deg=True)
    part_null, _ = partition_from_dense(A, np.arange(nL), pass_deg=False)
    assert part_null.deg is None
    np.testing.assert_array_equal(oracle.gcn_dinv(part_null), oracle.gcn_dinv(part_deg))


def test_partitions_with_fresh_tables_stitch_to_full_graph():
    N, f, hid, C = 45, 6, 5, 3
    A = random_sym_adjacency(N, 0.12, 33)
    rng = np.random.default_rng(33)
    X = rng.standard_normal((N, f))
    W0 = rng.standard_normal((f, hid))
    W1 = rng.standard_normal((hid, C))
    full, _ = partition_from_dense(A, np.arange(N))
    assert full.n_halo == 0
    # full graph, two layers: textbook GCN
    Ad = dense_gcn_block(A, np.arange(N), np.arange(N))
    H1 = np.maximum(Ad @ X @ W0, 0)
    H2 = Ad @ H1 @ W1
    _, h1 = oracle.layer_forward(full, X, W0, "gcn", relu=True)
    _, h2 = oracle.layer_forward(full, h1, W1, "gcn", relu=False)
    assert _rel(h2, H2) < 1e-12
    # three partitions exchanging through tables
    blocks = [np.arange(0, 15), np.arange(15, 30), np.arange(30, 45)]
    parts = [partition_from_dense(A, b)[0] for b in blocks]
    table1 = np.zeros((N, hid))
    outs0 = []
    for p in parts:
        H = np.zeros((p.n_total, f))
        H[:p.n_local] = X[p.local_ids]
        oracle.halo_pull(X, p.halo_ids, H, p.n_local, f)
        Z, Ho = oracle.layer_forward(p, H, W0, "gcn", relu=True)
        outs0.append((H, Z, Ho))
        assert oracle.halo_push(Ho, p.n_local, hid, p.local_ids, table1) == oracle.OK
    outs1 = []
    for p, (_, _, Ho) in zip(parts, outs0):
        H = np.zeros((p.n_total, hid))
        H[:p.n_local] = Ho
        oracle.halo_pull(table1, p.halo_ids, H, p.n_local, hid)
        Z, Ho2 = oracle.layer_forward(p, H, W1, "gcn", relu=False)
        outs1.append((H, Z, Ho2))
    stitched = np.concatenate([o[2] for o in outs1])
    assert _rel(stitched, H2) < 1e-12
    # backward with halo-gradient return: gradients of H1 from every partition,
    # summed at the owners, equal the full-graph gradient
    R = rng.standard_normal((N, C))
    Tfull = oracle.transpose(full)
    _, _, dH1_full = oracle.layer_backward(full, Tfull, R, h2, oracle.aggregate(full, h1, hid, "gcn"), W1, "gcn",
                                           relu=False)
    dH1 = np.zeros((N, hid))
    dW1 = np.zeros_like(W1)
    for p, (H, Z, Ho2) in zip(parts, outs1):
        dW, _, dH = oracle.layer_backward(p, oracle.transpose(p), R[p.local_ids], Ho2, Z, W1, "gcn", relu=False)
        dW1 += dW
        dH1[p.local_ids] += dH[:p.n_local]
        dH1[p.halo_ids] += dH[p.n_local:]
    assert _rel(dH1, dH1_full) < 1e-12
    assert _rel(dW1, (Ad @ H1).T @ R) < 1e-12


# ---------------------------------------------------------------------------
# T6: bit-exact index work - transpose, pull, push
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_transpose_matches_scipy_and_is_an_involution(seed):
    p = synth.rmat_block_partition(10, 600, 300, 6000.0, seed=seed)
    rT, cT, pT = oracle.transpose(p)
    M = sp.csr_matrix((np.arange(p.nnz, dtype=np.int64) + 1, p.colidx, p.rowptr), shape=(p.n_local, p.n_total))
    Mt = M.T.tocsr()
    Mt.sort_indices()
    np.testing.assert_array_equal(rT, Mt.indptr)
    np.testing.assert_array_equal(cT, Mt.indices)
    np.testing.assert_array_equal(pT, Mt.data - 1)
    # transposing the transpose gives the block back
    back = synth.Partition(rT, cT, p.n_total, 0, None, np.zeros(0, np.int64), np.zeros(0, np.int64), 0)
    rTT, cTT, _ = oracle.transpose(back)
    np.testing.assert_array_equal(rTT[:p.n_local + 1], p.rowptr)
    assert np.all(rTT[p.n_local:] == p.nnz)
    np.testing.assert_array_equal(cTT, p.colidx)


def test_pull_is_a_row_gather():
    rng = np.random.default_rng(3)
    table = rng.standard_normal((50, 8)).astype(np.float32)
    ids = rng.integers(0, 50, size=12)
    H = np.zeros((20, 8), np.float32)
    assert oracle.halo_pull(table, ids, H, 8, 6) == oracle.OK
    np.testing.assert_array_equal(H[8:, :6], table[ids, :6])
    assert np.all(H[:8] == 0) and np.all(H[8:, 6:] == 0)
    bad = ids.copy()
    bad[3] = 50
    H2 = np.zeros((20, 8), np.float32)
    assert oracle.halo_pull(table, bad, H2, 8, 6) == oracle.ERR_INDEX
    assert np.all(H2[8 + 3] == 0)


def test_push_is_a_row_scatter_and_rejects_repeated_ids():
    rng = np.random.default_rng(4)
    H = rng.integers(0, 60000, size=(10, 8)).astype(np.uint16)  # bf16 bit patterns: copied as bytes
    ids = rng.permutation(40)[:10]
    table = np.zeros((40, 8), np.uint16)
    assert oracle.halo_push(H, 10, 8, ids, table) == oracle.OK
    ref = np.zeros((40, 8), np.uint16)
    ref[ids] = H
    np.testing.assert_array_equal(table, ref)
    dup = ids.copy()
    dup[7] = dup[2]
    table2 = np.zeros((40, 8), np.uint16)
    assert oracle.halo_push(H, 10, 8, dup, table2) == oracle.ERR_INDEX
    assert np.all(table2[dup[2]] == 0)
    ok_rows = [v for v in range(10) if v not in (2, 7)]
    np.testing.assert_array_equal(table2[dup[ok_rows]], H[ok_rows])


# ---------------------------------------------------------------------------
# T7: the Fig. 3 narrative of the Sylvie page (structure only)
# ---------------------------------------------------------------------------

def test_fig3_toy_halo_sets():
    g = json.load(open(os.path.join(HERE, "golden", "fig3_toy.json")))
    N = g["n_nodes"]
    A = np.zeros((N, N), dtype=np.int64)
    for u, v in g["edges"]:
        A[u, v] = A[v, u] = 1
    parts = {k: partition_from_dense(A, np.array(v))[0] for k, v in g["partitions"].items()}
    for k, p in parts.items():
        assert p.halo_ids.tolist() == g["expected_halo"][k]
    needed = sorted({int(u) for k, p in parts.items() if k != "gpu1" for u in p.halo_ids
                     if u in g["partitions"]["gpu1"]})
    assert needed == g["gpu1_needed_by_others"]
    # one-hot features: node 4's aggregate has support exactly on what it needs
    p = parts["gpu1"]
    X = np.eye(N)
    H = np.zeros((p.n_total, N))
    H[:p.n_local] = X[p.local_ids]
    oracle.halo_pull(X, p.halo_ids, H, p.n_local, N)
    Z = oracle.aggregate(p, H, N, "gcn")
    v4 = g["partitions"]["gpu1"].index(4)
    assert np.nonzero(Z[v4])[0].tolist() == g["node4_aggregates_from"]


# ---------------------------------------------------------------------------
# precision helpers against torch's CPU casts (an independent implementation)
# ---------------------------------------------------------------------------

def test_bf16_helpers_match_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(5000) * 10 ** rng.uniform(-5, 5, 5000),
                        [0.0, -0.0, 1.0, 65504.0, 1e-40, -3.0e38]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), ref.astype(np.float64))
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.widen(bits, True), ref.astype(np.float64))
