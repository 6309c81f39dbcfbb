"""Pins of the oracle's graph-attention (GAT) layer, without its code.

The layer is the textbook single-head GAT (the Sylvie and DIGEST pages name
GAT without printing its formula): scores z_vu = a_dst . T[v] + a_src . T[u]
over the entries of A + I, LeakyReLU (slope 0.2), a softmax over each row, and
the attention-weighted sum of T = H W.  References: a dense masked-softmax
evaluation with numpy, torch autograd on that dense form, special cases with
closed forms (zero attention vectors give the plain neighbour mean; each row of
alpha sums to 1), and central finite differences of the layer.
"""
import numpy as np
import pytest

import oracle
from tests._problems import partition_from_dense, random_sym_adjacency

torch = pytest.importorskip("torch")


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


def _case(seed, N=36, nL=22, p=0.18, f=5, fo=4):
    A = random_sym_adjacency(N, p, seed)
    part, cols = partition_from_dense(A, np.arange(nL))
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((part.n_total, f))
    W = rng.standard_normal((f, fo)) * 0.7
    a_src = rng.standard_normal(fo)
    a_dst = rng.standard_normal(fo)
    mask = (A + np.eye(N, dtype=np.int64))[np.ix_(np.arange(nL), cols)] > 0
    return part, mask, H, W, a_src, a_dst


def _dense(mask, H, W, a_src, a_dst, relu, lib=np):
    """Dense form: Y = softmax_rows(masked LeakyReLU(scores)) (H W)."""
    T = H @ W
    nL = mask.shape[0]
    z = (T[:nL] @ a_dst)[:, None] + (T @ a_src)[None, :]
    if lib is np:
        e = np.where(z > 0, z, 0.2 * z)
        e = np.where(mask, e, -np.inf)
        e = e - e.max(axis=1, keepdims=True)
        alpha = np.exp(e)
        alpha /= alpha.sum(axis=1, keepdims=True)
        Y = alpha @ T
        return alpha, (np.maximum(Y, 0) if relu else Y)
    e = torch.where(z > 0, z, 0.2 * z)
    e = e.masked_fill(~torch.from_numpy(mask), float("-inf"))
    alpha = torch.softmax(e, dim=1)
    Y = alpha @ T
    return alpha, (torch.relu(Y) if relu else Y)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gat_forward_matches_dense_masked_softmax(seed):
    part, mask, H, W, a_src, a_dst = _case(seed)
    fw = oracle.gat_layer_forward(part, H, W, a_src, a_dst, relu=True)
    alpha_d, Hout_d = _dense(mask, H, W, a_src, a_dst, True)
    rows = np.repeat(np.arange(part.n_local), np.diff(part.rowptr))
    assert _rel(fw["alpha"], alpha_d[rows, part.colidx]) < 1e-13
    assert _rel(fw["Hout"], Hout_d) < 1e-13
    # every row's attention sums to one
    np.testing.assert_allclose(np.bincount(rows, weights=fw["alpha"]), 1.0, atol=1e-14)


def test_gat_with_zero_attention_vectors_is_the_neighbour_mean():
    part, mask, H, W, a_src, a_dst = _case(5)
    fw = oracle.gat_layer_forward(part, H, W, np.zeros_like(a_src), np.zeros_like(a_dst), relu=False)
    T = H @ W
    mean = (mask @ T) / mask.sum(axis=1, keepdims=True)
    assert _rel(fw["Hout"], mean) < 1e-13


@pytest.mark.parametrize("relu", [False, True])
def test_gat_backward_matches_dense_autograd(relu):
    part, mask, H, W, a_src, a_dst = _case(3)
    R = np.random.default_rng(9).standard_normal((part.n_local, W.shape[1]))
    fw = oracle.gat_layer_forward(part, H, W, a_src, a_dst, relu=relu)
    bw = oracle.gat_layer_backward(part, fw, H, R, W, a_src, a_dst, relu=relu)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True)
         for k, v in dict(H=H, W=W, a_src=a_src, a_dst=a_dst).items()}
    _, Hout = _dense(mask, t["H"], t["W"], t["a_src"], t["a_dst"], relu, lib=torch)
    (Hout * torch.from_numpy(R)).sum().backward()
    assert _rel(bw["dW"], t["W"].grad.numpy()) < 1e-12
    assert _rel(bw["da_src"], t["a_src"].grad.numpy()) < 1e-12
    assert _rel(bw["da_dst"], t["a_dst"].grad.numpy()) < 1e-12
    assert _rel(bw["dH"], t["H"].grad.numpy()) < 1e-12
    assert np.abs(bw["dH"][part.n_local:]).max() > 0  # halo rows receive gradient (J)


def test_gat_gradients_match_finite_differences():
    part, mask, H, W, a_src, a_dst = _case(4, N=20, nL=12, p=0.3, f=3, fo=3)
    R = np.random.default_rng(4).standard_normal((part.n_local, 3))

    def loss(Hx, Wx, asx, adx):
        return float(np.sum(R * oracle.gat_layer_forward(part, Hx, Wx, asx, adx, relu=True)["Hout"]))

    fw = oracle.gat_layer_forward(part, H, W, a_src, a_dst, relu=True)
    pre = oracle.gat_attend(part, fw["T"], fw["s_src"], fw["s_dst"])[1]
    assert np.min(np.abs(pre)) > 1e-4
    bw = oracle.gat_layer_backward(part, fw, H, R, W, a_src, a_dst, relu=True)
    eps = 1e-6
    args = [H, W, a_src, a_dst]
    for i, name in enumerate(["dH", "dW", "da_src", "da_dst"]):
        x = args[i]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = list(args), list(args)
            ap[i], am[i] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * eps)
        assert _rel(bw[name], num) < 1e-6, name


def test_gat_epoch_gradients_match_finite_differences_of_its_loss():
    # a 3-layer GAT on a partition with stale halo tables: dW, da_src, da_dst of
    # every layer and the halo rows of every dH are the derivatives of the loss
    N, nL = 26, 16
    A = random_sym_adjacency(N, 0.2, 8)
    part, _ = partition_from_dense(A, np.arange(nL))
    rng = np.random.default_rng(8)
    widths = [4, 5, 4, 3]
    Ws = [rng.standard_normal((widths[l], widths[l + 1])) * 0.7 for l in range(3)]
    a_s = [rng.standard_normal(widths[l + 1]) * 0.5 for l in range(3)]
    a_d = [rng.standard_normal(widths[l + 1]) * 0.5 for l in range(3)]
    tables = [rng.standard_normal((N, f)) for f in widths[:-1]]
    y = rng.integers(0, widths[-1], nL).astype(np.int32)
    ref = oracle.gat_epoch(part, tables, Ws, a_s, a_d, y)
    for l in range(2):
        pre = oracle.gat_attend(part, ref["fwd"][l]["T"], ref["fwd"][l]["s_src"], ref["fwd"][l]["s_dst"])[1]
        assert np.min(np.abs(pre)) > 2e-5

    def loss(Wx, asx, adx, tx):
        return oracle.gat_epoch(part, tx, Wx, asx, adx, y)["loss"]

    eps = 1e-6
    for name, params, key in (("W", Ws, "dW"), ("a_src", a_s, "da_src"), ("a_dst", a_d, "da_dst")):
        for l in range(3):
            num = np.zeros_like(params[l])
            for idx in np.ndindex(*params[l].shape):
                pp = [p.copy() for p in params]
                pm = [p.copy() for p in params]
                pp[l][idx] += eps
                pm[l][idx] -= eps
                args_p = {"W": Ws, "a_src": a_s, "a_dst": a_d}
                args_m = dict(args_p)
                args_p[name], args_m[name] = pp, pm
                num[idx] = (loss(args_p["W"], args_p["a_src"], args_p["a_dst"], tables)
                            - loss(args_m["W"], args_m["a_src"], args_m["a_dst"], tables)) / (2 * eps)
            assert _rel(ref[key][l], num) < 1e-6, (name, l)
    for l in (1, 2):
        num = np.zeros((part.n_halo, widths[l]))
        for i, u in enumerate(part.halo_ids):
            for c in range(widths[l]):
                tp = [t.copy() for t in tables]
                tm = [t.copy() for t in tables]
                tp[l][u, c] += eps
                tm[l][u, c] -= eps
                num[i, c] = (loss(Ws, a_s, a_d, tp) - loss(Ws, a_s, a_d, tm)) / (2 * eps)
        assert _rel(ref["dH"][l][nL:], num) < 1e-6, l
