"""Pins of the oracle's epoch (``oracle.epoch``): the composition of the layer
functions into one training epoch, and its precision modes.

The references here do not share the oracle's code:

* the textbook full-graph model written with dense torch float64 matrices and
  torch autograd (CAGNET page, GNN section: H = sigma(A^T H W) with the
  normalised adjacency, ReLU on all layers but the last, mean softmax
  cross-entropy over the training rows); storage rounding is inserted as an
  autograd node that rounds its value (activations) and / or its incoming
  gradient (activation gradients, and dY as an operand of the bf16 products)
  through torch's own bf16 cast;
* partitions with fresh tables, which must stitch into that full-graph model
  (DIGEST page, matrix form P = P_in + P_out with exact representations);
* central finite differences of the epoch's own loss, with the stale tables
  held constant, for every weight and for every halo row (Sylvie page,
  backward propagation: the halo gradients J).

A mistake in the composition - ReLU on the last layer, a wrong table index, G
fed from the halo rows, a missing or misplaced rounding point - fails one of
them.  The last tests check the ReLU-flip bounds that the GPU epoch tests use
(``tests/_flip.py``) against flips planted in the oracle.
"""
import numpy as np
import pytest

import oracle
from tests._flip import ambiguous_masks, forward_difference_bounds, relu_flip_bounds
from tests._problems import dense_gcn_block, dense_mean_block, partition_from_dense, random_sym_adjacency

torch = pytest.importorskip("torch")

WIDTHS = [6, 7, 5, 4]


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


def _rb_t(x):
    return x.to(torch.float32).to(torch.bfloat16).to(torch.float64)


class _Store(torch.autograd.Function):
    """Identity that stores its value (forward) and its gradient (backward) in
    bf16 when asked: the rounding points of a bf16 path."""

    @staticmethod
    def forward(ctx, x, act, grad):
        ctx.grad = grad
        return _rb_t(x) if act else x.clone()

    @staticmethod
    def backward(ctx, g):
        return (_rb_t(g) if ctx.grad else g), None, None


def textbook(A, X, Ws, y, agg, act=False, grad=False):
    """Full-graph model with dense operators and autograd (float64)."""
    N = A.shape[0]
    idx = np.arange(N)
    op = torch.from_numpy(dense_gcn_block(A, idx, idx) if agg == "gcn" else dense_mean_block(A, idx, idx))
    Wt = [torch.tensor(w, dtype=torch.float64, requires_grad=True) for w in Ws]
    H = torch.from_numpy(np.asarray(X, dtype=np.float64))
    L = len(Ws)
    pre, Zs, Hs = [], [], [H]
    for l in range(L):
        Zp = op @ H if agg == "gcn" else torch.cat([H, op @ H], dim=1)
        Z = _Store.apply(Zp, act, grad)
        Y = _Store.apply(Z @ Wt[l], False, act)  # with bf16 activations dY enters the products as bf16
        Hp = torch.relu(Y) if l < L - 1 else Y
        Hp.retain_grad()
        H = _Store.apply(Hp, act, grad)
        pre.append(Hp)
        Zs.append(Z)
        Hs.append(H)
    loss = torch.nn.functional.cross_entropy(H, torch.from_numpy(np.asarray(y, dtype=np.int64)))
    loss.backward()
    return dict(logits=H.detach().numpy(), loss=loss.item(), dW=[w.grad.numpy() for w in Wt],
                Z=[z.detach().numpy() for z in Zs], H=[h.detach().numpy() for h in Hs],
                dH=[None] + [pre[l - 1].grad.numpy() for l in range(1, L)], G=[p.grad.numpy() for p in pre])


def _problem(seed, N=40, p=0.15, agg="gcn", bf16=False):
    A = random_sym_adjacency(N, p, seed)
    rng = np.random.default_rng(seed)
    K = [(2 if agg == "sage" else 1) * w for w in WIDTHS[:-1]]
    X = rng.standard_normal((N, WIDTHS[0]))
    Ws = [rng.uniform(-1, 1, (K[l], WIDTHS[l + 1])) * np.sqrt(6 / (K[l] + WIDTHS[l + 1])) for l in range(3)]
    y = rng.integers(0, WIDTHS[-1], N).astype(np.int32)
    if bf16:
        X = oracle.round_bf16(X)
        Ws = [oracle.round_bf16(w) for w in Ws]
    return A, X, Ws, y


MODES = [(False, False), (True, False), (True, True)]  # (bf16 activations, bf16 activation gradients)


@pytest.mark.parametrize("agg", ["gcn", "sage"])
@pytest.mark.parametrize("act,grad", MODES)
def test_whole_graph_epoch_matches_textbook_autograd(agg, act, grad):
    A, X, Ws, y = _problem(1, agg=agg, bf16=act)
    N = A.shape[0]
    full, _ = partition_from_dense(A, np.arange(N))
    assert full.n_halo == 0
    tables = [X] + [np.zeros((N, f)) for f in WIDTHS[1:-1]]
    ref = oracle.epoch(full, tables, Ws, y, agg, bf16=act, grad_bf16=grad)
    tb = textbook(A, X, Ws, y, agg, act, grad)
    L = len(Ws)
    assert _rel(ref["Hout"][-1], tb["logits"]) < 1e-12
    assert abs(ref["loss"] - tb["loss"]) < 1e-12 * abs(tb["loss"])
    for l in range(L):
        assert _rel(ref["Z"][l], tb["Z"][l]) < 1e-12, f"Z[{l}]"
        assert _rel(ref["dW"][l], tb["dW"][l]) < 1e-11, f"dW[{l}]"
        assert _rel(ref["G"][l], tb["G"][l]) < 1e-11, f"G[{l}]"
    for l in range(1, L):
        assert _rel(ref["dH"][l], tb["dH"][l]) < 1e-11, f"dH[{l}]"
        assert _rel(ref["tables"][l], tb["H"][l]) < 1e-12, f"pushed table {l}"
    # each rounding mode is observable: without it the reference moves by far more than the comparison allows
    if act or grad:
        plain = textbook(A, X, Ws, y, agg, act=act and not grad, grad=False) if grad else \
            textbook(A, X, Ws, y, agg, act=False, grad=False)
        assert _rel(ref["dW"][0], plain["dW"][0]) > 1e-6


@pytest.mark.parametrize("agg", ["gcn", "sage"])
@pytest.mark.parametrize("act", [False, True])
def test_partitions_with_fresh_tables_stitch_into_whole_graph_epoch(agg, act):
    A, X, Ws, y = _problem(2, N=45, p=0.12, agg=agg, bf16=act)
    N = A.shape[0]
    tb = textbook(A, X, Ws, y, agg, act, False)
    fresh = [tb["H"][l] for l in range(len(WIDTHS) - 1)]  # exact (stored) representations of every layer
    perm = np.random.default_rng(2).permutation(N)
    blocks = [np.sort(b) for b in np.array_split(perm, 3)]
    L = len(Ws)
    loss = 0.0
    dW_top = np.zeros_like(Ws[-1])
    dH_top = np.zeros((N, WIDTHS[L - 1]))
    for b in blocks:
        p, _ = partition_from_dense(A, b)
        assert p.n_halo > 0
        ref = oracle.epoch(p, fresh, Ws, y[p.local_ids], agg, bf16=act)
        share = p.n_local / N
        assert _rel(ref["Hout"][-1], tb["logits"][p.local_ids]) < 1e-12
        for l in range(1, L):
            assert _rel(ref["tables"][l][p.local_ids], tb["H"][l][p.local_ids]) < 1e-12
        loss += share * ref["loss"]
        dW_top += share * ref["dW"][-1]
        dH = share * ref["dH"][-1]
        dH_top[p.local_ids] += dH[:p.n_local]
        dH_top[p.halo_ids] += dH[p.n_local:]  # the halo gradients J, added at their owners
    assert abs(loss - tb["loss"]) < 1e-12 * abs(tb["loss"])
    if act:
        # bf16 products round each partition's dY = G / n_p, which does not
        # scale into the whole graph's G / N: the stitched backward is checked
        # in double only
        return
    assert _rel(dW_top, tb["dW"][-1]) < 1e-11
    assert _rel(dH_top, tb["dH"][-1]) < 1e-11


@pytest.mark.parametrize("agg", ["gcn", "sage"])
def test_epoch_gradients_match_finite_differences_of_its_loss(agg):
    # one partition with stale tables: the loss depends on W and, through the
    # halo rows of layer l, on tables[l]; dW and the halo rows of dH are its
    # exact derivatives (the tables are constants of the epoch)
    N, nL = 30, 18
    A = random_sym_adjacency(N, 0.18, 4)
    part, _ = partition_from_dense(A, np.arange(nL))
    assert part.n_halo >= 5
    rng = np.random.default_rng(4)
    K = [(2 if agg == "sage" else 1) * w for w in WIDTHS[:-1]]
    Ws = [rng.standard_normal((K[l], WIDTHS[l + 1])) * 0.6 for l in range(3)]
    tables = [rng.standard_normal((N, f)) for f in WIDTHS[:-1]]
    y = rng.integers(0, WIDTHS[-1], nL).astype(np.int32)
    ref = oracle.epoch(part, tables, Ws, y, agg)
    for l in range(2):
        assert np.min(np.abs(ref["Z"][l] @ Ws[l])) > 2e-5  # the steps below cross no ReLU kink

    def loss(Wx, tx):
        return oracle.epoch(part, tx, Wx, y, agg)["loss"]

    eps = 1e-6
    for l in range(3):
        num = np.zeros_like(Ws[l])
        for idx in np.ndindex(*Ws[l].shape):
            Wp = [w.copy() for w in Ws]
            Wm = [w.copy() for w in Ws]
            Wp[l][idx] += eps
            Wm[l][idx] -= eps
            num[idx] = (loss(Wp, tables) - loss(Wm, tables)) / (2 * eps)
        assert _rel(ref["dW"][l], num) < 1e-6, f"dW[{l}]"
    for l in (1, 2):
        num = np.zeros((part.n_halo, WIDTHS[l]))
        for i, u in enumerate(part.halo_ids):
            for c in range(WIDTHS[l]):
                tp = [t.copy() for t in tables]
                tm = [t.copy() for t in tables]
                tp[l][u, c] += eps
                tm[l][u, c] -= eps
                num[i, c] = (loss(Ws, tp) - loss(Ws, tm)) / (2 * eps)
        assert np.abs(num).max() > 1e-3
        assert _rel(ref["dH"][l][nL:], num) < 1e-6, f"halo rows of dH[{l}]"


# ---------------------------------------------------------------------------
# the ReLU-flip bounds of the chained GPU comparisons
# ---------------------------------------------------------------------------

def _flip_problem(agg):
    N, nL = 60, 36
    A = random_sym_adjacency(N, 0.1, 5)
    part, _ = partition_from_dense(A, np.arange(nL))
    rng = np.random.default_rng(5)
    K = [(2 if agg == "sage" else 1) * w for w in WIDTHS[:-1]]
    f32 = lambda a: a.astype(np.float32).astype(np.float64)  # inputs an fp32 path holds exactly
    Ws = [f32(rng.standard_normal((K[l], WIDTHS[l + 1])) * 0.5) for l in range(3)]
    tables = [f32(rng.standard_normal((N, f))) for f in WIDTHS[:-1]]
    y = rng.integers(0, WIDTHS[-1], nL).astype(np.int32)
    return part, Ws, tables, y


@pytest.mark.parametrize("agg", ["gcn", "sage"])
def test_flip_bounds_cover_flips_planted_in_the_oracle(agg):
    part, Ws, tables, y = _flip_problem(agg)
    ref = oracle.epoch(part, tables, Ws, y, agg)
    L = len(Ws)
    planted = [(1, 3, 2), (1, 10, 0), (0, 5, 1)]  # (layer, row, column) whose ReLU decision goes the other way
    amb = [np.zeros(ref["Hout"][l].shape, dtype=bool) for l in range(L - 1)] + [None]
    Hmod = [h.copy() for h in ref["Hout"]]
    for l, v, j in planted:
        Hmod[l][v, j] = 0.0 if Hmod[l][v, j] > 0 else 1.0
        amb[l][v, j] = True
    G = ref["G"][L - 1]
    dWf, dHf = [None] * L, [None] * L
    for l in reversed(range(L)):
        dWf[l], _, dHf[l] = oracle.layer_backward(part, ref["T"], G, Hmod[l], ref["Z"][l], Ws[l], agg,
                                                  relu=l < L - 1, want_dh=l > 0)
        if l > 0:
            G = dHf[l][:part.n_local]
    dWb, dHb = relu_flip_bounds(part, ref, Ws, agg, amb)
    moved = 0
    for got, want, b in list(zip(dWf, ref["dW"], dWb)) + list(zip(dHf[1:], ref["dH"][1:], dHb[1:])):
        diff = np.abs(got - want)
        assert np.all(diff <= b * (1 + 1e-9) + 1e-13)
        assert np.all(got[b == 0] == want[b == 0])  # nothing downstream of a flip: the very same sums
        moved += int(np.count_nonzero(diff > 1e-12))
    assert moved > 0
    # the top layer sees no flip; in layer 1 only the flipped columns of dW move
    assert np.all(dWb[L - 1] == 0)
    cols = np.nonzero(dWb[1].any(axis=0))[0].tolist()
    assert cols == [0, 2]


def test_forward_bounds_cover_an_fp32_evaluation():
    # the same epoch evaluated in float32 (numpy, its own summation order) stays
    # within the propagated bounds on the pre-activations
    part, Ws, tables, y = _flip_problem("gcn")
    ref = oracle.epoch(part, tables, Ws, y, "gcn")
    fwd = forward_difference_bounds(part, ref, Ws, "gcn", act_bf16=False)
    import scipy.sparse as sp
    dinv = oracle.gcn_dinv(part).astype(np.float32)
    rows = np.repeat(np.arange(part.n_local), np.diff(part.rowptr))
    vals = dinv[rows] * dinv[part.colidx]
    Ablk = sp.csr_matrix((vals.astype(np.float32), part.colidx, part.rowptr), shape=(part.n_local, part.n_total))
    h_local = tables[0][part.local_ids].astype(np.float32)
    for l in range(len(Ws)):
        H = np.concatenate([h_local, tables[l][part.halo_ids].astype(np.float32)])[:, :WIDTHS[l]]
        Y32 = (Ablk @ H).astype(np.float32) @ Ws[l].astype(np.float32)
        Y, dY = fwd[l]
        assert np.all(np.abs(Y32.astype(np.float64) - Y) <= dY)
        h_local = np.maximum(Y32, 0).astype(np.float32)
    assert all(a is None or a.sum() == 0 for a in ambiguous_masks(fwd))  # nothing near zero on this input


def test_forward_bounds_cover_a_multiply_first_fp32_evaluation():
    # the same, with layers 1 and 2 evaluated as A (H W) in float32
    part, Ws, tables, y = _flip_problem("gcn")
    ref = oracle.epoch(part, tables, Ws, y, "gcn")
    mf = [False, True, True]
    fwd = forward_difference_bounds(part, ref, Ws, "gcn", act_bf16=False, multiply_first=mf)
    import scipy.sparse as sp
    dinv = oracle.gcn_dinv(part).astype(np.float32)
    rows = np.repeat(np.arange(part.n_local), np.diff(part.rowptr))
    vals = dinv[rows] * dinv[part.colidx]
    Ablk = sp.csr_matrix((vals.astype(np.float32), part.colidx, part.rowptr), shape=(part.n_local, part.n_total))
    h_local = tables[0][part.local_ids].astype(np.float32)
    for l in range(len(Ws)):
        H = np.concatenate([h_local, tables[l][part.halo_ids].astype(np.float32)])[:, :WIDTHS[l]]
        W32 = Ws[l].astype(np.float32)
        Y32 = (Ablk @ (H @ W32)).astype(np.float32) if mf[l] else (Ablk @ H).astype(np.float32) @ W32
        Y, dY = fwd[l]
        assert np.all(np.abs(Y32.astype(np.float64) - Y) <= dY)
        h_local = np.maximum(Y32, 0).astype(np.float32)
