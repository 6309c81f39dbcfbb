"""Parity of the graph-attention layer (gnn_gat_forward / gnn_gat_backward)
with the oracle's textbook single-head GAT.

The attention is compared per row as a multiset (the library keeps each row's
entries in its own order), everything else elementwise: 1e-4 (fp32) or 2e-2
(bf16 activations, fp32 or bf16 gradients).  The forward runs on N(0, 1)
features and Glorot weights, with and without the ReLU.

The backward is compared on inputs whose products are exact in fp32: features,
weights and attention vectors are small integers times powers of two, so
T = H W, the bf16 rounding of T and the scores are identical on both sides and
every LeakyReLU decision (z > 0) is the same.  With general inputs the two
sides' T can round to neighbouring bf16 values (an fp32 against an fp64 sum
near a rounding boundary); that moves the scores of every entry of the row, and
the softmax gradient amplifies it past the tolerance in a few elements of the
hub rows, which is a decision like a ReLU flip rather than an arithmetic error.
The backward is run without the ReLU, so both sides also take identical mask
decisions.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.configs import TINY, WORKLOADS
from sparse_aggregation_dense_gb300 import gnn, ld_for, padded
from tests._gpu import TOL, assert_ok, close, gen_matrix, maybe_round, to_device, to_host, torch_dtype, widen

pytestmark = pytest.mark.gpu

_cache = {}


def _graph(name, size):
    key = (name, size)
    if key not in _cache:
        part = (TINY if size == "tiny" else WORKLOADS)[name].make(0)
        g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(),
                             part.n_local, part.n_halo, None, "gat")
        _cache[key] = (part, g)
    return _cache[key]


def _attention_by_row(part, alpha):
    """alpha (per entry, any order within each row) sorted within each row."""
    rows = np.repeat(np.arange(part.n_local), np.diff(part.rowptr))
    order = np.lexsort((alpha, rows))
    return alpha[order]


def _dyadic(rows, f, dt, rng, step, kmax):
    """Host matrix (storage form, rows x ld) of k * step with k uniform in [-kmax, kmax]."""
    ld = ld_for(f, torch_dtype(dt))
    x = np.zeros((rows, ld), dtype=np.float32)
    x[:, :f] = rng.integers(-kmax, kmax + 1, (rows, f)) * np.float32(step)
    return (x.view(np.uint32) >> 16).astype(np.uint16) if dt == "bf16" else x


def _exact_inputs(part, f_in, f_out, dt, seed):
    """H = k/4 (|k| <= 4), W = k/32 (|k| <= 8), a = k/16 (|k| <= 4): every product and sum of
    T = H W (f_in <= 256) and of the scores (f_out <= 256) is a multiple of 2^-7 or 2^-11 below
    2^24 units, so exact in fp32 in any order."""
    rng = np.random.default_rng(1000 + seed)
    H_h = _dyadic(part.n_total, f_in, dt, rng, 0.25, 4)
    W = (rng.integers(-8, 9, (f_in, f_out)) / 32.0).astype(np.float32)
    a_src = (rng.integers(-4, 5, f_out) / 16.0).astype(np.float32)
    a_dst = (rng.integers(-4, 5, f_out) / 16.0).astype(np.float32)
    return H_h, W, a_src, a_dst


def _inputs(part, f_in, f_out, dt, seed):
    H_h = gen_matrix(part.n_total, f_in, dt, seed, 1)
    W = synth.glorot(f_in, f_out, seed, 2)
    rng = np.random.default_rng(seed)
    a_src = (rng.standard_normal(f_out) * 0.3).astype(np.float32)
    a_dst = (rng.standard_normal(f_out) * 0.3).astype(np.float32)
    return H_h, W, a_src, a_dst


PRECISIONS = [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")]
GRAPHS = [(n, "tiny") for n in ["er5k", "rmat131k", "powerlaw233k", "sage2m", "rmat16m"]] + [("rmat131k", "full")]


@pytest.mark.parametrize("dt,gd", PRECISIONS)
@pytest.mark.parametrize("graph", GRAPHS, ids=lambda c: f"{c[0]}-{c[1]}")
@pytest.mark.parametrize("f_in,f_out", [(64, 64), (100, 47), (256, 172)])
def test_gat_layer(graph, dt, gd, f_in, f_out):
    part, g = _graph(*graph)
    tdt, gdt = torch_dtype(dt), torch_dtype(gd)
    nL, nT = part.n_local, part.n_total
    H_h, W, a_src, a_dst = _inputs(part, f_in, f_out, dt, 5)
    H = to_device(H_h, dt, f_in)
    Wd = torch.from_numpy(W).cuda()
    asd, add = torch.from_numpy(a_src).cuda(), torch.from_numpy(a_dst).cuda()
    T = padded(nT, f_out, tdt, "cuda")
    scores = torch.empty(nT + nL, dtype=torch.float32, device="cuda")
    alpha = torch.empty(part.nnz, dtype=torch.float32, device="cuda")
    tol = TOL[dt]
    Wr = maybe_round(W.astype(np.float64), dt)
    Hw = widen(H_h, dt, f_in)
    for relu in (True, False):
        Hout = padded(nL, f_out, tdt, "cuda")
        gnn.gat_forward(g, H, Wd, asd, add, relu, T, scores, alpha, Hout)
        assert_ok(g)
        ref = oracle.gat_layer_forward(part, Hw, Wr, a_src, a_dst, relu, bf16=dt == "bf16")
        close(to_host(T), ref["T"], tol, "T = H W")
        sc = scores.cpu().numpy().astype(np.float64)
        close(sc[:nT], ref["s_src"], tol, "s_src")
        close(sc[nT:], ref["s_dst"], tol, "s_dst")
        a = alpha.cpu().numpy()
        assert np.all(np.signbit(a)[np.cumsum(np.diff(part.rowptr))[np.diff(part.rowptr) > 0] - 1])  # row ends
        a = np.abs(a).astype(np.float64)
        close(_attention_by_row(part, a), _attention_by_row(part, ref["alpha"]), tol, "alpha (per row)")
        close(to_host(Hout), ref["Hout"], tol, f"H_out (relu={relu})")
    # backward on exact-product inputs (no ReLU: both sides use the same dY)
    H_h, W, a_src, a_dst = _exact_inputs(part, f_in, f_out, dt, 5)
    H = to_device(H_h, dt, f_in)
    Wd = torch.from_numpy(W).cuda()
    asd, add = torch.from_numpy(a_src).cuda(), torch.from_numpy(a_dst).cuda()
    Hw = widen(H_h, dt, f_in)
    Wr = W.astype(np.float64)
    Hout = padded(nL, f_out, tdt, "cuda")
    gnn.gat_forward(g, H, Wd, asd, add, False, T, scores, alpha, Hout)
    assert_ok(g)
    ref = oracle.gat_layer_forward(part, Hw, Wr, a_src, a_dst, False, bf16=dt == "bf16")
    assert np.array_equal(to_host(T), ref["T"]), "T = H W is exact on these inputs"
    sc = scores.cpu().numpy().astype(np.float64)
    assert np.array_equal(sc[:nT], ref["s_src"]) and np.array_equal(sc[nT:], ref["s_dst"]), "exact scores"
    close(to_host(Hout), ref["Hout"], tol, "H_out (exact-product inputs)")
    G_h = gen_matrix(nL, f_out, gd, 5, 3)
    dW = torch.zeros((f_in, f_out), dtype=torch.float32, device="cuda")
    da_s = torch.zeros(f_out, dtype=torch.float32, device="cuda")
    da_d = torch.zeros(f_out, dtype=torch.float32, device="cuda")
    dT = padded(nT, f_out, gdt, "cuda")
    dH = padded(nT, f_in, gdt, "cuda")
    gnn.gat_backward(g, to_device(G_h, gd, f_out), Hout, H, Wd, asd, add, False, T, scores, alpha, dW, da_s, da_d, dT,
                     dH)
    assert_ok(g)
    bw = oracle.gat_layer_backward(part, ref, Hw, widen(G_h, gd, f_out), Wr, a_src, a_dst, relu=False,
                                   bf16=dt == "bf16", grad_bf16=gd == "bf16")
    close(dW.cpu().numpy(), bw["dW"], tol, "dW")
    close(da_s.cpu().numpy(), bw["da_src"], tol, "da_src")
    close(da_d.cpu().numpy(), bw["da_dst"], tol, "da_dst")
    close(to_host(dT), bw["dT"], tol, "dT")
    close(to_host(dH), bw["dH"], tol, "dH (local and halo rows)")


def test_gat_graph_rejects_the_gcn_calls_and_back():
    part, g = _graph("er5k", "tiny")
    H = padded(part.n_total, 8, torch.float32, "cuda")
    Z = padded(part.n_local, 8, torch.float32, "cuda")
    Ho = padded(part.n_local, 4, torch.float32, "cuda")
    with pytest.raises(gnn.GnnError):
        gnn.layer_forward(g, H, torch.zeros((8, 4), device="cuda"), True, Z, Ho)


@pytest.mark.parametrize("hidden_relu", [False, True])
@pytest.mark.parametrize("name,gd", [("er5k", "f32"), ("rmat131k", "f32"), ("rmat16m", "f32"), ("rmat16m", "bf16")])
def test_gat_epoch_matches_oracle(name, gd, hidden_relu):
    from sparse_aggregation_dense_gb300 import GatModel

    w = TINY[name]
    part = w.make(0)
    dt = w.dtype
    widths = [w.widths[0], 32, 24, w.widths[-1]]
    m = GatModel(part, widths, torch_dtype(dt), "cuda", grad_dtype=torch_dtype(gd), hidden_relu=hidden_relu)
    rng = np.random.default_rng(3)
    tables_h = []
    for l in range(3):
        t = gen_matrix(part.n_table, widths[l], dt, 0, 700 + l)
        tables_h.append(t)
        m.tables[l] = to_device(t, dt, widths[l])
    m.H[0][:part.n_local] = m.tables[0][torch.from_numpy(part.local_ids).cuda()]
    Ws = [synth.glorot(widths[l], widths[l + 1], 0, 710 + l) for l in range(3)]
    a_s = [(rng.standard_normal(widths[l + 1]) * 0.3).astype(np.float32) for l in range(3)]
    a_d = [(rng.standard_normal(widths[l + 1]) * 0.3).astype(np.float32) for l in range(3)]
    for l in range(3):
        m.W[l].copy_(torch.from_numpy(Ws[l]))
        m.a_src[l].copy_(torch.from_numpy(a_s[l]))
        m.a_dst[l].copy_(torch.from_numpy(a_d[l]))
    y = synth.labels(part.n_local, widths[-1], 0, ids=part.local_ids)
    m.labels.copy_(torch.from_numpy(y))
    m.step()
    m.check_errors()
    ref = oracle.gat_epoch(part, [widen(t, dt, f) for t, f in zip(tables_h, widths)],
                           [maybe_round(x.astype(np.float64), dt) for x in Ws], a_s, a_d, y, bf16=dt == "bf16",
                           grad_bf16=gd == "bf16", hidden_relu=hidden_relu)
    tol = TOL[dt]
    close(to_host(m.out_last), ref["Hout"][-1], tol, "logits")
    assert abs(float(m.loss.item()) - ref["loss"]) <= tol * abs(ref["loss"])
    for l in range(1, 3):
        pushed = to_host(m.tables[l].index_select(0, torch.from_numpy(part.local_ids).cuda()))
        close(pushed, ref["Hout"][l - 1], tol, f"pushed table {l}")
    # Without hidden ReLUs every gradient is compared elementwise.  With them, a
    # hidden pre-activation within rounding of zero may take the other branch on
    # the two sides, which moves the gradients below it; the top layer's
    # gradients involve no such decision and stay elementwise.
    layers = range(3) if not hidden_relu else [2]
    for l in layers:
        close(m.dW[l].cpu().numpy(), ref["dW"][l], tol, f"dW[{l}]")
        close(m.da_src[l].cpu().numpy(), ref["da_src"][l], tol, f"da_src[{l}]")
        close(m.da_dst[l].cpu().numpy(), ref["da_dst"][l], tol, f"da_dst[{l}]")
    for l in [l for l in layers if l > 0]:
        close(to_host(m.dH[l]), ref["dH"][l], tol, f"dH[{l}] (local and halo rows)")
