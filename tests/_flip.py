"""Chained-layer parity: where a ReLU decision can legitimately differ.

The backward of a ReLU layer masks its gradient with 1[H_out > 0].  The GPU
takes that decision on its own fp32 pre-activation Y = Z W, the oracle on its
double one; both are correct to within rounding, so a pre-activation closer to
zero than the two sides can differ may take the other branch, and the
gradients downstream of it move by a bounded amount.

This module bounds that effect elementwise, from the oracle's side only:

* ``forward_difference_bounds`` propagates, layer by layer, a worst-case bound
  on |Y_gpu - Y| from the fp32 accumulation error of every sum (a standard
  n-term bound, Higham's gamma_n, with a safety factor) and the storage
  rounding of activations; a bf16 rounding absorbs a difference entirely unless
  a rounding midpoint lies inside it.  A pre-activation is *ambiguous* when
  |Y| is within that bound of zero.
* ``relu_flip_bounds`` pushes the largest change an ambiguous decision can make
  (the whole gradient entry |G|) through the backward: dW, dZ and the
  transposed aggregation are linear, all aggregation weights are nonnegative,
  so the same operators applied to absolute values bound the change exactly to
  first order.

Outputs that no ambiguous decision reaches get a bound of exactly zero and are
checked strictly elementwise; the others are allowed the tolerance plus their
bound.  Nothing here comes from the GPU: the bounds are functions of the
oracle's own intermediates.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

import oracle

U32 = 2.0 ** -24  # unit roundoff of fp32
SAFETY = 4.0      # room for fused / truncating accumulators and the fp32 weights


def forward_difference_bounds(part, ref: dict, Ws: Sequence[np.ndarray], agg: str, act_bf16: bool,
                              multiply_first: Optional[Sequence[bool]] = None):
    """[(Y, dY) per layer]: the oracle's pre-activation and a bound on |Y_gpu - Y|.

    multiply_first[l]: the GPU ran layer l as A_hat (H W) (fp32 GCN layers only),
    whose rounding differs from the textbook order's."""
    L = len(Ws)
    nL = part.n_local
    mf = list(multiply_first) if multiply_first is not None else [False] * L
    wts = oracle.gcn_dinv(part) if agg == "gcn" else oracle.sage_invcnt(part)
    m = np.diff(np.asarray(part.rowptr, dtype=np.int64)).astype(np.float64)
    gam_row = ((m + 4.0) * U32 * SAFETY)[:, None]
    dH = np.zeros_like(ref["H"][0])  # layer 0: the features and the table rows are exact copies
    out = []
    for l in range(L):
        H = ref["H"][l]
        f = H.shape[1]
        Z, W = ref["Z"][l], Ws[l]
        K = W.shape[0]
        gam_k = (K + 4.0) * U32 * SAFETY
        Y = Z @ W
        if mf[l]:
            assert agg == "gcn" and not act_bf16
            # T = H W on every row (fp32), then the aggregation of T
            dT = dH @ np.abs(W) + gam_k * (np.abs(H) @ np.abs(W))
            T = H @ W
            dY = (oracle.aggregate(part, dT, W.shape[1], agg, weights=wts)
                  + gam_row * oracle.aggregate(part, np.abs(T), W.shape[1], agg, weights=wts) + U32 * np.abs(Y))
        else:
            Zraw = oracle.aggregate(part, H, f, agg, weights=wts)
            Zabs = oracle.aggregate(part, np.abs(H), f, agg, weights=wts)
            D = oracle.aggregate(part, dH, f, agg, weights=wts) + gam_row * Zabs
            if agg == "sage":
                D[:, :f] = dH[:nL]  # the self half is a copy of the input row
            if act_bf16:
                dZ = oracle.round_bf16(Zraw + D) - oracle.round_bf16(Zraw - D)
            else:
                dZ = D + U32 * np.abs(Zraw)
            dY = dZ @ np.abs(W) + gam_k * (np.abs(Z) @ np.abs(W))
        out.append((Y, dY))
        if l + 1 < L:
            hi, lo = np.maximum(Y + dY, 0.0), np.maximum(Y - dY, 0.0)
            if act_bf16:
                dHo = oracle.round_bf16(hi) - oracle.round_bf16(lo)
            else:
                dHo = (hi - lo) + U32 * np.abs(Y)
            dH = np.zeros_like(ref["H"][l + 1])
            dH[:nL] = dHo
    return out


def ambiguous_masks(fwd) -> List[Optional[np.ndarray]]:
    """Per layer, the pre-activations whose ReLU decision may differ (None for the last layer)."""
    return [np.abs(Y) <= dY for (Y, dY) in fwd[:-1]] + [None]


def relu_flip_bounds(part, ref: dict, Ws: Sequence[np.ndarray], agg: str, amb: Sequence[Optional[np.ndarray]]):
    """(dW bounds, dH bounds) per layer: how far any choice of the ambiguous
    decisions can move each gradient entry from the oracle's value."""
    L = len(Ws)
    nL = part.n_local
    T = ref["T"]
    Gb = np.zeros_like(ref["G"][L - 1])  # the loss gradient involves no ReLU decision
    dWb: List[Optional[np.ndarray]] = [None] * L
    dHb: List[Optional[np.ndarray]] = [None] * L
    for l in reversed(range(L)):
        Z, W, G = ref["Z"][l], Ws[l], ref["G"][l]
        if amb[l] is not None:
            on = ref["Hout"][l] > 0
            E = Gb * (on | amb[l]) + np.abs(G) * amb[l]
        else:
            E = Gb
        dWb[l] = np.abs(Z).T @ E
        if l > 0:
            f = Z.shape[1] if agg == "gcn" else Z.shape[1] // 2
            dHb[l] = oracle.aggregate_backward(part, T, E @ np.abs(W).T, f, agg)
            Gb = dHb[l][:nL]
    return dWb, dHb


def epoch_bounds(part, ref: dict, Ws: Sequence[np.ndarray], agg: str, act_bf16: bool,
                 multiply_first: Optional[Sequence[bool]] = None):
    """(dW bounds, dH bounds, number of ambiguous decisions) of an oracle epoch."""
    amb = ambiguous_masks(forward_difference_bounds(part, ref, Ws, agg, act_bf16, multiply_first))
    dWb, dHb = relu_flip_bounds(part, ref, Ws, agg, amb)
    return dWb, dHb, int(sum(int(a.sum()) for a in amb if a is not None))


def close_bounded(gpu: np.ndarray, ref: np.ndarray, tol: float, bound: Optional[np.ndarray], what: str = ""):
    """|x - r| <= tol * (|r| + rms(r)) + bound, elementwise (bound None or 0: strict)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    slack = tol * (np.abs(ref) + rms)
    if bound is not None:
        slack = slack + np.asarray(bound, dtype=np.float64)
    bad = np.abs(gpu - ref) > slack
    if np.any(bad):
        i = tuple(np.argwhere(bad)[0])
        excused = 0 if bound is None else int(np.count_nonzero(bound))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance "
                             f"({excused} entries carry a ReLU-flip bound); first at {i}: gpu {gpu[i]!r} "
                             f"ref {ref[i]!r} bound {0.0 if bound is None else float(bound[i])!r} (rms {rms:.3g})")
