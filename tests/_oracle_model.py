"""A CPU stand-in for PartitionModel whose layers are computed by the oracle
(test infrastructure: it lets the process-per-partition driver run on gloo
ranks without a GPU).  Same attributes and methods as the driver uses."""
from __future__ import annotations

import numpy as np
import torch

import oracle


class OracleModel:
    def __init__(self, part, widths, agg, Ws):
        self.part = part
        self.widths = list(widths)
        self.L = len(widths) - 1
        self.agg = agg
        self.n_local, self.n_halo = part.n_local, part.n_halo
        nT = part.n_local + part.n_halo
        self.H = [torch.zeros((nT, widths[l]), dtype=torch.float64) for l in range(self.L)]
        self.out_last = torch.zeros((part.n_local, widths[-1]), dtype=torch.float64)
        self.dH = [None] + [torch.zeros((nT, widths[l]), dtype=torch.float64) for l in range(1, self.L)]
        self.W = [np.asarray(w, np.float64) for w in Ws]
        self.dW = [torch.zeros(w.shape, dtype=torch.float64) for w in self.W]
        self.Z = [None] * self.L
        self.Hout = [None] * self.L
        self.G_last = None
        self.labels = np.zeros(part.n_local, np.int32)
        self.loss = torch.zeros(1, dtype=torch.float64)
        self.T = oracle.transpose(part)

    def layer_out(self, l):
        return self.out_last if l == self.L - 1 else self.H[l + 1][:self.n_local]

    def layer_forward(self, l):
        Z, Ho = oracle.layer_forward(self.part, self.H[l].numpy(), self.W[l], self.agg, relu=l < self.L - 1)
        self.Z[l], self.Hout[l] = Z, Ho
        self.layer_out(l)[:] = torch.from_numpy(Ho)

    def loss_grad(self, n_mean=None):
        loss, G = oracle.softmax_ce(self.out_last.numpy(), self.labels)
        share = self.n_local / (n_mean or self.n_local)
        self.loss[0] = loss * share
        self.G_last = G * share

    def layer_backward(self, l, want_halo_grad=True):
        G = self.G_last if l == self.L - 1 else self.dH[l + 1][:self.n_local].numpy()
        dW, _, dH = oracle.layer_backward(self.part, self.T, G, self.Hout[l], self.Z[l], self.W[l], self.agg,
                                          relu=l < self.L - 1, want_dh=l > 0)
        self.dW[l][:] = torch.from_numpy(dW)
        if l > 0:
            self.dH[l][:] = torch.from_numpy(dH)

    def check_errors(self):
        pass


class NumpyRowOps:
    """Row gather and ordered scatter-add on CPU tensors (numpy indexing)."""

    @staticmethod
    def gather_rows(src, ids, dst):
        dst[:] = src[ids.long()]

    @staticmethod
    def scatter_add_rows(src, ids, dst):
        idx = ids.long()
        assert idx.unique().numel() == idx.numel()
        dst[idx] += src

    @staticmethod
    def quantize_rows(X, keys, codes, sz, bits, seed):
        c, z = oracle.quantize_rows(X.numpy().astype(np.float32), keys.numpy(), bits, seed, ld_codes=codes.shape[1])
        codes[:] = torch.from_numpy(c)
        sz[:] = torch.from_numpy(z)

    @staticmethod
    def dequantize_rows(codes, sz, bits, dst, ids=None, add=False):
        f = dst.shape[1]
        y = torch.from_numpy(oracle.dequantize_rows(codes.numpy(), sz.numpy(), f, bits).astype(np.float64))
        idx = torch.arange(codes.shape[0]) if ids is None else ids.long()
        if add:
            dst[idx] += y
        else:
            dst[idx] = y
