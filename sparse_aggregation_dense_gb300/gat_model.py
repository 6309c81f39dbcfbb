"""One partition's L-layer graph-attention model driven through the C ABI.

The same epoch as PartitionModel (DIGEST pull / push of the stale tables,
Sylvie's halo gradients J out of every backward layer), with attention layers
(gnn_gat_forward / gnn_gat_backward) instead of GCN / GraphSAGE ones.  No
arithmetic happens here; every step runs in libgnn's kernels.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import gnn
from .partition_model import padded


class GatModel:
    """Device state of one partition and its L-layer GAT.

    part: as for PartitionModel; widths [f_0, ..., f_L]; dtype: the activations,
    grad_dtype: the activation gradients (fp32 by default); hidden_relu: ReLU
    after the hidden layers (identity on the last layer either way)."""

    def __init__(self, part, widths: Sequence[int], dtype: torch.dtype, device="cuda",
                 grad_dtype: torch.dtype = torch.float32, hidden_relu: bool = True):
        if dtype == torch.float32 and grad_dtype != torch.float32:
            raise ValueError("fp32 activations take fp32 gradients")
        self.widths = list(widths)
        self.L = len(widths) - 1
        self.hidden_relu = hidden_relu
        self.dtype, self.grad_dtype = dtype, grad_dtype
        self.device = torch.device(device)
        dev = self.device
        self.n_local, self.n_halo, self.n_table = part.n_local, part.n_halo, part.n_table
        nL, nT = self.n_local, self.n_local + self.n_halo
        self.nnz = int(part.colidx.shape[0])
        self.rowptr = torch.from_numpy(np.ascontiguousarray(part.rowptr)).to(dev)
        self.colidx = torch.from_numpy(np.ascontiguousarray(part.colidx)).to(dev)
        self.local_ids = torch.from_numpy(np.ascontiguousarray(part.local_ids)).to(dev)
        self.halo_ids = torch.from_numpy(np.ascontiguousarray(part.halo_ids)).to(dev)
        self.graph = gnn.graph_create(self.rowptr, self.colidx, nL, self.n_halo, None, "gat")
        L = self.L
        self.H = [padded(nT, widths[l], dtype, dev) for l in range(L)]
        self.out_last = padded(nL, widths[-1], dtype, dev)
        self.T = [padded(nT, widths[l + 1], dtype, dev) for l in range(L)]
        self.scores = [torch.zeros(nT + nL, dtype=torch.float32, device=dev) for _ in range(L)]
        self.alpha = [torch.zeros(self.nnz, dtype=torch.float32, device=dev) for _ in range(L)]
        self.W = [torch.zeros((widths[l], widths[l + 1]), dtype=torch.float32, device=dev) for l in range(L)]
        self.a_src = [torch.zeros(widths[l + 1], dtype=torch.float32, device=dev) for l in range(L)]
        self.a_dst = [torch.zeros(widths[l + 1], dtype=torch.float32, device=dev) for l in range(L)]
        self.dW = [torch.zeros_like(w) for w in self.W]
        self.da_src = [torch.zeros_like(a) for a in self.a_src]
        self.da_dst = [torch.zeros_like(a) for a in self.a_dst]
        gdt = grad_dtype
        self.dT = padded(nT, max(widths[1:]), gdt, dev)
        self.dH = [None] + [padded(nT, widths[l], gdt, dev) for l in range(1, L)]
        self.G_last = padded(nL, widths[-1], gdt, dev)
        self.tables: List[Optional[torch.Tensor]] = [None] * L
        self.labels = torch.zeros(nL, dtype=torch.int32, device=dev)
        self.row_loss = torch.zeros(max(nL, 1), dtype=torch.float32, device=dev)
        self.loss = torch.zeros(1, dtype=torch.float32, device=dev)

    def _relu(self, l: int) -> bool:
        return self.hidden_relu and l < self.L - 1

    def layer_out(self, l: int) -> torch.Tensor:
        return self.out_last if l == self.L - 1 else self.H[l + 1][:self.n_local]

    def grad_out(self, l: int) -> torch.Tensor:
        return self.G_last if l == self.L - 1 else self.dH[l + 1][:self.n_local]

    def forward(self):
        for l in range(self.L):
            if self.n_halo:
                gnn.halo_pull(self.graph, self.tables[l], self.halo_ids, self.H[l])
            gnn.gat_forward(self.graph, self.H[l], self.W[l], self.a_src[l], self.a_dst[l], self._relu(l), self.T[l],
                            self.scores[l], self.alpha[l], self.layer_out(l))
            if l + 1 < self.L:
                gnn.halo_push(self.graph, self.layer_out(l), self.local_ids, self.tables[l + 1])

    def loss_grad(self):
        gnn.softmax_ce(self.out_last, self.labels, self.G_last, self.row_loss, self.loss)

    def backward(self):
        for l in reversed(range(self.L)):
            dT = self.dT[:, :self.widths[l + 1]]
            gnn.gat_backward(self.graph, self.grad_out(l), self.layer_out(l), self.H[l], self.W[l], self.a_src[l],
                             self.a_dst[l], self._relu(l), self.T[l], self.scores[l], self.alpha[l], self.dW[l],
                             self.da_src[l], self.da_dst[l], dT, self.dH[l] if l > 0 else None)

    def step(self):
        self.forward()
        self.loss_grad()
        self.backward()

    def check_errors(self):
        st = gnn.get_error(self.graph)
        if st != gnn.GNN_OK:
            raise gnn.GnnError(st, "device error word")
