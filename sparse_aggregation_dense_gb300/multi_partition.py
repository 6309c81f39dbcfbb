"""Several partitions of one graph trained together on one GPU.

The pages train one partition per GPU and exchange, every layer, the HALO
rows in the forward pass and the HALO feature gradients (J) in the backward
pass (Sylvie page, Alg. 1 / Alg. 2), or read and write a table of stale
representations instead of waiting for the exchange (DIGEST page, Fig. 1c;
Sylvie-A's pipelining).  This driver runs P partitions' kernels one after the
other on one GPU with the exchange going through tables in HBM:

* forward: table T_l holds layer l's input rows by global vertex id; each
  partition pulls its halo rows from it and pushes its fresh local rows to
  T_{l+1};
* backward: each partition's transposed aggregation also yields the gradients
  of its halo rows (J); they are added into an fp32 gradient table by global
  id (gnn_halo_grad_send) and every partition adds the entries of its own
  vertices to its local gradient (gnn_halo_grad_recv);
* the loss is the mean over all partitions' rows (gnn_softmax_ce_partial) and
  dW is the sum of the partitions' dW (the parameter synchronisation of data
  parallel training, a plain sum here because all partitions share one GPU).

Two schedules:

* "sync": layer by layer across partitions, so every pull reads rows pushed in
  the same epoch and every gradient is complete: the epoch computes exactly
  the unpartitioned layer (tested against the whole-graph oracle);
* "stale": each partition runs its whole epoch on the tables (and gradient
  table) of the previous epoch and writes the next epoch's, as DIGEST and
  Sylvie-A do; with sync_every = k every k-th epoch runs "sync" instead (the
  bounded-staleness forced synchronisation of Sylvie-A).
"""
from typing import List, Sequence

import torch

from . import gnn
from .partition_model import PartitionModel, ld_for


class MultiPartitionTrainer:
    def __init__(self, parts, widths: Sequence[int], agg: str, dtype: torch.dtype, n_table: int,
                 mode: str = "sync", sync_every: int = 0, device="cuda", narrow: bool = False,
                 grad_dtype: torch.dtype = torch.float32):
        assert mode in ("sync", "stale")
        self.parts = list(parts)
        self.widths = list(widths)
        self.L = len(widths) - 1
        self.mode, self.sync_every = mode, sync_every
        self.dtype = dtype
        self.n_table = n_table
        self.models: List[PartitionModel] = [PartitionModel(p, widths, agg, dtype, device, narrow=narrow,
                                                            grad_dtype=grad_dtype) for p in self.parts]
        self.n_rows = sum(m.n_local for m in self.models)
        dev = torch.device(device)
        # representation tables (current and, for the stale schedule, next) and gradient tables
        self.tables = [self._table(f, dev) for f in widths[:-1]]
        self.tables_next = [self._table(f, dev) for f in widths[:-1]] if mode == "stale" else None
        self.gtables = [torch.zeros((n_table, ld_for(f, torch.float32)), dtype=torch.float32, device=dev)[:, :f]
                        for f in widths[:-1]]
        self.gtables_next = ([torch.zeros_like(t) for t in self.gtables] if mode == "stale" else None)
        self.dW = [torch.zeros_like(w) for w in self.models[0].W]
        self.loss = torch.zeros(1, dtype=torch.float32, device=dev)
        self.epoch_index = 0

    def _table(self, f, dev):
        return torch.zeros((self.n_table, ld_for(f, self.dtype)), dtype=self.dtype, device=dev)[:, :f]

    # ---- inputs -----------------------------------------------------------
    def set_features(self, X: torch.Tensor):
        """Layer-0 table = X (n_table x f_0, all vertices); local rows of every partition copied in."""
        for t in ([self.tables[0]] + ([self.tables_next[0]] if self.tables_next else [])):
            t.copy_(X)
        for m in self.models:
            m.H[0][:m.n_local] = X[m.local_ids]

    def set_weights(self, Ws: Sequence[torch.Tensor]):
        for m in self.models:
            for w, src in zip(m.W, Ws):
                w.copy_(src)

    def set_labels(self, y: torch.Tensor):
        """y: int32 labels of all vertices, by global id."""
        for m in self.models:
            m.labels.copy_(y[m.local_ids])

    # ---- one epoch --------------------------------------------------------
    def epoch(self):
        sync = self.mode == "sync" or (self.sync_every > 0 and (self.epoch_index + 1) % self.sync_every == 0)
        if sync:
            self._epoch_sync()
        else:
            self._epoch_stale()
        self.epoch_index += 1

    def _loss(self):
        self.loss.zero_()
        for m in self.models:
            gnn.softmax_ce_partial(m.out_last, m.labels, m.G_last, m.row_loss, m.loss, self.n_rows)
        for m in self.models:
            self.loss += m.loss  # the partitions' shares of the mean

    def _sum_dw(self):
        for l in range(self.L):
            self.dW[l].zero_()
            for m in self.models:
                self.dW[l] += m.dW[l]

    def _epoch_sync(self):
        ms = self.models
        for l in range(self.L):
            for m in ms:
                if m.n_halo:
                    gnn.halo_pull(m.graph, self.tables[l], m.halo_ids, m.H[l])
                m.layer_forward(l)
            if l + 1 < self.L:
                for m in ms:
                    gnn.halo_push(m.graph, m.layer_out(l), m.local_ids, self.tables[l + 1])
        self._loss()
        for l in reversed(range(self.L)):
            for m in ms:
                self._backward_layer(m, l)
            if l > 0:
                gt = self.gtables[l]
                gt.zero_()
                for m in ms:
                    if m.n_halo:
                        gnn.halo_grad_send(m.graph, m.dH[l], m.halo_ids, gt)
                for m in ms:
                    gnn.halo_grad_recv(m.graph, gt, m.local_ids, m.dH[l][:m.n_local])
        self._sum_dw()

    def _epoch_stale(self):
        for gt in self.gtables_next:
            gt.zero_()
        for m in self.models:
            for l in range(self.L):
                if m.n_halo:
                    gnn.halo_pull(m.graph, self.tables[l], m.halo_ids, m.H[l])
                m.layer_forward(l)
                if l + 1 < self.L:
                    gnn.halo_push(m.graph, m.layer_out(l), m.local_ids, self.tables_next[l + 1])
        self._loss()
        for m in self.models:
            for l in reversed(range(self.L)):
                self._backward_layer(m, l)
                if l > 0:
                    # last epoch's gradients of this partition's vertices from the others; this epoch's J out
                    gnn.halo_grad_recv(m.graph, self.gtables[l], m.local_ids, m.dH[l][:m.n_local])
                    if m.n_halo:
                        gnn.halo_grad_send(m.graph, m.dH[l], m.halo_ids, self.gtables_next[l])
        self._sum_dw()
        self.tables, self.tables_next = self.tables_next, self.tables
        self.gtables, self.gtables_next = self.gtables_next, self.gtables

    def _backward_layer(self, m: PartitionModel, l: int):
        m.layer_backward(l, want_halo_grad=True)

    def check_errors(self):
        for m in self.models:
            m.check_errors()
