"""One partition's L-layer GCN / GraphSAGE model driven through the C ABI.

This module only allocates device buffers (torch) and issues the library's calls
in the order of one full-graph training epoch on one partition:

  for each layer l:   pull halo rows of layer l from the stale table (DIGEST pull)
                      forward: aggregate + update (+ ReLU except the last layer)
                      push the new local rows into the table of layer l + 1
  loss gradient       softmax cross-entropy over the local rows
  for l = L-1 .. 0:   backward: dW_l, and dH_l (local + halo rows) for l > 0

No arithmetic happens here; every step runs in libgnn's CUDA kernels.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import gnn


def ld_for(f: int, dtype: torch.dtype) -> int:
    m = 8 if dtype == torch.bfloat16 else 4
    return (f + m - 1) // m * m


def padded(rows: int, f: int, dtype: torch.dtype, device, fill: Optional[float] = 0.0) -> torch.Tensor:
    """A (rows x ld) buffer returned as its (rows x f) view."""
    buf = torch.empty((rows, ld_for(f, dtype)), dtype=dtype, device=device)
    if fill is not None:
        buf.zero_()
    return buf[:, :f]


class PartitionModel:
    """Device state of one partition and its L-layer model.

    part: an object with rowptr, colidx (int32 numpy), n_local, n_halo, deg (float32 numpy or
    None), local_ids, halo_ids (int64 numpy), n_table.
    widths: [f_0, ..., f_L]; agg "gcn" | "sage"; dtype torch.float32 | torch.bfloat16: the activations
    (features, tables, Z, layer outputs).  grad_dtype: the activation gradients (G, dZ, dH); fp32 by default,
    bf16 allowed with bf16 activations.  reorder: the backward of GCN layers l > 0 (bf16 activations, fp32
    gradients) gathers dY instead of dZ: dH = (A_hat^T dY) W^T, the other order of the same products.
    """

    def __init__(self, part, widths: Sequence[int], agg: str, dtype: torch.dtype, device="cuda",
                 overlap: bool = False, narrow: bool = False, grad_dtype: torch.dtype = torch.float32,
                 reorder: bool = False):
        if dtype == torch.float32 and grad_dtype != torch.float32:
            raise ValueError("fp32 activations take fp32 gradients")
        if narrow and grad_dtype != dtype:
            raise ValueError("the multiplication-first layers store their gradients in the activations' dtype")
        self.grad_dtype = grad_dtype
        self.widths = list(widths)
        # overlap: pulls and pushes run on a second stream, concurrently with the layers (DIGEST
        # system design, Fig. 1c: the table traffic is decoupled from the computation).  The rows a
        # partition pulls (its halo) and pushes (its local vertices) are disjoint, so the schedule
        # computes exactly what the sequential one does.
        self.overlap = overlap
        self.side = torch.cuda.Stream(device=device) if overlap else None
        self.L = len(widths) - 1
        self.agg = agg
        self.dtype = dtype
        self.device = torch.device(device)
        self.n_local, self.n_halo, self.n_table = part.n_local, part.n_halo, part.n_table
        dev = self.device
        self.rowptr = torch.from_numpy(np.ascontiguousarray(part.rowptr)).to(dev)
        self.colidx = torch.from_numpy(np.ascontiguousarray(part.colidx)).to(dev)
        self.deg = None if part.deg is None else torch.from_numpy(np.ascontiguousarray(part.deg)).to(dev)
        self.local_ids = torch.from_numpy(np.ascontiguousarray(part.local_ids)).to(dev)
        self.halo_ids = torch.from_numpy(np.ascontiguousarray(part.halo_ids)).to(dev)
        self.graph = gnn.graph_create(self.rowptr, self.colidx, self.n_local, self.n_halo, self.deg, agg)
        nL, nT = self.n_local, self.n_local + self.n_halo
        self.nnz = int(part.colidx.shape[0])
        sage = agg == "sage"
        self.Kp = [2 * gnn.sage_half_offset(f, dtype) if sage else f for f in widths[:-1]]
        # layer inputs H[l] (local + halo rows); the local rows of H[l+1] are layer l's output
        self.H = [padded(nT, widths[l], dtype, dev) for l in range(self.L)]
        self.out_last = padded(nL, widths[-1], dtype, dev)
        # narrow layers (GCN, output narrower than input) multiply first: A (H W), so their aggregations run
        # at the output width; they keep T = H W (all rows) instead of Z
        self.narrow = [narrow and not sage and widths[l + 1] < widths[l] for l in range(self.L)]
        self.Z = [None if self.narrow[l] else padded(nL, self.Kp[l], dtype, dev) for l in range(self.L)]
        self.T = [padded(nT, widths[l + 1], dtype, dev) if self.narrow[l] else None for l in range(self.L)]
        self.P = padded(nT, max([widths[l + 1] for l in range(self.L) if self.narrow[l]] + [1]), grad_dtype, dev) \
            if any(self.narrow) else None
        self._alloc_grads()
        self.reorder = False
        self.Pr = None
        if reorder:
            self.set_reorder(True)
        self.W: List[torch.Tensor] = []
        self.dW: List[torch.Tensor] = []
        for l in range(self.L):
            K = (2 if sage else 1) * widths[l]
            self.W.append(torch.zeros((K, widths[l + 1]), dtype=torch.float32, device=dev))
            self.dW.append(torch.zeros((K, widths[l + 1]), dtype=torch.float32, device=dev))
        self.tables: List[Optional[torch.Tensor]] = [None] * self.L
        self.labels = torch.zeros(nL, dtype=torch.int32, device=dev)
        self.row_loss = torch.zeros(max(nL, 1), dtype=torch.float32, device=dev)
        self.loss = torch.zeros(1, dtype=torch.float32, device=dev)
        # inputs of the next epoch staged by stage_inputs, and the event its copies complete
        self._staged = None
        self._inputs_ready = None
        self._copy_stream = None

    def _alloc_grads(self):
        nL, nT, gdt, dev = self.n_local, self.n_local + self.n_halo, self.grad_dtype, self.device
        self.dZ = padded(nL, max(self.Kp[1:] + [1]), gdt, dev)
        self.dH = [None] + [padded(nT, self.widths[l], gdt, dev) for l in range(1, self.L)]
        self.G_last = padded(nL, self.widths[-1], gdt, dev)

    def set_grad_dtype(self, grad_dtype: torch.dtype):
        """Store the activation gradients in another dtype from the next step on
        (the gradient buffers are reallocated)."""
        if self.dtype == torch.float32 and grad_dtype != torch.float32:
            raise ValueError("fp32 activations take fp32 gradients")
        if any(self.narrow) and grad_dtype != self.dtype:
            raise ValueError("the multiplication-first layers store their gradients in the activations' dtype")
        if self.reorder and grad_dtype != torch.float32:
            raise ValueError("the reordered backward takes fp32 gradients")
        if grad_dtype != self.grad_dtype:
            self.dZ = self.dH = self.G_last = None
            self.grad_dtype = grad_dtype
            self._alloc_grads()

    def _reordered(self, l: int) -> bool:
        return self.reorder and l > 0 and not self.narrow[l]

    def set_reorder(self, on: bool):
        """Run the backward of GCN layers l > 0 in the other product order from the next step on: P = A_hat^T dY
        (bf16, local and halo rows), dH = P W^T.  Needs bf16 activations with fp32 gradients."""
        if on and (self.agg != "gcn" or self.dtype != torch.bfloat16 or self.grad_dtype != torch.float32):
            raise ValueError("the reordered backward takes GCN layers with bf16 activations and fp32 gradients")
        if on and self.Pr is None:
            nT = self.n_local + self.n_halo
            self.Pr = padded(nT, max([self.widths[l + 1] for l in range(1, self.L)] + [1]), torch.bfloat16,
                             self.device)
        self.reorder = on

    # ---- views ------------------------------------------------------------
    def layer_out(self, l: int) -> torch.Tensor:
        """Output of layer l (n_local x f_{l+1})."""
        return self.out_last if l == self.L - 1 else self.H[l + 1][:self.n_local]

    def grad_out(self, l: int) -> torch.Tensor:
        """Gradient with respect to the output of layer l."""
        return self.G_last if l == self.L - 1 else self.dH[l + 1][:self.n_local]

    def dZ_view(self, l: int) -> torch.Tensor:
        return self.dZ[:, :self.Kp[l]]

    # ---- input staging ----------------------------------------------------
    def stage_inputs(self, x: torch.Tensor, y: torch.Tensor):
        """Copy the next epoch's inputs while the next call of step() runs: x, the features of the local rows
        (n_local x f_0, or n_local x the row stride of H[0] with its padding columns), and y, the n_local
        labels, both pinned host tensors.  The features are copied once layer 0 has read H[0] (after its
        backward for a multiplication-first layer 0), the labels once the loss has read them, on a copy
        stream; the epoch after that waits for both copies before it starts."""
        if x.shape[0] != self.n_local or y.shape[0] != self.n_local:
            raise ValueError("stage_inputs takes n_local rows of features and n_local labels")
        if self._copy_stream is None:
            self._copy_stream = torch.cuda.Stream(device=self.device)
        self._staged = (x, y)

    def _h0_local(self, width: int) -> torch.Tensor:
        ld = self.H[0].stride(0)
        if width == ld:
            return self.H[0].as_strided((self.n_local + self.n_halo, ld), (ld, 1))[:self.n_local]
        return self.H[0][:self.n_local]

    def _copy_after(self, src: torch.Tensor, dst: torch.Tensor):
        """dst <- src on the copy stream, after the work queued so far on the current stream."""
        done = torch.cuda.Event()
        done.record(torch.cuda.current_stream(self.device))
        self._copy_stream.wait_event(done)
        with torch.cuda.stream(self._copy_stream):
            dst.copy_(src, non_blocking=True)

    def _wait_inputs(self):
        if self._inputs_ready is not None:
            torch.cuda.current_stream(self.device).wait_event(self._inputs_ready)
            self._inputs_ready = None

    def _stage_features(self, l: int, after_backward: bool):
        if self._staged is not None and l == 0 and self.narrow[0] == after_backward:
            x = self._staged[0]
            self._copy_after(x, self._h0_local(x.shape[1]))

    def _stage_labels(self):
        if self._staged is not None:
            self._copy_after(self._staged[1], self.labels)

    def _staging_done(self):
        """End of the epoch's backward: both copies are queued; the next epoch waits for them."""
        if self._staged is not None:
            ready = torch.cuda.Event()
            ready.record(self._copy_stream)
            self._inputs_ready = ready
            self._staged = None

    # ---- one epoch --------------------------------------------------------
    def forward(self):
        self._wait_inputs()
        if self.overlap:
            return self._forward_overlapped()
        for l in range(self.L):
            if self.n_halo:
                gnn.halo_pull(self.graph, self.tables[l], self.halo_ids, self.H[l])
            self._layer_forward(l)
            self._stage_features(l, False)
            if l + 1 < self.L:
                gnn.halo_push(self.graph, self.layer_out(l), self.local_ids, self.tables[l + 1])

    def _forward_overlapped(self):
        main = torch.cuda.current_stream(self.device)
        start = torch.cuda.Event()
        start.record(main)  # everything before this epoch (earlier readers of the halo rows) is done
        pulled = [torch.cuda.Event() for _ in range(self.L)]
        with torch.cuda.stream(self.side):
            self.side.wait_event(start)
            for l in range(self.L):
                if self.n_halo:
                    gnn.halo_pull(self.graph, self.tables[l], self.halo_ids, self.H[l])
                pulled[l].record(self.side)
        for l in range(self.L):
            main.wait_event(pulled[l])
            self._layer_forward(l)
            self._stage_features(l, False)
            if l + 1 < self.L:
                done = torch.cuda.Event()
                done.record(main)
                with torch.cuda.stream(self.side):
                    self.side.wait_event(done)
                    gnn.halo_push(self.graph, self.layer_out(l), self.local_ids, self.tables[l + 1])
        pushed = torch.cuda.Event()
        pushed.record(self.side)
        main.wait_event(pushed)  # the epoch ends when its pushes have landed

    def layer_forward(self, l: int):
        """Forward of layer l from H[l] (pulled halo rows included) into its output."""
        self._layer_forward(l)

    def _layer_forward(self, l: int):
        if self.narrow[l]:
            gnn.layer_forward_narrow(self.graph, self.H[l], self.W[l], l < self.L - 1, self.T[l], self.layer_out(l))
        else:
            gnn.layer_forward(self.graph, self.H[l], self.W[l], l < self.L - 1, self.Z[l], self.layer_out(l))

    def loss_grad(self, n_mean: Optional[int] = None):
        """Mean softmax cross-entropy of the local rows and its gradient; with n_mean, this partition's share of
        the mean over n_mean rows held by several partitions."""
        if n_mean is None:
            gnn.softmax_ce(self.out_last, self.labels, self.G_last, self.row_loss, self.loss)
        else:
            gnn.softmax_ce_partial(self.out_last, self.labels, self.G_last, self.row_loss, self.loss, n_mean)
        self._stage_labels()

    def backward(self, want_halo_grad: bool = True):
        for l in reversed(range(self.L)):
            self.layer_backward(l, want_halo_grad)

    def layer_backward(self, l: int, want_halo_grad: bool = True):
        """Backward of layer l: dW[l], and for l > 0 the gradient dH[l] of its input (halo rows too when
        want_halo_grad; a narrow layer always writes them)."""
        if self.narrow[l]:
            P = self.P[:, :self.widths[l + 1]]
            gnn.layer_backward_narrow(self.graph, self.grad_out(l), self.layer_out(l), self.H[l], self.W[l],
                                      l < self.L - 1, self.dW[l], P, self.dH[l] if l > 0 else None)
        elif self._reordered(l):
            rows = self.n_local + self.n_halo if want_halo_grad else self.n_local
            gnn.layer_backward_reordered(self.graph, self.grad_out(l), self.layer_out(l), self.Z[l], self.W[l],
                                         l < self.L - 1, self.dW[l], self.Pr[:rows, :self.widths[l + 1]],
                                         self.dH[l][:rows], want_halo_grad=want_halo_grad)
        elif l > 0:
            gnn.layer_backward(self.graph, self.grad_out(l), self.layer_out(l), self.Z[l], self.W[l],
                               l < self.L - 1, self.dW[l], self.widths[l], dZ=self.dZ_view(l),
                               dH=self.dH[l] if want_halo_grad else self.dH[l][:self.n_local],
                               want_halo_grad=want_halo_grad)
        else:
            gnn.layer_backward(self.graph, self.grad_out(l), self.layer_out(l), self.Z[l], self.W[l],
                               l < self.L - 1, self.dW[l], self.widths[l])
        self._stage_features(l, True)
        if l == 0:
            self._staging_done()

    def step(self):
        self.forward()
        self.loss_grad()
        self.backward()

    def check_errors(self):
        st = gnn.get_error(self.graph)
        if st != gnn.GNN_OK:
            raise gnn.GnnError(st, "device error word")
