"""One graph partition per process: the halo exchange of full-graph training.

The pages train one partition per GPU (Sylvie page, Graph Engine and the
Communicator; DIGEST page, system design).  Every layer, a partition needs the
rows of its HALO vertices - vertices another partition owns - and in the
backward pass it returns the feature gradients J of those rows to their owners,
who add them to their own gradients before going down a layer (Sylvie Alg. 1
and Alg. 2).  The parameter gradients are summed over the partitions (data
parallel training).

This driver runs the rank's partition through :class:`PartitionModel` (the C
ABI) and moves rows between ranks with ``torch.distributed``:

* set-up (host, once): every rank's vertex lists are gathered; the partition's
  halo vertices are reordered by owning rank, so the rows received from rank q
  form one contiguous block of the halo rows; each rank learns which of its
  rows every other rank needs (an :class:`ExchangePlan`);
* forward, per layer: the rows to send are gathered on the device
  (``gnn_gather_rows``) and one all-to-all delivers every rank's halo rows
  straight into the halo rows of its layer input;
* backward, per layer above the first: the halo rows of dH (J) go back with the
  reverse all-to-all and each owner adds them to its local rows
  (``gnn_scatter_add_rows``, one call per sending rank, in rank order, so the
  sums are reproducible);
* the loss is each rank's share of the mean over all ranks' rows, and the
  parameter gradients dW are all-reduced (summed).

With ``codec_bits`` the rows and the J rows cross as b-bit codes with a
per-row scale and zero point (Sylvie page, Quantizer / Dequantizer): the
sender quantises (``gnn_quantize_rows``, stochastic rounding keyed by the
vertex's global id, the epoch, layer and direction), the receiver
dequantises into the halo rows or adds into its own rows
(``gnn_dequantize_rows``).

Schedules: "sync" exchanges each layer's fresh rows before that layer (the
epoch computes exactly the unpartitioned layer); "stale" exchanges at the
start of the epoch the rows every rank computed in the previous epoch, and adds
the J rows received in the previous epoch (DIGEST's stale representations,
Sylvie-A's asynchronous pipeline); with ``sync_every = k`` every k-th epoch is
a sync epoch (Sylvie-A's bounded staleness).

The collective runs on the process group's backend: NCCL moves device
buffers directly; gloo (CPU ranks, or processes that share one GPU) stages them
through host memory.  No kernel waits on another rank: every exchange is a
collective between launches.
"""
from __future__ import annotations

from types import SimpleNamespace
from typing import List, Optional, Sequence

import numpy as np
import torch
import torch.distributed as dist

from . import gnn
from .partition_model import PartitionModel, ld_for


def _full_rows(t: torch.Tensor) -> torch.Tensor:
    """The whole leading-dimension rows behind a (rows x f) column view."""
    ld = t.stride(0) if t.dim() == 2 and t.shape[0] > 0 else t.shape[1]
    return t.as_strided((t.shape[0], ld), (ld, 1))


def order_halo_by_owner(part, owner: np.ndarray):
    """The partition with its halo vertices reordered by owning rank (stable
    within a rank): columns, halo ids and degrees permuted alike."""
    nL, nH = part.n_local, part.n_halo
    own = owner[part.halo_ids] if nH else np.zeros(0, np.int64)
    order = np.argsort(own, kind="stable")
    newpos = np.empty(nH, np.int64)
    newpos[order] = np.arange(nH)
    colmap = np.concatenate([np.arange(nL), nL + newpos]).astype(np.int32)
    deg = None
    if part.deg is not None:
        deg = np.concatenate([part.deg[:nL], part.deg[nL:][order]]).astype(np.float32)
    return SimpleNamespace(rowptr=part.rowptr, colidx=colmap[part.colidx], n_local=nL, n_halo=nH, deg=deg,
                           local_ids=part.local_ids, halo_ids=part.halo_ids[order], n_table=part.n_table,
                           nnz=int(part.colidx.shape[0]), n_total=nL + nH)


class ExchangePlan:
    """Rows a rank sends to and receives from every rank.

    recv_counts[q]: halo rows owned by rank q (contiguous, in rank order);
    send_counts[q]: rows of this rank that rank q holds as halo rows;
    send_pos: local row positions, concatenated by destination rank, each
    destination's rows in the order of that rank's halo list."""

    def __init__(self, rank: int, world: int, local_ids_all: Sequence[np.ndarray],
                 halo_ids_all: Sequence[np.ndarray], n_table: int):
        owner = np.full(n_table, -1, np.int64)
        for q, ids in enumerate(local_ids_all):
            if np.any(owner[ids] >= 0):
                raise ValueError("partitions overlap: a vertex is local to two ranks")
            owner[ids] = q
        mine = np.asarray(halo_ids_all[rank], np.int64)
        if mine.size and (np.any(owner[mine] < 0) or np.any(owner[mine] == rank)):
            raise ValueError("a halo vertex is owned by no other rank")
        self.owner = owner
        self.recv_counts = [int(np.sum(owner[mine] == q)) for q in range(world)]
        if np.any(np.diff(owner[mine]) < 0):
            raise ValueError("halo rows must be ordered by owning rank")
        pos = np.full(n_table, -1, np.int64)
        pos[local_ids_all[rank]] = np.arange(len(local_ids_all[rank]))
        send = []
        for q in range(world):
            h = np.asarray(halo_ids_all[q], np.int64)
            send.append(pos[h[owner[h] == rank]])
        self.send_counts = [int(s.shape[0]) for s in send]
        self.send_pos = np.concatenate(send) if send else np.zeros(0, np.int64)
        self.send_off = np.concatenate([[0], np.cumsum(self.send_counts)]).astype(np.int64)


class _Comm:
    """all-to-all and all-reduce of row buffers; gloo stages device buffers through host memory."""

    def __init__(self, group=None):
        self.group = group
        self.staged = dist.get_backend(group) != "nccl"

    def all_to_all(self, out: torch.Tensor, inp: torch.Tensor, out_splits: List[int], in_splits: List[int]):
        if self.staged and (out.is_cuda or inp.is_cuda):
            o = torch.empty(out.shape, dtype=out.dtype)
            dist.all_to_all_single(o, inp.cpu(), out_splits, in_splits, group=self.group)
            out.copy_(o)
        else:
            dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)

    def all_reduce_sum(self, t: torch.Tensor):
        if self.staged and t.is_cuda:
            h = t.cpu()
            dist.all_reduce(h, group=self.group)
            t.copy_(h)
        else:
            dist.all_reduce(t, group=self.group)


class _LibOps:
    """The device row kernels of the exchange (the C ABI)."""

    gather_rows = staticmethod(gnn.gather_rows)
    scatter_add_rows = staticmethod(gnn.scatter_add_rows)
    quantize_rows = staticmethod(gnn.quantize_rows)
    dequantize_rows = staticmethod(gnn.dequantize_rows)


class DistributedPartitionTrainer:
    """This rank's partition of one graph, trained with the other ranks' partitions.

    part: this rank's partition (rowptr, colidx, n_local, n_halo, deg, local_ids,
    halo_ids, n_table); widths, agg, dtype, grad_dtype as for PartitionModel.
    model_factory(part) builds the rank's model (default: PartitionModel on
    `device`); ops gives gather_rows / scatter_add_rows (default: libgnn's)."""

    def __init__(self, part, widths: Sequence[int], agg: str, dtype: torch.dtype, mode: str = "sync",
                 sync_every: int = 0, device="cuda", grad_dtype: torch.dtype = torch.float32, group=None,
                 model_factory=None, ops=None, codec_bits: Optional[int] = None, codec_seed: int = 0):
        assert mode in ("sync", "stale")
        assert codec_bits in (None, 1, 2, 4, 8)
        # Sylvie's low-bit messages: halo rows and returned J rows cross as b-bit
        # codes with a per-row scale and zero point (None: exact rows)
        self.codec_bits, self.codec_seed = codec_bits, codec_seed
        self.rank, self.world = dist.get_rank(group), dist.get_world_size(group)
        self.mode, self.sync_every = mode, sync_every
        self.comm = _Comm(group)
        self.ops = ops or _LibOps
        gathered: List = [None] * self.world
        dist.all_gather_object(gathered, np.asarray(part.local_ids, np.int64), group=group)
        owner = np.full(part.n_table, -1, np.int64)
        for q, ids in enumerate(gathered):
            owner[ids] = q
        self.part = order_halo_by_owner(part, owner)
        halos: List = [None] * self.world
        dist.all_gather_object(halos, self.part.halo_ids, group=group)
        self.plan = ExchangePlan(self.rank, self.world, gathered, halos, part.n_table)
        if model_factory is None:
            self.model = PartitionModel(self.part, widths, agg, dtype, device, grad_dtype=grad_dtype)
        else:
            self.model = model_factory(self.part)
        m = self.model
        self.L = m.L
        self.widths = list(widths)
        dev = m.H[0].device
        self.send_pos = torch.from_numpy(self.plan.send_pos).to(dev)
        n_send = int(self.plan.send_pos.shape[0])
        # send buffers of the forward rows (whole leading-dimension rows, like the layer inputs)
        self.send_rows = [torch.zeros((n_send, _full_rows(m.H[l]).shape[1]), dtype=m.H[l].dtype, device=dev)
                          for l in range(self.L)]
        # receive buffers of the returned J rows (like the local rows of dH)
        self.recv_J = [None] + [torch.zeros((n_send, _full_rows(m.dH[l]).shape[1]), dtype=m.dH[l].dtype,
                                            device=dev) for l in range(1, self.L)]
        self.J_pending = [None] * self.L  # stale schedule: J rows received last epoch, added this epoch
        if codec_bits:
            lid = torch.from_numpy(np.asarray(self.part.local_ids, np.int64)).to(dev)
            self.send_keys = lid[self.send_pos]  # global ids of the rows sent: the draws' keys
            self.halo_keys = torch.from_numpy(np.asarray(self.part.halo_ids, np.int64)).to(dev)
            n_halo = m.n_halo
            self.codes_send = [self._codes(n_send, self.widths[l], dev) for l in range(self.L)]
            self.codes_recv = [self._codes(n_halo, self.widths[l], dev) for l in range(self.L)]
            self.codesJ_send = [None] + [self._codes(n_halo, self.widths[l], dev) for l in range(1, self.L)]
            self.codesJ_recv = [None] + [self._codes(n_send, self.widths[l], dev) for l in range(1, self.L)]
        n_rows = torch.tensor([float(m.n_local)], dtype=torch.float64)
        dist.all_reduce(n_rows, group=group)
        self.n_rows = int(n_rows.item())
        self.epoch_index = 0

    def _codes(self, n: int, f: int, dev):
        """A message of n rows of f b-bit codes: (codes uint8 n x ld, scale / zero point float32 n x 2)."""
        return (torch.zeros((n, gnn.codec_row_bytes(f, self.codec_bits)), dtype=torch.uint8, device=dev),
                torch.zeros((n, 2), dtype=torch.float32, device=dev))

    def _seed(self, l: int, backward: bool) -> int:
        """Draws differ per epoch, layer and direction."""
        return self.codec_seed + (self.epoch_index << 9) + (l << 1) + int(backward)

    # ---- the two exchanges -----------------------------------------------
    def _send_rows(self, l: int):
        m = self.model
        f = self.widths[l]
        self.ops.gather_rows(m.H[l][:m.n_local], self.send_pos, self.send_rows[l][:, :f])

    def _exchange_rows(self, l: int):
        """All-to-all of the gathered rows of layer l into the halo rows of its input."""
        m = self.model
        if self.codec_bits:
            f = self.widths[l]
            (cs, zs), (cr, zr) = self.codes_send[l], self.codes_recv[l]
            self.ops.quantize_rows(self.send_rows[l][:, :f], self.send_keys, cs, zs, self.codec_bits,
                                   self._seed(l, False))
            self.comm.all_to_all(cr, cs, self.plan.recv_counts, self.plan.send_counts)
            self.comm.all_to_all(zr, zs, self.plan.recv_counts, self.plan.send_counts)
            self.ops.dequantize_rows(cr, zr, self.codec_bits, m.H[l][m.n_local:m.n_local + m.n_halo])
            return
        recv = _full_rows(m.H[l])[m.n_local:m.n_local + m.n_halo]
        self.comm.all_to_all(recv, self.send_rows[l], self.plan.recv_counts, self.plan.send_counts)

    def _return_J(self, l: int):
        """The halo rows of dH go back to their owners (into recv_J[l], or its codes)."""
        m = self.model
        if self.codec_bits:
            f = self.widths[l]
            (cs, zs), (cr, zr) = self.codesJ_send[l], self.codesJ_recv[l]
            self.ops.quantize_rows(m.dH[l][m.n_local:m.n_local + m.n_halo], self.halo_keys, cs, zs, self.codec_bits,
                                   self._seed(l, True))
            self.comm.all_to_all(cr, cs, self.plan.send_counts, self.plan.recv_counts)
            self.comm.all_to_all(zr, zs, self.plan.send_counts, self.plan.recv_counts)
            return
        J = _full_rows(m.dH[l])[m.n_local:m.n_local + m.n_halo]
        self.comm.all_to_all(self.recv_J[l], J, self.plan.send_counts, self.plan.recv_counts)

    def _add_J(self, l: int, J):
        """dH[l][v] += the J rows other ranks returned for v, one rank after another
        (J: rows, or (codes, scale / zero point) with the codec)."""
        m = self.model
        f = self.widths[l]
        off = self.plan.send_off
        for q in range(self.world):
            a, b = int(off[q]), int(off[q + 1])
            if b <= a:
                continue
            if self.codec_bits:
                codes, sz = J
                self.ops.dequantize_rows(codes[a:b], sz[a:b], self.codec_bits, m.dH[l][:m.n_local],
                                         ids=self.send_pos[a:b], add=True)
            else:
                self.ops.scatter_add_rows(J[a:b, :f], self.send_pos[a:b], m.dH[l][:m.n_local])

    # ---- one epoch --------------------------------------------------------
    def epoch(self):
        sync = self.mode == "sync" or (self.sync_every > 0 and (self.epoch_index + 1) % self.sync_every == 0)
        m = self.model
        if sync:
            for l in range(self.L):
                self._send_rows(l)
                self._exchange_rows(l)
                m.layer_forward(l)
        else:
            # last epoch's rows of every layer (layer 0: the features) travel before any compute
            for l in range(self.L):
                self._send_rows(l)
                self._exchange_rows(l)
            for l in range(self.L):
                m.layer_forward(l)
        m.loss_grad(n_mean=self.n_rows)
        self.comm.all_reduce_sum(m.loss)
        for l in reversed(range(self.L)):
            m.layer_backward(l, want_halo_grad=True)
            if l == 0:
                continue
            received = self.codesJ_recv[l] if self.codec_bits else self.recv_J[l]
            if sync:
                self._return_J(l)
                self._add_J(l, received)
                self.J_pending[l] = None
            else:
                if self.J_pending[l] is not None:
                    self._add_J(l, self.J_pending[l])
                self._return_J(l)
                self.J_pending[l] = tuple(t.clone() for t in received) if self.codec_bits else received.clone()
        for l in range(self.L):
            self.comm.all_reduce_sum(m.dW[l])
        self.epoch_index += 1

    def check_errors(self):
        self.model.check_errors()
