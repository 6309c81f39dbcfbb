"""Thin Python binding of libgnn (include/gnn.h): argument marshalling only.

Every function here has the name of a C entry point without the ``gnn_`` prefix
and forwards torch tensors as raw device pointers plus the current CUDA stream.
All computation happens in the library's CUDA kernels; if ``libgnn.so`` cannot be
loaded the import fails loudly (there is no fallback).

Matrix arguments are 2-D CUDA tensors whose last dimension is contiguous; the
leading dimension is ``tensor.stride(0)`` and the logical width is
``tensor.shape[1]``, so a padded buffer is passed as a column slice
(``buf[:, :f]``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgnn.so")

GNN_OK, GNN_EINVAL, GNN_ENOMEM, GNN_ECUDA, GNN_EUNSUPPORTED, GNN_EINDEX, GNN_ETIMEOUT = range(7)
GNN_F32, GNN_BF16 = 0, 1
GNN_AGG_GCN_SYM, GNN_AGG_SAGE_MEAN, GNN_AGG_GAT = 0, 1, 2

EXPORTS = (
    "gnn_graph_create", "gnn_graph_destroy", "gnn_halo_pull", "gnn_halo_push", "gnn_sage_half_offset",
    "gnn_layer_forward", "gnn_layer_backward", "gnn_softmax_ce", "gnn_get_error", "gnn_graph_sizes",
    "gnn_graph_copy_transpose", "gnn_status_string", "gnn_last_cuda_error", "gnn_halo_push_quantized",
    "gnn_halo_pull_quantized", "gnn_softmax_ce_partial", "gnn_halo_grad_send", "gnn_halo_grad_recv",
    "gnn_layer_forward_narrow", "gnn_layer_backward_narrow", "gnn_profile_enable", "gnn_profile_read", "gnn_launch_count",
    "gnn_aggregate_forward_noalloc", "gnn_debug_expire_next_wait", "gnn_gather_rows", "gnn_scatter_add_rows",
    "gnn_gat_forward", "gnn_gat_backward", "gnn_quantize_rows", "gnn_dequantize_rows", "gnn_layer_backward_reordered",
)

PROF_KINDS = ("agg_fwd", "agg_bwd", "upd_fwd", "upd_bwd", "pull", "push")


class GnnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {_lib().gnn_status_string(status).decode()} (status {status})"
        if status in (GNN_ECUDA, GNN_ENOMEM):
            msg += f": {last_cuda_error()}"
        super().__init__(msg)


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libgnn.so not built at {LIB_PATH}; run sparse_aggregation_dense_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.gnn_graph_create.argtypes = [vp, vp, i64, i64, i64, vp, i32, vp, ctypes.POINTER(vp)]
        L.gnn_graph_destroy.argtypes = [vp]
        L.gnn_halo_pull.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i32, vp]
        L.gnn_halo_push.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i32, vp]
        L.gnn_halo_push_quantized.argtypes = [vp, vp, i64, i64, vp, vp, i64, vp, i64, i32, ctypes.c_uint64, i32, vp]
        L.gnn_halo_pull_quantized.argtypes = [vp, vp, i64, vp, i64, i32, vp, vp, i64, i64, i32, vp]
        L.gnn_sage_half_offset.argtypes = [i64, i32]
        L.gnn_sage_half_offset.restype = i64
        L.gnn_layer_forward.argtypes = [vp, vp, i64, i64, vp, i64, i32, vp, i64, vp, i64, i32, vp]
        L.gnn_layer_backward.argtypes = [vp, vp, i64, vp, i64, vp, i64, vp, i64, i64, i32, vp, vp, i64, vp, i64, i32,
                                         i32, i32, vp]
        L.gnn_layer_backward_reordered.argtypes = [vp, vp, i64, vp, i64, vp, i64, vp, i64, i64, i32, vp, vp, i64, vp,
                                                   i64, i32, i32, i32, vp]
        L.gnn_softmax_ce.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, vp, i32, i32, vp]
        L.gnn_layer_forward_narrow.argtypes = [vp, vp, i64, i64, vp, i64, i32, vp, i64, vp, i64, i32, vp]
        L.gnn_layer_backward_narrow.argtypes = [vp, vp, i64, vp, i64, vp, i64, vp, i64, i64, i32, vp, vp, i64, vp,
                                                i64, i32, vp]
        L.gnn_softmax_ce_partial.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, vp, i64, i32, i32, vp]
        L.gnn_halo_grad_send.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i32, vp]
        L.gnn_halo_grad_recv.argtypes = [vp, vp, i64, i64, vp, vp, i64, i64, i32, vp]
        L.gnn_get_error.argtypes = [vp]
        L.gnn_graph_sizes.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.gnn_graph_copy_transpose.argtypes = [vp, vp, vp, vp, vp]
        L.gnn_profile_enable.argtypes = [vp, i32]
        L.gnn_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
        L.gnn_aggregate_forward_noalloc.argtypes = [vp, vp, i64, i64, vp, i64, i32, vp]
        L.gnn_debug_expire_next_wait.argtypes = [i64]
        L.gnn_gat_forward.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, vp, i64, vp, vp, vp, i64, i32, vp]
        L.gnn_gat_backward.argtypes = [vp, vp, i64, vp, i64, vp, i64, i64, vp, vp, vp, i64, i32, vp, i64, vp, vp, vp,
                                       vp, vp, vp, i64, vp, i64, i32, i32, vp]
        L.gnn_gather_rows.argtypes = [vp, i64, i64, vp, i64, vp, i64, i64, i32, vp, vp]
        L.gnn_quantize_rows.argtypes = [vp, i64, i64, i64, vp, i32, ctypes.c_uint64, vp, i64, vp, i32, vp]
        L.gnn_dequantize_rows.argtypes = [vp, i64, vp, i64, i64, i32, vp, vp, i64, i64, i32, i32, vp, vp]
        L.gnn_scatter_add_rows.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i32, vp, vp]
        L.gnn_launch_count.argtypes = []
        L.gnn_launch_count.restype = i64
        L.gnn_status_string.argtypes = [i32]
        L.gnn_last_cuda_error.argtypes = []
        L.gnn_last_cuda_error.restype = ctypes.c_char_p
        L.gnn_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name not in ("gnn_sage_half_offset", "gnn_status_string", "gnn_last_cuda_error", "gnn_launch_count"):
                getattr(L, name).restype = i32
        _L = L
    return _L


def _check(status: int, what: str):
    if status != GNN_OK:
        raise GnnError(status, what)


def _need(cond: bool, what: str, why: str):
    """Host-side check of what the C ABI cannot see (buffer rows, widths and
    dtypes against the graph): a failure is reported like the library's own
    GNN_EINVAL, before any device work is issued."""
    if not cond:
        raise GnnError(GNN_EINVAL, f"{what} ({why})")


def _rows(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.shape[0])


def _width(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.shape[1])


def _numel(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.numel())


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GNN_F32
    if t.dtype == torch.bfloat16:
        return GNN_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _mat(t: torch.Tensor) -> Tuple[int, int]:
    """(ld, f) of a 2-D tensor with a contiguous last dimension."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("expected a 2-D tensor with contiguous rows")
    return max(t.stride(0), t.shape[1]), t.shape[1]


def agg_code(agg: str) -> int:
    return {"gcn": GNN_AGG_GCN_SYM, "sage": GNN_AGG_SAGE_MEAN, "gat": GNN_AGG_GAT}[agg]


def _k(g, f_in: int) -> int:
    """Rows of W: the update's input width (twice f_in for the GraphSAGE concat)."""
    return 2 * f_in if g.agg == "sage" else f_in


def _z_width(g, f_in: int, dtype: torch.dtype) -> int:
    """Columns the aggregation writes: f_in, or both GraphSAGE halves (the mean
    starting at its 16-byte aligned offset)."""
    return 2 * sage_half_offset(f_in, dtype) if g.agg == "sage" else f_in


def _weights(what: str, W: torch.Tensor, K: int, f_out: int):
    _need(W.dtype == torch.float32 and W.is_contiguous() and tuple(W.shape) == (K, f_out), what,
          f"weights must be a contiguous float32 ({K} x {f_out}) matrix")


class Graph:
    """Owner of a ``gnn_graph*``; freed by :func:`graph_destroy` or on collection."""

    def __init__(self, handle: int, n_local: int, n_halo: int, nnz: int, agg: str):
        self.handle = handle
        self.n_local, self.n_halo, self.nnz, self.agg = n_local, n_halo, nnz, agg

    @property
    def n_total(self) -> int:
        return self.n_local + self.n_halo

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                _lib().gnn_graph_destroy(ctypes.c_void_p(self.handle))
            except Exception:
                pass
            self.handle = None


def graph_create(rowptr: torch.Tensor, colidx: torch.Tensor, n_local: int, n_halo: int,
                 deg: Optional[torch.Tensor] = None, agg: str = "gcn") -> Graph:
    what = "gnn_graph_create"
    _need(rowptr.dtype == torch.int32 and colidx.dtype == torch.int32, what, "rowptr and colidx must be int32")
    _need(rowptr.numel() == n_local + 1, what, "rowptr must hold n_local + 1 entries")
    if deg is not None:
        _need(deg.dtype == torch.float32 and deg.numel() == n_local + n_halo, what,
              "deg must be float32 with n_local + n_halo entries")
    out = ctypes.c_void_p()
    nnz = colidx.numel()
    _check(_lib().gnn_graph_create(_ptr(rowptr), _ptr(colidx) if nnz else None, n_local, n_halo, nnz, _ptr(deg),
                                   agg_code(agg), ctypes.c_void_p(_stream()), ctypes.byref(out)), "gnn_graph_create")
    return Graph(out.value, n_local, n_halo, nnz, agg)


def graph_destroy(g: Graph):
    if g.handle:
        h, g.handle = g.handle, None
        _check(_lib().gnn_graph_destroy(ctypes.c_void_p(h)), "gnn_graph_destroy")


def get_error(g: Graph) -> int:
    """Synchronise; return (and clear) the graph's device error status."""
    return int(_lib().gnn_get_error(ctypes.c_void_p(g.handle)))


def last_cuda_error() -> str:
    """Text of the last CUDA runtime error behind a GNN_ECUDA status."""
    return _lib().gnn_last_cuda_error().decode()


def graph_copy_transpose(g: Graph):
    """Copies of the transpose (rowptrT, colidxT, permT) as int32 CUDA tensors."""
    rT = torch.empty(g.n_total + 1, dtype=torch.int32, device="cuda")
    cT = torch.empty(max(g.nnz, 1), dtype=torch.int32, device="cuda")
    pT = torch.empty(max(g.nnz, 1), dtype=torch.int32, device="cuda")
    _check(_lib().gnn_graph_copy_transpose(ctypes.c_void_p(g.handle), _ptr(rT), _ptr(cT), _ptr(pT),
                                           ctypes.c_void_p(_stream())), "gnn_graph_copy_transpose")
    return rT, cT[:g.nnz], pT[:g.nnz]


def profile_enable(g: Graph, on: bool = True):
    _check(_lib().gnn_profile_enable(ctypes.c_void_p(g.handle), int(on)), "gnn_profile_enable")


def profile_read(g: Graph) -> dict:
    """{kind: (total_ms, groups)} for the groups recorded since the last read."""
    ms = (ctypes.c_double * len(PROF_KINDS))()
    n = (ctypes.c_int64 * len(PROF_KINDS))()
    _check(_lib().gnn_profile_read(ctypes.c_void_p(g.handle), ms, n), "gnn_profile_read")
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(PROF_KINDS)}


def aggregate_forward_noalloc(g: Graph, H: torch.Tensor, Z: torch.Tensor):
    """Z of layer_forward for H, computed without any device allocation."""
    ld_h, f = _mat(H)
    ld_z, _ = _mat(Z)
    what = "gnn_aggregate_forward_noalloc"
    _need(H.dtype == Z.dtype, what, "H and Z must share a dtype")
    _need(_rows(H) >= g.n_total and _rows(Z) >= g.n_local, what, "H needs n_local + n_halo rows, Z n_local rows")
    _need(_width(Z) >= _z_width(g, f, H.dtype), what, "Z is narrower than the aggregation output")
    _check(_lib().gnn_aggregate_forward_noalloc(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f, _ptr(Z), ld_z,
                                                _dtype(H), ctypes.c_void_p(_stream())),
           "gnn_aggregate_forward_noalloc")


def debug_expire_next_wait(wait_ns: int):
    """Failure-detection test hook: the next aggregation's first batch is never issued, so its bounded wait runs
    out after wait_ns and the call's graph reports GNN_ETIMEOUT (nothing faults)."""
    _check(_lib().gnn_debug_expire_next_wait(int(wait_ns)), "gnn_debug_expire_next_wait")


def _vec(what: str, t: torch.Tensor, n: int, name: str):
    _need(t.dtype == torch.float32 and t.is_contiguous() and t.numel() == n, what,
          f"{name} must be a contiguous float32 vector of {n} values")


def gat_forward(g: Graph, H: torch.Tensor, W: torch.Tensor, a_src: torch.Tensor, a_dst: torch.Tensor, relu: bool,
                T: torch.Tensor, scores: torch.Tensor, alpha: torch.Tensor, H_out: torch.Tensor):
    """Graph attention layer: T = H W (every row), scores, alpha (per entry), H_out = act(sum alpha T)."""
    ld_h, f_in = _mat(H)
    ld_t, _ = _mat(T)
    ld_o, f_out = _mat(H_out)
    what = "gnn_gat_forward"
    _need(g.agg == "gat", what, "the graph was not created for attention")
    _weights(what, W, f_in, f_out)
    _vec(what, a_src, f_out, "a_src")
    _vec(what, a_dst, f_out, "a_dst")
    _vec(what, scores, g.n_total + g.n_local, "scores")
    _vec(what, alpha, max(g.nnz, 0), "alpha")
    _need(H.dtype == T.dtype == H_out.dtype, what, "H, T and H_out share a dtype")
    _need(_rows(H) >= g.n_total and _rows(T) >= g.n_total and _rows(H_out) >= g.n_local and _width(T) >= f_out, what,
          "H and T need n_local + n_halo rows, H_out n_local rows")
    _check(_lib().gnn_gat_forward(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f_in, _ptr(W), _ptr(a_src), _ptr(a_dst),
                                  f_out, int(relu), _ptr(T), ld_t, _ptr(scores), _ptr(alpha), _ptr(H_out), ld_o,
                                  _dtype(H), ctypes.c_void_p(_stream())), what)


def gat_backward(g: Graph, G: torch.Tensor, H_out: torch.Tensor, H: torch.Tensor, W: torch.Tensor,
                 a_src: torch.Tensor, a_dst: torch.Tensor, relu: bool, T: torch.Tensor, scores: torch.Tensor,
                 alpha: torch.Tensor, dW: torch.Tensor, da_src: torch.Tensor, da_dst: torch.Tensor, dT: torch.Tensor,
                 dH: Optional[torch.Tensor] = None):
    """Backward of gat_forward: dW, da_src, da_dst, the work dT, and dH (every row) unless dH is None."""
    ld_g, f_out = _mat(G)
    ld_o, _ = _mat(H_out)
    ld_h, f_in = _mat(H)
    ld_t, _ = _mat(T)
    ld_dt, _ = _mat(dT)
    ld_dh = _mat(dH)[0] if dH is not None else 0
    what = "gnn_gat_backward"
    _need(g.agg == "gat", what, "the graph was not created for attention")
    _weights(what, W, f_in, f_out)
    _weights(what, dW, f_in, f_out)
    for name, t in (("a_src", a_src), ("a_dst", a_dst), ("da_src", da_src), ("da_dst", da_dst)):
        _vec(what, t, f_out, name)
    _vec(what, scores, g.n_total + g.n_local, "scores")
    _vec(what, alpha, max(g.nnz, 0), "alpha")
    _need(H_out.dtype == H.dtype == T.dtype, what, "H_out, H and T share the activations' dtype")
    _need(all(t is None or t.dtype == G.dtype for t in (dT, dH)), what, "G, dT and dH share the gradients' dtype")
    _need(not (H.dtype == torch.float32 and G.dtype != torch.float32), what, "fp32 activations take fp32 gradients")
    _need(_rows(G) >= g.n_local and _rows(H_out) >= g.n_local and _rows(H) >= g.n_total and _rows(T) >= g.n_total
          and _rows(dT) >= g.n_total and _width(dT) >= f_out, what, "row counts of G, H_out, H, T and dT")
    _need(dH is None or (_rows(dH) >= g.n_total and _width(dH) >= f_in), what,
          "dH needs n_local + n_halo rows of f_in columns")
    _check(_lib().gnn_gat_backward(ctypes.c_void_p(g.handle), _ptr(G), ld_g, _ptr(H_out), ld_o, _ptr(H), ld_h, f_in,
                                   _ptr(W), _ptr(a_src), _ptr(a_dst), f_out, int(relu), _ptr(T), ld_t, _ptr(scores),
                                   _ptr(alpha), _ptr(dW), _ptr(da_src), _ptr(da_dst), _ptr(dT), ld_dt, _ptr(dH), ld_dh,
                                   _dtype(H), _dtype(G), ctypes.c_void_p(_stream())), what)


def quantize_rows(X: torch.Tensor, keys: torch.Tensor, codes: torch.Tensor, scale_zero: torch.Tensor, bits: int,
                  seed: int):
    """Rows of X's view as b-bit codes (codes row i, scale_zero[i]); draws keyed by keys[i] and seed."""
    ld_x, f = _mat(X)
    what = "gnn_quantize_rows"
    _codec_args(what, codes, scale_zero, keys, f, bits)
    _need(_numel(keys) >= _rows(X) and codes.shape[0] >= _rows(X), what, "a key and a code row per row of X")
    _check(_lib().gnn_quantize_rows(_ptr(X), ld_x, _rows(X), f, _ptr(keys), int(bits),
                                    ctypes.c_uint64(seed & (2**64 - 1)), _ptr(codes), codes.stride(0),
                                    _ptr(scale_zero), _dtype(X), ctypes.c_void_p(_stream())), what)


def dequantize_rows(codes: torch.Tensor, scale_zero: torch.Tensor, bits: int, dst: torch.Tensor,
                    ids: Optional[torch.Tensor] = None, add: bool = False, n: Optional[int] = None,
                    err: Optional[torch.Tensor] = None):
    """dst[ids[i]] (+)= code * scale + zero of codes row i, over the columns of dst's view (ids None: row i)."""
    ld_d, f = _mat(dst)
    n = codes.shape[0] if n is None else n
    what = "gnn_dequantize_rows"
    _codec_args(what, codes, scale_zero, ids if ids is not None else torch.zeros(0, dtype=torch.int64), f, bits)
    _need(ids is None or _numel(ids) >= n, what, "an id per code row")
    _need(err is None or err.dtype == torch.int32, what, "int32 error word")
    _check(_lib().gnn_dequantize_rows(_ptr(codes), codes.stride(0), _ptr(scale_zero), n, f, int(bits), _ptr(ids),
                                      _ptr(dst), ld_d, _rows(dst), int(add), _dtype(dst), _ptr(err),
                                      ctypes.c_void_p(_stream())), what)


def gather_rows(src: torch.Tensor, ids: torch.Tensor, dst: torch.Tensor, err: Optional[torch.Tensor] = None):
    """dst[i] = src[ids[i]] over the columns of dst's view (a bit-exact row copy)."""
    ld_s, _ = _mat(src)
    ld_d, f = _mat(dst)
    what = "gnn_gather_rows"
    _need(src.dtype == dst.dtype and ids.dtype == torch.int64, what, "src and dst share a dtype; int64 ids")
    _need(_numel(ids) >= _rows(dst) and _width(src) >= f, what, "an id per dst row; src as wide as dst's view")
    _need(err is None or err.dtype == torch.int32, what, "int32 error word")
    _check(_lib().gnn_gather_rows(_ptr(src), ld_s, _rows(src), _ptr(ids), _rows(dst), _ptr(dst), ld_d, f,
                                  _dtype(dst), _ptr(err), ctypes.c_void_p(_stream())), what)


def scatter_add_rows(src: torch.Tensor, ids: torch.Tensor, dst: torch.Tensor, err: Optional[torch.Tensor] = None):
    """dst[ids[i]] += src[i] over the columns of src's view (fp32 sums; ids distinct)."""
    ld_s, f = _mat(src)
    ld_d, _ = _mat(dst)
    what = "gnn_scatter_add_rows"
    _need(src.dtype == dst.dtype and ids.dtype == torch.int64, what, "src and dst share a dtype; int64 ids")
    _need(_numel(ids) >= _rows(src) and _width(dst) >= f, what, "an id per src row; dst as wide as src's view")
    _need(err is None or err.dtype == torch.int32, what, "int32 error word")
    _check(_lib().gnn_scatter_add_rows(_ptr(src), ld_s, _ptr(ids), _rows(src), _ptr(dst), ld_d, _rows(dst), f,
                                       _dtype(src), _ptr(err), ctypes.c_void_p(_stream())), what)


def launch_count() -> int:
    """Kernels launched by libgnn in this process so far."""
    return int(_lib().gnn_launch_count())


def sage_half_offset(f: int, dtype: torch.dtype) -> int:
    return int(_lib().gnn_sage_half_offset(f, GNN_BF16 if dtype == torch.bfloat16 else GNN_F32))


def halo_pull(g: Graph, table: torch.Tensor, halo_ids: torch.Tensor, H: torch.Tensor):
    """H[n_local + i] = table[halo_ids[i]] over the columns of H's view."""
    ld_t, _ = _mat(table)
    ld_h, f = _mat(H)
    what = "gnn_halo_pull"
    _need(halo_ids.dtype == torch.int64 and table.dtype == H.dtype, what, "int64 ids; table and H share a dtype")
    _need(_numel(halo_ids) >= g.n_halo and _rows(H) >= g.n_total, what,
          "n_halo ids and n_local + n_halo rows of H")
    _need(_width(table) >= f, what, "table rows narrower than H's view")
    _check(_lib().gnn_halo_pull(ctypes.c_void_p(g.handle), _ptr(table), ld_t, table.shape[0], _ptr(halo_ids),
                                _ptr(H), ld_h, f, _dtype(H), ctypes.c_void_p(_stream())), "gnn_halo_pull")


def halo_push(g: Graph, H: torch.Tensor, local_ids: torch.Tensor, table: torch.Tensor):
    """table[local_ids[v]] = H[v] over the columns of H's view (v < n_local)."""
    ld_t, _ = _mat(table)
    ld_h, f = _mat(H)
    what = "gnn_halo_push"
    _need(local_ids.dtype == torch.int64 and table.dtype == H.dtype, what, "int64 ids; table and H share a dtype")
    _need(_numel(local_ids) >= g.n_local and _rows(H) >= g.n_local, what, "n_local ids and n_local rows of H")
    _need(_width(table) >= f, what, "table rows narrower than H's view")
    _check(_lib().gnn_halo_push(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f, _ptr(local_ids), _ptr(table), ld_t,
                                table.shape[0], _dtype(H), ctypes.c_void_p(_stream())), "gnn_halo_push")


def codec_row_bytes(f: int, bits: int) -> int:
    """Bytes of one row of f packed b-bit codes, padded to 16."""
    return (f * bits + 127) // 128 * 16


def _codec_args(what: str, codes: torch.Tensor, scale_zero: torch.Tensor, ids: torch.Tensor, f: int, bits: int):
    _need(ids.dtype == torch.int64 and codes.dtype == torch.uint8 and scale_zero.dtype == torch.float32, what,
          "int64 ids, uint8 codes, float32 scale / zero point")
    _need(codes.dim() == 2 and codes.stride(1) == 1 and scale_zero.is_contiguous(), what,
          "codes with contiguous rows, contiguous scale / zero point")
    _need(scale_zero.dim() == 2 and scale_zero.shape[1] == 2 and scale_zero.shape[0] >= codes.shape[0], what,
          "scale_zero must be (n_table x 2)")
    if bits in (1, 2, 4, 8):  # other widths are the library's to reject
        _need(codes.shape[1] >= codec_row_bytes(f, bits), what, "code rows shorter than one packed row")


def halo_push_quantized(g: Graph, H: torch.Tensor, local_ids: torch.Tensor, codes: torch.Tensor,
                        scale_zero: torch.Tensor, bits: int, seed: int):
    """Quantise the local rows of H's view (b-bit stochastic rounding, per-row scale and zero point) into
    codes[local_ids[v]] and scale_zero[local_ids[v]] (codes: uint8 n_table x ld_codes, scale_zero: float32
    n_table x 2)."""
    ld_h, f = _mat(H)
    what = "gnn_halo_push_quantized"
    _codec_args(what, codes, scale_zero, local_ids, f, bits)
    _need(_numel(local_ids) >= g.n_local and _rows(H) >= g.n_local, what, "n_local ids and n_local rows of H")
    _check(_lib().gnn_halo_push_quantized(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f, _ptr(local_ids), _ptr(codes),
                                          codes.stride(0), _ptr(scale_zero), codes.shape[0], int(bits),
                                          ctypes.c_uint64(seed & (2**64 - 1)), _dtype(H), ctypes.c_void_p(_stream())),
           "gnn_halo_push_quantized")


def halo_pull_quantized(g: Graph, codes: torch.Tensor, scale_zero: torch.Tensor, bits: int, halo_ids: torch.Tensor,
                        H: torch.Tensor):
    """H[n_local + i] = dequantised codes[halo_ids[i]] over the columns of H's view."""
    ld_h, f = _mat(H)
    what = "gnn_halo_pull_quantized"
    _codec_args(what, codes, scale_zero, halo_ids, f, bits)
    _need(_numel(halo_ids) >= g.n_halo and _rows(H) >= g.n_total, what, "n_halo ids and n_local + n_halo rows of H")
    _check(_lib().gnn_halo_pull_quantized(ctypes.c_void_p(g.handle), _ptr(codes), codes.stride(0), _ptr(scale_zero),
                                          codes.shape[0], int(bits), _ptr(halo_ids), _ptr(H), ld_h, f, _dtype(H),
                                          ctypes.c_void_p(_stream())), "gnn_halo_pull_quantized")


def layer_forward_narrow(g: Graph, H: torch.Tensor, W: torch.Tensor, relu: bool, T: torch.Tensor,
                         H_out: torch.Tensor):
    """T = H W (every row), H_out = act(A_block T): the GCN layer with the multiplication first."""
    ld_h, f_in = _mat(H)
    ld_t, _ = _mat(T)
    ld_o, f_out = _mat(H_out)
    what = "gnn_layer_forward_narrow"
    _weights(what, W, f_in, f_out)
    _need(H.dtype == T.dtype == H_out.dtype, what, "H, T and H_out share a dtype")
    _need(_rows(H) >= g.n_total and _rows(T) >= g.n_total and _rows(H_out) >= g.n_local, what,
          "H and T need n_local + n_halo rows, H_out n_local rows")
    _need(_width(T) >= f_out, what, "T narrower than H_out")
    _check(_lib().gnn_layer_forward_narrow(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f_in, _ptr(W), f_out, int(relu),
                                           _ptr(T), ld_t, _ptr(H_out), ld_o, _dtype(H), ctypes.c_void_p(_stream())),
           "gnn_layer_forward_narrow")


def layer_backward_narrow(g: Graph, G: torch.Tensor, H_out: torch.Tensor, H: torch.Tensor, W: torch.Tensor,
                          relu: bool, dW: torch.Tensor, P: torch.Tensor, dH: Optional[torch.Tensor] = None):
    """P = A_block^T dY (every row), dW = H^T P, dH = P W^T (every row; skipped when dH is None)."""
    ld_g, f_out = _mat(G)
    ld_o, _ = _mat(H_out)
    ld_h, f_in = _mat(H)
    ld_p, _ = _mat(P)
    ld_dh = _mat(dH)[0] if dH is not None else 0
    what = "gnn_layer_backward_narrow"
    _weights(what, W, f_in, f_out)
    _weights(what, dW, f_in, f_out)
    _need(all(t is None or t.dtype == G.dtype for t in (H_out, H, P, dH)), what, "activations share one dtype")
    _need(_rows(G) >= g.n_local and _rows(H_out) >= g.n_local, what, "G and H_out need n_local rows")
    _need(_rows(H) >= g.n_total and _rows(P) >= g.n_total and _width(P) >= f_out, what,
          "H and P need n_local + n_halo rows, P f_out columns")
    _need(dH is None or (_rows(dH) >= g.n_total and _width(dH) >= f_in), what,
          "dH needs n_local + n_halo rows of f_in columns")
    _check(_lib().gnn_layer_backward_narrow(ctypes.c_void_p(g.handle), _ptr(G), ld_g, _ptr(H_out), ld_o, _ptr(H),
                                            ld_h, _ptr(W), f_in, f_out, int(relu), _ptr(dW), _ptr(P), ld_p, _ptr(dH),
                                            ld_dh, _dtype(G), ctypes.c_void_p(_stream())), "gnn_layer_backward_narrow")


def layer_forward(g: Graph, H: torch.Tensor, W: torch.Tensor, relu: bool, Z: torch.Tensor, H_out: torch.Tensor):
    """Z = A_block H (or the SAGE concat), H_out = act(Z W).  Widths from the views of H and H_out."""
    ld_h, f_in = _mat(H)
    ld_z, _ = _mat(Z)
    ld_o, f_out = _mat(H_out)
    what = "gnn_layer_forward"
    _weights(what, W, _k(g, f_in), f_out)
    _need(H.dtype == Z.dtype == H_out.dtype, what, "H, Z and H_out share a dtype")
    _need(_rows(H) >= g.n_total and _rows(Z) >= g.n_local and _rows(H_out) >= g.n_local, what,
          "H needs n_local + n_halo rows, Z and H_out n_local rows")
    _need(_width(Z) >= _z_width(g, f_in, H.dtype), what, "Z is narrower than the aggregation output")
    _check(_lib().gnn_layer_forward(ctypes.c_void_p(g.handle), _ptr(H), ld_h, f_in, _ptr(W), f_out, int(relu),
                                    _ptr(Z), ld_z, _ptr(H_out), ld_o, _dtype(H), ctypes.c_void_p(_stream())),
           "gnn_layer_forward")


def layer_backward(g: Graph, G: torch.Tensor, H_out: torch.Tensor, Z: torch.Tensor, W: torch.Tensor, relu: bool,
                   dW: torch.Tensor, f_in: int, dZ: Optional[torch.Tensor] = None, dH: Optional[torch.Tensor] = None,
                   want_halo_grad: bool = False):
    """dW = Z^T dY; with dH: dZ = dY W^T and dH = A_block^T dZ (halo rows too if want_halo_grad).

    The activations (H_out, Z) share one dtype, the gradients (G, dZ, dH) another:
    fp32 activations take fp32 gradients, bf16 activations bf16 or fp32 gradients."""
    ld_g, f_out = _mat(G)
    ld_o, _ = _mat(H_out)
    ld_z, _ = _mat(Z)
    ld_dz = _mat(dZ)[0] if dZ is not None else 0
    ld_dh = _mat(dH)[0] if dH is not None else 0
    what = "gnn_layer_backward"
    K, Kp = _k(g, f_in), _z_width(g, f_in, Z.dtype)
    _weights(what, W, K, f_out)
    _weights(what, dW, K, f_out)
    _need(H_out.dtype == Z.dtype, what, "H_out and Z share the activations' dtype")
    _need(all(t is None or t.dtype == G.dtype for t in (dZ, dH)), what, "G, dZ and dH share the gradients' dtype")
    _need(not (Z.dtype == torch.float32 and G.dtype != torch.float32), what,
          "fp32 activations take fp32 gradients")
    _need(_rows(G) >= g.n_local and _rows(H_out) >= g.n_local and _rows(Z) >= g.n_local, what,
          "G, H_out and Z need n_local rows")
    _need(_width(Z) >= Kp, what, "Z is narrower than the aggregation output")
    _need(dZ is None or (_rows(dZ) >= g.n_local and _width(dZ) >= Kp), what, "dZ needs n_local rows as wide as Z")
    _need(dH is None or (_rows(dH) >= (g.n_total if want_halo_grad else g.n_local) and _width(dH) >= f_in), what,
          "dH needs n_local rows (n_local + n_halo with the halo gradient) of f_in columns")
    _check(_lib().gnn_layer_backward(ctypes.c_void_p(g.handle), _ptr(G), ld_g, _ptr(H_out), ld_o, _ptr(Z), ld_z,
                                     _ptr(W), f_in, f_out, int(relu), _ptr(dW), _ptr(dZ), ld_dz, _ptr(dH), ld_dh,
                                     int(want_halo_grad), _dtype(Z), _dtype(G), ctypes.c_void_p(_stream())),
           "gnn_layer_backward")


def layer_backward_reordered(g: Graph, G: torch.Tensor, H_out: torch.Tensor, Z: torch.Tensor, W: torch.Tensor,
                             relu: bool, dW: torch.Tensor, P: torch.Tensor, dH: torch.Tensor,
                             want_halo_grad: bool = True):
    """GCN layer backward in the other product order: dW = Z^T dY, P = A_block^T dY (bf16), dH = P W^T (fp32).
    bf16 activations (H_out, Z) with fp32 gradients (G, dH) only; halo rows too if want_halo_grad."""
    ld_g, f_out = _mat(G)
    ld_o, _ = _mat(H_out)
    ld_z, f_in = _mat(Z)
    ld_p, _ = _mat(P)
    ld_dh, _ = _mat(dH)
    what = "gnn_layer_backward_reordered"
    rows = g.n_total if want_halo_grad else g.n_local
    _weights(what, W, f_in, f_out)
    _weights(what, dW, f_in, f_out)
    _need(Z.dtype == H_out.dtype == P.dtype == torch.bfloat16 and G.dtype == dH.dtype == torch.float32, what,
          "bf16 activations and P, fp32 gradients")
    _need(_rows(G) >= g.n_local and _rows(H_out) >= g.n_local and _rows(Z) >= g.n_local, what,
          "G, H_out and Z need n_local rows")
    _need(_rows(P) >= rows and _width(P) >= f_out and _rows(dH) >= rows and _width(dH) >= f_in, what,
          "P and dH need a row per output row (halo rows too with the halo gradient)")
    _check(_lib().gnn_layer_backward_reordered(ctypes.c_void_p(g.handle), _ptr(G), ld_g, _ptr(H_out), ld_o, _ptr(Z),
                                               ld_z, _ptr(W), f_in, f_out, int(relu), _ptr(dW), _ptr(P), ld_p,
                                               _ptr(dH), ld_dh, int(want_halo_grad), _dtype(Z), _dtype(G),
                                               ctypes.c_void_p(_stream())), what)


def _softmax_args(what: str, logits, labels, G, row_loss, loss):
    n, C = int(logits.shape[0]), int(logits.shape[1])
    _need(labels.dtype == torch.int32 and row_loss.dtype == torch.float32 and loss.dtype == torch.float32, what,
          "int32 labels, float32 row_loss and loss")
    _need(G.dtype in (torch.float32, torch.bfloat16) and _rows(G) >= n and _width(G) >= C, what,
          "G (fp32 or bf16) shaped like the logits")
    _need(_numel(labels) >= n and _numel(row_loss) >= n and _numel(loss) >= 1, what,
          "a label and a row_loss entry per row, one loss")


def softmax_ce(logits: torch.Tensor, labels: torch.Tensor, G: torch.Tensor, row_loss: torch.Tensor,
               loss: torch.Tensor):
    """Mean softmax cross-entropy of the rows of logits; G (in its own dtype) = (softmax - onehot) / n."""
    ld, C = _mat(logits)
    ld_g, _ = _mat(G)
    _softmax_args("gnn_softmax_ce", logits, labels, G, row_loss, loss)
    _check(_lib().gnn_softmax_ce(_ptr(logits), ld, logits.shape[0], C, _ptr(labels), _ptr(G), ld_g, _ptr(row_loss),
                                 _ptr(loss), _dtype(logits), _dtype(G), ctypes.c_void_p(_stream())), "gnn_softmax_ce")


def softmax_ce_partial(logits: torch.Tensor, labels: torch.Tensor, G: torch.Tensor, row_loss: torch.Tensor,
                       loss: torch.Tensor, n_mean: int):
    """softmax_ce whose mean (and gradient) divides by n_mean >= the rows of logits."""
    ld, C = _mat(logits)
    ld_g, _ = _mat(G)
    _softmax_args("gnn_softmax_ce_partial", logits, labels, G, row_loss, loss)
    _check(_lib().gnn_softmax_ce_partial(_ptr(logits), ld, logits.shape[0], C, _ptr(labels), _ptr(G), ld_g,
                                         _ptr(row_loss), _ptr(loss), int(n_mean), _dtype(logits), _dtype(G),
                                         ctypes.c_void_p(_stream())), "gnn_softmax_ce_partial")


def halo_grad_send(g: Graph, dH: torch.Tensor, halo_ids: torch.Tensor, gtable: torch.Tensor):
    """gtable[halo_ids[i]] += dH[n_local + i] over the columns of dH's view (gtable: float32)."""
    ld_h, f = _mat(dH)
    ld_t, _ = _mat(gtable)
    what = "gnn_halo_grad_send"
    _need(halo_ids.dtype == torch.int64 and gtable.dtype == torch.float32, what, "int64 ids, float32 gradient table")
    _need(_numel(halo_ids) >= g.n_halo and _rows(dH) >= g.n_total and _width(gtable) >= f, what,
          "n_halo ids, n_local + n_halo rows of dH, table rows as wide as dH's view")
    _check(_lib().gnn_halo_grad_send(ctypes.c_void_p(g.handle), _ptr(dH), ld_h, f, _ptr(halo_ids), _ptr(gtable),
                                     ld_t, gtable.shape[0], _dtype(dH), ctypes.c_void_p(_stream())),
           "gnn_halo_grad_send")


def halo_grad_recv(g: Graph, gtable: torch.Tensor, local_ids: torch.Tensor, dH: torch.Tensor):
    """dH[v] += gtable[local_ids[v]] for the local rows, over the columns of dH's view."""
    ld_h, f = _mat(dH)
    ld_t, _ = _mat(gtable)
    what = "gnn_halo_grad_recv"
    _need(local_ids.dtype == torch.int64 and gtable.dtype == torch.float32, what, "int64 ids, float32 gradient table")
    _need(_numel(local_ids) >= g.n_local and _rows(dH) >= g.n_local and _width(gtable) >= f, what,
          "n_local ids, n_local rows of dH, table rows as wide as dH's view")
    _check(_lib().gnn_halo_grad_recv(ctypes.c_void_p(g.handle), _ptr(gtable), ld_t, gtable.shape[0],
                                     _ptr(local_ids), _ptr(dH), ld_h, f, _dtype(dH), ctypes.c_void_p(_stream())),
           "gnn_halo_grad_recv")
