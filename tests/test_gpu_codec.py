"""Parity of the low-bit halo codec (Sylvie page, Quantizer / Dequantizer)
through the C ABI with the oracle: codes, scales and zero points bit for bit,
dequantised rows bit for bit (after the same bf16 rounding), on the tiny
workloads for every bit width and on sampled rows of the full-size partition.
"""
import numpy as np
import pytest
import torch

import oracle
from synth.configs import TINY, WORKLOADS
from sparse_aggregation_dense_gb300 import gnn, padded
from tests._gpu import assert_ok, gen_matrix, to_device, torch_dtype, widen

pytestmark = pytest.mark.gpu

SEED = 0
_cache = {}


def problem(name, size):
    key = (name, size)
    if key not in _cache:
        w = (TINY if size == "tiny" else WORKLOADS)[name]
        part = w.make(SEED)
        deg = None if part.deg is None else torch.from_numpy(part.deg).cuda()
        g = gnn.graph_create(torch.from_numpy(part.rowptr).cuda(), torch.from_numpy(part.colidx).cuda(),
                             part.n_local, part.n_halo, deg, w.agg)
        _cache[key] = (w, part, g)
    return _cache[key]


def _values(host, dt, f):
    """fp32 values of a generator matrix (bf16 bits widened exactly)."""
    return widen(host, dt, f).astype(np.float32)


@pytest.mark.parametrize("name", ["er5k", "rmat16m", "sage2m"])
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_push_quantized_matches_oracle(name, bits):
    w, part, g = problem(name, "tiny")
    dt, f = w.dtype, w.widths[1]
    H_h = gen_matrix(part.n_local, f, dt, SEED, 300 + bits)
    H = to_device(H_h, dt, f)
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.full((part.n_table, ldc), 0xAB, dtype=torch.uint8, device="cuda")
    sz = torch.full((part.n_table, 2), -7.0, dtype=torch.float32, device="cuda")
    seed = 0x5EED + bits
    gnn.halo_push_quantized(g, H, torch.from_numpy(part.local_ids).cuda(), codes, sz, bits, seed)
    assert_ok(g)
    ref_c, ref_sz = oracle.quantize_rows(_values(H_h, dt, f), part.local_ids, bits, seed, ldc)
    got_c, got_sz = codes.cpu().numpy(), sz.cpu().numpy()
    np.testing.assert_array_equal(got_c[part.local_ids], ref_c)
    np.testing.assert_array_equal(got_sz[part.local_ids].view(np.uint32), ref_sz.view(np.uint32))
    other = np.setdiff1d(np.arange(part.n_table), part.local_ids)
    assert np.all(got_c[other] == 0xAB) and np.all(got_sz[other] == -7.0)


def _special_rows(n, f, rng):
    """Rows that reach every branch of the quantiser: magnitudes far below and
    above 1, integer rows (exact quotients), rows whose quotients are powers of
    two, constant rows (zero scale), two-valued rows, numerators just above
    zero, a range so small that the reciprocal of the scale is infinite, and
    rows holding an infinite value (infinite scale)."""
    H = np.empty((n, f), np.float32)
    for i in range(n):
        kind = i % 10
        x = rng.standard_normal(f)
        if kind == 0:
            x = x * 2.0 ** -70
        elif kind == 1:
            x = x * 2.0 ** 70
        elif kind == 2:
            x = x * 2.0 ** -58
        elif kind == 3:
            x = rng.integers(0, 256, f).astype(np.float64)
        elif kind == 4:
            x = 2.0 ** rng.integers(-3, 9, f)
            x[0] = 0.0
        elif kind == 5:
            x = np.full(f, 1.5)
        elif kind == 6:
            x = np.where(rng.random(f) < 0.5, -3.0, 5.0)
        elif kind == 7:  # values a hair above the minimum: tiny numerators
            x = np.abs(x)
            x[:3] = [0.0, 2.0 ** -70, 2.0 ** -64]
        elif kind == 8:  # range 2^-140 (subnormal): 1 / scale overflows
            x = np.where(rng.random(f) < 0.5, 0.0, 2.0 ** -140)
        else:  # an infinite value: the scale is infinite
            x[rng.integers(0, f)] = np.inf
        H[i] = x.astype(np.float32)
    return H


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_push_quantized_special_magnitudes(bits):
    w, part, g = problem("er5k", "tiny")
    f = w.widths[1]
    Hv = _special_rows(part.n_local, f, np.random.default_rng(bits))
    H = padded(part.n_local, f, torch.float32, "cuda")
    H.copy_(torch.from_numpy(Hv).cuda())
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.zeros((part.n_table, ldc), dtype=torch.uint8, device="cuda")
    sz = torch.zeros((part.n_table, 2), dtype=torch.float32, device="cuda")
    seed = 77 + bits
    gnn.halo_push_quantized(g, H, torch.from_numpy(part.local_ids).cuda(), codes, sz, bits, seed)
    assert_ok(g)
    ref_c, ref_sz = oracle.quantize_rows(Hv, part.local_ids, bits, seed, ldc)
    np.testing.assert_array_equal(codes.cpu().numpy()[part.local_ids], ref_c)
    np.testing.assert_array_equal(sz.cpu().numpy()[part.local_ids].view(np.uint32), ref_sz.view(np.uint32))


@pytest.mark.parametrize("name", ["er5k", "rmat16m", "powerlaw233k"])
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_pull_quantized_matches_oracle(name, bits):
    w, part, g = problem(name, "tiny")
    dt, f = w.dtype, w.widths[0]
    T_h = gen_matrix(part.n_table, f, dt, SEED, 400 + bits)
    ldc = gnn.codec_row_bytes(f, bits)
    c, s = oracle.quantize_rows(_values(T_h, dt, f), np.arange(part.n_table), bits, 99, ldc)
    H = padded(part.n_total, f, torch_dtype(dt), "cuda")
    gnn.halo_pull_quantized(g, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), bits,
                            torch.from_numpy(part.halo_ids).cuda(), H)
    assert_ok(g)
    ref = oracle.dequantize_rows(c[part.halo_ids], s[part.halo_ids], f, bits)
    got = H[part.n_local:].float().cpu().numpy()
    if dt == "bf16":
        ref = oracle.round_bf16(ref.astype(np.float64)).astype(np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    # local rows untouched (zero)
    assert float(H[:part.n_local].abs().max()) == 0.0


def test_round_trip_full_size_sampled():
    # the bench partition: push all 8.4M local rows at 1 bit, pull the 4.2M
    # halo rows back; sampled rows against the oracle
    w, part, g = problem("rmat16m", "full")
    f, bits, seed = w.widths[1], 1, 2024
    H = padded(part.n_local, f, torch.bfloat16, "cuda")
    H.copy_(torch.randn(part.n_local, f, device="cuda", generator=torch.Generator("cuda").manual_seed(3)))
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.zeros((part.n_table, ldc), dtype=torch.uint8, device="cuda")
    sz = torch.zeros((part.n_table, 2), dtype=torch.float32, device="cuda")
    lid = torch.from_numpy(part.local_ids).cuda()
    gnn.halo_push_quantized(g, H, lid, codes, sz, bits, seed)
    assert_ok(g)
    rng = np.random.default_rng(1)
    rows = rng.choice(part.n_local, 2000, replace=False)
    hv = H[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    ref_c, ref_sz = oracle.quantize_rows(hv, part.local_ids[rows], bits, seed, ldc)
    tid = torch.from_numpy(part.local_ids[rows]).cuda()
    np.testing.assert_array_equal(codes[tid].cpu().numpy(), ref_c)
    np.testing.assert_array_equal(sz[tid].cpu().numpy().view(np.uint32), ref_sz.view(np.uint32))
    Hin = padded(part.n_total, f, torch.bfloat16, "cuda")
    gnn.halo_pull_quantized(g, codes, sz, bits, torch.from_numpy(part.halo_ids).cuda(), Hin)
    assert_ok(g)
    hs = rng.choice(part.n_halo, 2000, replace=False)
    hid = part.halo_ids[hs]
    ref = oracle.dequantize_rows(codes[torch.from_numpy(hid).cuda()].cpu().numpy(),
                                 sz[torch.from_numpy(hid).cuda()].cpu().numpy(), f, bits)
    ref = oracle.round_bf16(ref.astype(np.float64)).astype(np.float32)
    got = Hin[part.n_local + torch.from_numpy(hs).cuda()].float().cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_codec_bad_ids_and_arguments():
    w, part, g = problem("er5k", "tiny")
    f, bits = w.widths[1], 2
    H = to_device(gen_matrix(part.n_local, f, "f32", SEED, 5), "f32", f)
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.zeros((part.n_table, ldc), dtype=torch.uint8, device="cuda")
    sz = torch.zeros((part.n_table, 2), dtype=torch.float32, device="cuda")
    ids = part.local_ids.copy()
    ids[3] = ids[4]  # repeated id: both rows skipped, error word set
    gnn.halo_push_quantized(g, H, torch.from_numpy(ids).cuda(), codes, sz, bits, 1)
    assert gnn.get_error(g) == gnn.GNN_EINDEX
    assert int(codes[ids[4]].abs().sum()) == 0
    hids = part.halo_ids.copy()
    hids[0] = part.n_table  # outside the table
    Hin = padded(part.n_total, f, torch.float32, "cuda")
    gnn.halo_pull_quantized(g, codes, sz, bits, torch.from_numpy(hids).cuda(), Hin)
    assert gnn.get_error(g) == gnn.GNN_EINDEX
    with pytest.raises(gnn.GnnError):
        gnn.halo_push_quantized(g, H, torch.from_numpy(part.local_ids).cuda(), codes, sz, 3, 1)
    with pytest.raises(gnn.GnnError):
        narrow = torch.zeros((part.n_table, 8), dtype=torch.uint8, device="cuda")  # row pitch not a multiple of 16
        gnn.halo_pull_quantized(g, narrow, sz, bits, torch.from_numpy(part.halo_ids).cuda(), Hin)
    assert_ok(g)


# ---------------------------------------------------------------------------
# the codec on rows of a message between processes (gnn_quantize_rows /
# gnn_dequantize_rows): codes keyed by the rows' global ids, dequantised into
# place or added onto rows of another matrix
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
@pytest.mark.parametrize("f", [3, 40, 64, 100, 128, 200, 256, 300])
def test_message_rows_special_magnitudes(bits, f):
    # every branch of the quantiser at widths that take 1, 2 or 4 chunks of 8 values per lane (with ragged
    # last lanes) and at a width past the eight-lanes-per-row kernels
    n = 1000
    Xv = _special_rows(n, f, np.random.default_rng(10 * bits + f))
    X = padded(n, f, torch.float32, "cuda")
    X.copy_(torch.from_numpy(Xv).cuda())
    keys = np.random.default_rng(f).permutation(4 * n)[:n].astype(np.int64)
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.full((n, ldc), 0x5A, dtype=torch.uint8, device="cuda")
    sz = torch.zeros((n, 2), dtype=torch.float32, device="cuda")
    seed = 123 + bits
    gnn.quantize_rows(X, torch.from_numpy(keys).cuda(), codes, sz, bits, seed)
    ref_c, ref_sz = oracle.quantize_rows(Xv, keys, bits, seed, ldc)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)
    np.testing.assert_array_equal(sz.cpu().numpy().view(np.uint32), ref_sz.view(np.uint32))


# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
@pytest.mark.parametrize("f", [5, 64, 100, 128, 200, 256, 300])
def test_message_rows_codec_matches_oracle(dt, bits, f):
    rng = np.random.default_rng(bits * 1000 + f)
    n = 2000
    X_h = gen_matrix(n, f, dt, SEED, 900 + bits)
    X = to_device(X_h, dt, f)
    keys = rng.permutation(10 * n)[:n].astype(np.int64)
    ldc = gnn.codec_row_bytes(f, bits)
    codes = torch.full((n, ldc), 0xCD, dtype=torch.uint8, device="cuda")
    sz = torch.zeros((n, 2), dtype=torch.float32, device="cuda")
    seed = 0xABC + bits
    gnn.quantize_rows(X, torch.from_numpy(keys).cuda(), codes, sz, bits, seed)
    ref_c, ref_sz = oracle.quantize_rows(_values(X_h, dt, f), keys, bits, seed, ldc)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)
    np.testing.assert_array_equal(sz.cpu().numpy().view(np.uint32), ref_sz.view(np.uint32))
    # dequantise into place
    tdt = torch_dtype(dt)
    Y = padded(n, f, tdt, "cuda")
    gnn.dequantize_rows(codes, sz, bits, Y)
    ref_y = oracle.dequantize_rows(ref_c, ref_sz, f, bits)
    ref_y = oracle.round_bf16(ref_y.astype(np.float64)) if dt == "bf16" else ref_y.astype(np.float64)
    np.testing.assert_array_equal(Y.float().cpu().numpy().astype(np.float64), ref_y)
    # dequantise and add onto distinct rows of another matrix
    m_rows = 3 * n
    D_h = gen_matrix(m_rows, f, dt, SEED, 950 + bits)
    D = to_device(D_h, dt, f)
    ids = rng.permutation(m_rows)[:n].astype(np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gnn.dequantize_rows(codes, sz, bits, D, ids=torch.from_numpy(ids).cuda(), add=True, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    base = widen(D_h, dt, f).astype(np.float32)
    want = base.copy()
    want[ids] = base[ids] + oracle.dequantize_rows(ref_c, ref_sz, f, bits)  # one fp32 rounding per element
    want = oracle.round_bf16(want.astype(np.float64)) if dt == "bf16" else want.astype(np.float64)
    np.testing.assert_array_equal(D.float().cpu().numpy().astype(np.float64), want)
