"""The seeded input generators: determinism, structure and value distributions."""
import numpy as np
import pytest

import synth


def _check_partition(p, symmetric_deg=True):
    assert p.rowptr[0] == 0 and p.rowptr[-1] == p.nnz
    assert np.all(np.diff(p.rowptr) >= 1)  # every row holds at least its self loop
    for v in range(p.n_local):
        row = p.colidx[p.rowptr[v]:p.rowptr[v + 1]]
        assert np.all(np.diff(row) > 0)
        assert v in row
        assert row.min() >= 0 and row.max() < p.n_total
    ids = np.concatenate([p.local_ids, p.halo_ids])
    assert np.unique(ids).shape[0] == ids.shape[0]
    assert ids.min() >= 0 and ids.max() < p.n_table
    if p.deg is not None:
        rowlen = np.diff(p.rowptr)
        np.testing.assert_array_equal(p.deg[:p.n_local], rowlen.astype(np.float32))


def test_er_partition_shape_and_determinism():
    a = synth.er_partition(512, 400, 16 / 511, seed=0)
    b = synth.er_partition(512, 400, 16 / 511, seed=0)
    c = synth.er_partition(512, 400, 16 / 511, seed=1)
    np.testing.assert_array_equal(a.colidx, b.colidx)
    assert not np.array_equal(a.colidx, c.colidx) or a.nnz != c.nnz
    assert a.n_local == 400 and a.n_halo == 112
    _check_partition(a)
    mean_deg = (a.nnz - a.n_local) / a.n_local
    assert 13 < mean_deg < 19


def test_rmat_and_chunglu_partitions_are_valid():
    r = synth.rmat_sym_partition(10, 3000, 900, seed=0)
    _check_partition(r)
    assert r.n_halo == 1024 - 900
    cl = synth.chunglu_partition(3000, 20000, 13.3, 4, seed=0)
    _check_partition(cl)
    assert cl.n_local == 750
    d = np.diff(cl.rowptr)
    assert d.max() > 5 * d.mean()  # heavy tail


def test_rmat_block_partition_is_valid_and_skewed():
    p = synth.rmat_block_partition(12, 2048, 1024, 40000.0, seed=0)
    assert p.deg is None
    _check_partition(p, symmetric_deg=False)
    assert p.n_table == 4096
    d = np.diff(p.rowptr)
    assert d.max() > 10 * d.mean()
    q = synth.rmat_block_partition(12, 2048, 1024, 40000.0, seed=0)
    np.testing.assert_array_equal(p.colidx, q.colidx)
    np.testing.assert_array_equal(p.local_ids, q.local_ids)


def test_features_depend_only_on_id_and_column():
    full = synth.features(100, 10, 12, seed=0, stream=synth.STREAM_FEATURES)
    ids = np.array([5, 99, 0, 5])
    some = synth.features(0, 10, 16, seed=0, stream=synth.STREAM_FEATURES, ids=ids)
    np.testing.assert_array_equal(some[:, :10], full[ids, :10])
    assert np.all(full[:, 10:] == 0) and np.all(some[:, 10:] == 0)
    x = synth.features(4000, 64, 64, seed=0, stream=3)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    u = synth.features(4000, 64, 64, seed=0, stream=3, dist="uniform")
    assert u.min() >= -1 and u.max() <= 1 and abs(u.std() - (1 / 3) ** 0.5) < 0.01


def test_bf16_features_round_to_nearest_even_like_torch():
    torch = pytest.importorskip("torch")
    x = synth.features(300, 50, 56, seed=2, stream=7)
    b = synth.features(300, 50, 56, seed=2, stream=7, bf16=True)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(b, ref)


def test_glorot_and_labels():
    W = synth.glorot(256, 32, 0, synth.STREAM_WEIGHT)
    a = (6 / 288) ** 0.5
    assert np.abs(W).max() <= a and np.abs(W).max() > 0.95 * a
    y = synth.labels(10000, 41, 0)
    assert y.min() == 0 and y.max() == 40
    assert np.all(np.bincount(y) > 150)
    rows = synth.sample_rows(1000, 50, 0)
    assert rows.shape == (50,) and np.all(np.diff(rows) > 0)
