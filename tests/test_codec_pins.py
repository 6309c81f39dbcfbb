"""Pins of the oracle's low-bit halo codec (Sylvie page, Quantizer and
Dequantizer; unbiasedness theorems of its convergence section).

The codec's formulas are stripped from the page text; the reading used is: per
row, zero point = min, scale = (max - min) / B with B = 2^b - 1, code =
stochastic rounding of (h - min) / scale into [0, B], recovered value =
code * scale + min.  These tests pin the oracle's implementation to facts that
do not depend on it: the published SplitMix64 outputs, closed-form cases, the
error bound of stochastic rounding, its unbiasedness (the page's theorem),
the variance falling with the bit width, and the 32x byte ratio of 1-bit codes
against fp32 rows that the page's communication table reports.
"""
import numpy as np
import pytest

import oracle


def test_splitmix64_published_outputs():
    # first outputs of SplitMix64 seeded with 0 (reference implementation's stream)
    assert oracle.splitmix64(0, 1) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64(0, 2) == 0x6E789E6AA1B965F4
    assert oracle.splitmix64(0, 3) == 0x06C45D188009454F


def test_constant_row_is_exact():
    x = np.full((3, 37), 1.25, np.float32)
    for b in (1, 2, 4, 8):
        codes, sz = oracle.quantize_rows(x, np.arange(3), b, seed=9)
        assert np.all(codes == 0) and np.all(sz[:, 0] == 0) and np.all(sz[:, 1] == 1.25)
        assert np.array_equal(oracle.dequantize_rows(codes, sz, 37, b), x)


def test_grid_row_is_exact_and_packed_little_endian():
    # values already on the quantisation grid come back exactly (u < 1 never
    # lifts an exact integer for these small magnitudes)
    x = np.array([[0.0, 1.0, 2.0, 3.0, 3.0, 0.0, 1.0, 2.0]], np.float32)
    codes, sz = oracle.quantize_rows(x, np.array([5]), 2, seed=3)
    assert sz[0, 0] == 1.0 and sz[0, 1] == 0.0
    assert codes[0, 0] == 0b11100100 and codes[0, 1] == 0b10010011  # codes 0,1,2,3 | 3,0,1,2
    assert np.array_equal(oracle.dequantize_rows(codes, sz, 8, 2), x)


def test_one_bit_middle_value_follows_its_draw():
    # b = 1, row [0, 0.5, 1]: the middle value rounds up exactly when its
    # uniform draw (16 bits of its SplitMix64 output) is >= 1/2
    x = np.array([[0.0, 0.5, 1.0]], np.float32)
    for r in range(64):
        codes, _ = oracle.quantize_rows(x, np.array([r]), 1, seed=11)
        # element 1 takes bits 32..47 of output k = r * 2^14 + 0 + 1
        u = ((oracle.splitmix64(11, (r << 14) + 1) >> 32) & 0xFFFF) / 2.0**16
        assert (codes[0, 0] >> 1) & 1 == (1 if u >= 0.5 else 0)
        assert codes[0, 0] & 1 == 0 and (codes[0, 0] >> 2) & 1 == 1


@pytest.mark.parametrize("b", [1, 2, 4, 8])
def test_error_bound_and_code_range(b):
    rng = np.random.default_rng(b)
    x = rng.standard_normal((200, 75)).astype(np.float32)
    codes, sz = oracle.quantize_rows(x, np.arange(200) * 7 + 1, b, seed=123)
    y = oracle.dequantize_rows(codes, sz, 75, b)
    scale = sz[:, :1].astype(np.float64)
    err = np.abs(y.astype(np.float64) - x)
    assert np.all(err <= scale * (1 + 1e-5) + 1e-7)
    # the smallest and the largest value of each row are recovered exactly
    assert np.array_equal(y.min(axis=1), x.min(axis=1))
    # row bytes past the f codes stay zero
    used = (75 * b + 7) // 8
    assert np.all(codes[:, used + 1:] == 0)


def test_unbiased_mean_over_draws():
    # the page's theorem: dequantise(quantise(h)) is an unbiased estimate of h.
    # N independent draws (one per table id) of the same row; the mean must
    # sit within 6 standard errors (per-element standard deviation <= scale / 2)
    rng = np.random.default_rng(0)
    h = rng.uniform(-2, 3, 48).astype(np.float32)
    N = 20000
    x = np.repeat(h[None, :], N, axis=0)
    for b in (1, 2, 4):
        codes, sz = oracle.quantize_rows(x, np.arange(N), b, seed=77)
        y = oracle.dequantize_rows(codes, sz, 48, b).astype(np.float64)
        s = float(sz[0, 0])
        assert np.all(np.abs(y.mean(axis=0) - h) <= 6 * (s / 2) / np.sqrt(N))


def test_variance_falls_with_bits():
    rng = np.random.default_rng(1)
    h = rng.standard_normal(64).astype(np.float32)
    N = 4000
    x = np.repeat(h[None, :], N, axis=0)
    var = []
    for b in (1, 2, 4, 8):
        codes, sz = oracle.quantize_rows(x, np.arange(N), b, seed=5)
        y = oracle.dequantize_rows(codes, sz, 64, b).astype(np.float64)
        var.append(float(((y - h) ** 2).mean()))
        assert var[-1] <= float(sz[0, 0]) ** 2 / 4 * 1.05  # Bernoulli variance bound s^2 p (1 - p) <= s^2 / 4
    assert var[0] > var[1] > var[2] > var[3]


def test_one_bit_rows_are_32x_smaller_than_fp32():
    # the page's communication table: 1-bit codes cut fp32 embedding traffic ~32x
    for f in (128, 256, 1024):
        assert f * 4 / oracle.codec_row_bytes(f, 1) == 32
        assert oracle.codec_row_bytes(f, 8) == f
