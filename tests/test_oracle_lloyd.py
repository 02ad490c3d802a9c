"""Pins of the oracle's Lloyd-Max fit (page "mlx-bun 0.0.9 -> 0.0.11", file
turboquant-tables.ts: the value tables are an iterative Lloyd-Max fit on a
unit-normal sample, 500 iterations).

Pins used:
- a worked example by hand (cells, the boundary tie going to the lower
  cell, the fixed point reached);
- the empty-cell reading (an empty cell keeps its centroid);
- the closed form for two levels on N(0,1): centroids +-sqrt(2/pi);
- convergence to the page's printed 2-, 4- and 5-bit tables within the
  sampling error of each cell mean (the page fitted a different sample);
- Lloyd's descent property: the distortion never increases.
"""
import math

import numpy as np
import pytest

from oracle import lloyd_fit as lf


def test_worked_example():
    x = np.array([-3.0, -1.0, 0.0, 2.0, 4.0], np.float32)
    c1 = lf.lloyd_step(x, np.array([-1.0, 1.0], np.float32))
    # boundary 0: -3, -1 and 0 (not above the boundary) -> cell 0; 2, 4 -> cell 1
    assert c1[0] == np.float32(-4.0 / 3.0) and c1[1] == np.float32(3.0)
    c2 = lf.lloyd_step(x, c1)  # boundary 0.8333: same cells, a fixed point
    assert np.array_equal(c1, c2)
    c, b = lf.lloyd_max_fit(x, [-1.0, 1.0], 5)
    assert np.array_equal(c, c1) and b[0] == np.float32(np.float32(c1[0] + c1[1]) * np.float32(0.5))


def test_empty_cells_keep_their_centroids():
    x = np.array([1.0, 2.0, 3.0], np.float32)
    c = lf.lloyd_step(x, np.array([-10.0, 1.0, 10.0], np.float32))
    assert np.array_equal(c, np.array([-10.0, 2.0, 10.0], np.float32))


def _normal(n, seed):
    return np.random.default_rng(seed).standard_normal(n).astype(np.float32)


def test_two_levels_closed_form():
    x = _normal(1 << 20, 1)
    c, b = lf.lloyd_max_fit(x, [-1.0, 1.0], 30)
    want = math.sqrt(2.0 / math.pi)
    assert abs(c[0] + want) < 4e-3 and abs(c[1] - want) < 4e-3 and abs(b[0]) < 4e-3


# Max (1960), the minimum-mean-squared-error quantizer of a unit-variance
# Gaussian: the positive levels for 4, 8 and 16 levels.
MAX_1960 = {4: [0.4528, 1.510], 8: [0.2451, 0.7560, 1.344, 2.152],
            16: [0.1284, 0.3881, 0.6568, 0.9424, 1.256, 1.618, 2.069, 2.733]}


@pytest.mark.parametrize("K,tol", [(4, 2e-3), (8, 5e-3), (16, 3e-2)])
def test_converges_to_the_textbook_gaussian_quantizer(K, tol):
    """The fit of a large N(0,1) sample reaches Max's optimum within the
    sample's error (largest for the sparse outer cells of 16 levels)."""
    x = _normal(1 << 20, 2)
    c, _ = lf.lloyd_max_fit(x, np.linspace(-2.0, 2.0, K), 100)
    assert np.max(np.abs(c[K // 2:] - np.array(MAX_1960[K]))) < tol
    assert np.max(np.abs(c[: K // 2][::-1] + np.array(MAX_1960[K]))) < tol


@pytest.mark.parametrize("bits", [2, 4, 5])
def test_printed_tables_are_near_fixed_points(oracle_mod, bits):
    """Started from the page's printed table, the fit on a large N(0,1)
    sample moves no centroid by much more than the printed table's own
    departure from symmetry (the page fitted a smaller sample of its own, and
    the sparse outer cells vary most from sample to sample)."""
    x = _normal(1 << 20, 2)
    printed, _ = oracle_mod.lloyd_max(bits)
    c, _ = lf.lloyd_max_fit(x, printed, 60)
    asym = np.max(np.abs(printed + printed[::-1]))
    assert np.max(np.abs(c - printed)) < 1.5 * asym


def test_distortion_never_increases():
    x = _normal(50000, 3)
    c = np.linspace(-3.0, 3.0, 16).astype(np.float32)
    d = lf.distortion(x, c)
    for _ in range(40):
        c = lf.lloyd_step(x, c)
        d2 = lf.distortion(x, c)
        assert d2 <= d * (1 + 1e-12)
        d = d2
    assert np.all(np.diff(c) > 0)


# ---- the exact cell means ---------------------------------------------------------------
def test_cell_sums_are_the_correctly_rounded_sums():
    """float() of each exact cell sum equals math.fsum of the cell's samples
    (Python's fsum returns the correctly rounded sum of its inputs), on
    samples spanning 2^-40 .. 2^7 in magnitude."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-40, 6, 200000))).astype(np.float32)
    c = np.linspace(-1.0, 1.0, 8).astype(np.float32)
    idx = lf.cells(x, c)
    sums = lf.cell_sums(x, idx, 8)
    for k in range(8):
        assert float(sums[k]) == math.fsum(x[idx == k].astype(np.float64).tolist())


def test_round_f32_single_rounding_and_ties():
    from fractions import Fraction

    rng = np.random.default_rng(6)
    v = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 100, 20000))
    for d in v:  # a float64 value rounded once to fp32 is numpy's cast
        assert lf.round_f32(Fraction(float(d))) == np.float32(d)
    one = Fraction(1)
    assert lf.round_f32(one + Fraction(1, 1 << 24)) == np.float32(1.0)  # tie -> even
    assert lf.round_f32(one + Fraction(3, 1 << 24)) == np.float32(1.0 + 2.0 ** -22)
    assert lf.round_f32(Fraction(1, 1 << 150)) == np.float32(0.0)  # half the smallest subnormal
    assert lf.round_f32(Fraction(3, 1 << 150)) == np.float32(2.0 ** -148)
    assert lf.round_f32(-Fraction(5, 3)) == np.float32(-5.0 / 3.0)


def test_exact_mean_where_float64_accumulation_is_not():
    """A cell of 2^16 - 1 samples 255, one 255.5 and 2^16 samples 2^-30: the
    exact mean is 127.5 + 2^-18 + 2^-31, just above the midpoint between the
    fp32 neighbours 127.5 and 127.5 + 2^-17, so it rounds up. A float64
    running sum in sample order loses every 2^-30 (a quarter of its last bit
    at 2^24) and lands exactly on the midpoint, which rounds to the even
    127.5: the cell mean must be the exact one."""
    x = np.concatenate([np.full((1 << 16) - 1, 255.0), [255.5], np.full(1 << 16, 2.0 ** -30)]).astype(np.float32)
    c = lf.lloyd_step(x, np.array([-100.0, 100.0], np.float32))
    assert c[0] == np.float32(-100.0)  # empty cell
    assert c[1] == np.float32(127.5 + 2.0 ** -17)
    running = np.bincount(np.ones(x.size, np.int64), weights=x.astype(np.float64), minlength=2)[1]
    assert np.float32(running / x.size) == np.float32(127.5)


def test_samples_outside_the_exact_range_are_refused():
    with pytest.raises(ValueError):
        lf.lloyd_step(np.array([1.0, 2.0 ** -45], np.float32), np.array([-1.0, 1.0], np.float32))
    with pytest.raises(ValueError):
        lf.lloyd_step(np.array([300.0], np.float32), np.array([-1.0, 1.0], np.float32))


def test_sorted_sample_steps_equal_the_plain_steps():
    """The prefix-sum form of an iteration (sorted sample) equals the plain
    per-sample form, cell sums and all, including boundary ties and samples
    below 2^-9."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal(50000)
    x[:2000] = np.sign(x[:2000]) * np.exp2(rng.uniform(-40, -9, 2000))
    x = x.astype(np.float32)
    c = np.linspace(-2.0, 2.0, 16).astype(np.float32)
    x[2000:2100] = lf.midpoints(c)[3]  # samples exactly on a boundary
    ss = lf.SortedSample(x)
    for _ in range(6):
        sums, cnt, _ = ss.sums(c)
        idx = lf.cells(x, c)
        assert np.array_equal(cnt, np.bincount(idx, minlength=16))
        assert sums == lf.cell_sums(x, idx, 16)
        c2 = ss.step(c)
        assert np.array_equal(c2, lf.lloyd_step(x, c))
        c = c2
