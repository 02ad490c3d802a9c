"""Pins of the oracle's constant tables.

The tables are data printed on the page "mlx-bun 0.0.9 -> 0.0.11", file
package/src/mlx/turboquant-tables.ts (SIGN_VECTORS, LLOYD_MAX). They are
checked here against (a) a separate text transcription of the printed numbers
(tests/golden/turboquant_tables.txt), (b) the structural facts the page states
(one sign per head_dim element, 2^b centroids, 2^b-1 boundaries, boundaries as
decision points between adjacent centroids) and (c) the mathematics of a
Lloyd-Max quantiser for a unit normal source (centroid condition, closed-form
distortion against Max's published optimum for 2-4 bits).
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "turboquant_tables.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, toks = line.split(":", 1)
        kind, key = head.split()
        out[(kind, int(key))] = toks.split()
    return out


def _phi(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi) if math.isfinite(x) else 0.0


def _Phi(x):
    if x == math.inf:
        return 1.0
    if x == -math.inf:
        return 0.0
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def gaussian_mse(cent, bnd):
    """Closed-form E[(X - Q(X))^2] for X ~ N(0,1): cell i = (b_{i-1}, b_i]."""
    edges = [-math.inf] + [float(b) for b in bnd] + [math.inf]
    total = 0.0
    for i, c in enumerate(cent):
        a, b = edges[i], edges[i + 1]
        p = _Phi(b) - _Phi(a)
        m1 = _phi(a) - _phi(b)  # int x phi
        afa = a * _phi(a) if math.isfinite(a) else 0.0
        bfb = b * _phi(b) if math.isfinite(b) else 0.0
        m2 = p + afa - bfb  # int x^2 phi
        c = float(c)
        total += m2 - 2 * c * m1 + c * c * p
    return total


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_signs_match_printed_table(oracle_mod, d):
    g = _golden()[("signs", d)]
    s = oracle_mod.sign_vector(d)
    assert len(g) == d and s.shape == (d,)
    assert np.array_equal(s, np.array([int(t) for t in g], np.int8))
    assert set(np.unique(s).tolist()) <= {-1, 1}


def test_sign_counts(oracle_mod):
    # number of +1 entries in each printed table
    counts = {d: int((oracle_mod.sign_vector(d) == 1).sum()) for d in (64, 128, 256, 512)}
    assert counts == {64: 35, 128: 69, 256: 124, 512: 262}


def test_unsupported_tables(oracle_mod):
    for d in (32, 96, 1024):
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.sign_vector(d)
    for b in (1, 6, 7, 16):
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.lloyd_max(b)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_lloyd_max_matches_printed_table(oracle_mod, bits):
    gold = _golden()
    c, b = oracle_mod.lloyd_max(bits)
    gc = np.array([np.float32(float(t)) for t in gold[("centroids", bits)]], np.float32)
    gb = np.array([np.float32(float(t)) for t in gold[("boundaries", bits)]], np.float32)
    assert c.shape == (2 ** bits,) and b.shape == (2 ** bits - 1,)
    assert np.array_equal(c.view(np.uint32), gc.view(np.uint32))
    assert np.array_equal(b.view(np.uint32), gb.view(np.uint32))
    # every printed number is an exact float32 value
    for t in gold[("centroids", bits)] + gold[("boundaries", bits)]:
        assert float(np.float32(float(t))) == float(t)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_tables_ascend_and_interleave(oracle_mod, bits):
    c, b = oracle_mod.lloyd_max(bits)
    assert np.all(np.diff(c) > 0) and np.all(np.diff(b) > 0)
    # each boundary lies strictly between its two centroids
    assert np.all(c[:-1] < b) and np.all(b < c[1:])


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_boundaries_are_centroid_midpoints(oracle_mod, bits):
    c, b = oracle_mod.lloyd_max(bits)
    mid = ((c[:-1] + c[1:]) / np.float32(2)).astype(np.float32)
    ulps = np.abs(mid.view(np.int32).astype(np.int64) - b.view(np.int32).astype(np.int64))
    if bits == 3:
        # the hard-coded 3-bit table differs from the fp32 midpoint by 1 ulp twice
        assert ulps.max() <= 1 and int((ulps != 0).sum()) == 2
    else:
        assert ulps.max() == 0


def test_three_bit_table_is_symmetric(oracle_mod):
    c, b = oracle_mod.lloyd_max(3)
    assert np.array_equal(c, -c[::-1]) and np.array_equal(b, -b[::-1])


@pytest.mark.parametrize("bits,tol", [(2, 0.02), (3, 2e-4), (4, 0.02), (5, 0.03)])
def test_centroid_condition_for_unit_normal(oracle_mod, bits, tol):
    """Lloyd-Max optimality: each centroid is the conditional mean of its cell
    under N(0,1). The 3-bit table is the textbook table (tight tolerance); the
    others were fitted on a finite sample (looser tolerance)."""
    c, b = oracle_mod.lloyd_max(bits)
    edges = [-math.inf] + [float(x) for x in b] + [math.inf]
    for i in range(len(c)):
        a, e = edges[i], edges[i + 1]
        cond_mean = (_phi(a) - _phi(e)) / (_Phi(e) - _Phi(a))
        assert abs(float(c[i]) - cond_mean) < tol, (i, float(c[i]), cond_mean)


@pytest.mark.parametrize("bits,max_mse", [(2, 0.1175), (3, 0.03455), (4, 0.009497)])
def test_distortion_matches_max_optimum(oracle_mod, bits, max_mse):
    """Max (1960) optimum mean-square error of a b-bit quantiser for a unit
    normal source; the tables must reach it within 0.5%."""
    c, b = oracle_mod.lloyd_max(bits)
    assert abs(gaussian_mse(c, b) / max_mse - 1.0) < 5e-3


def test_distortion_decreases_with_bits(oracle_mod):
    m = [gaussian_mse(*oracle_mod.lloyd_max(bits)) for bits in (2, 3, 4, 5, 8)]
    assert all(m[i] > m[i + 1] for i in range(4))
    # high-resolution (Panter-Dite) regime for 5 bits: ~ sqrt(3) pi / 2 * 4^-b
    assert abs(m[3] / (math.sqrt(3) * math.pi / 2 * 4.0 ** -5) - 1) < 0.08
