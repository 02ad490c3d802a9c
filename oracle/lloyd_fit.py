"""Oracle of the Lloyd-Max table fit.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the CUDA library
never imports it.

What it follows: page "mlx-bun 0.0.9 -> 0.0.11", file
package/src/mlx/turboquant-tables.ts, header comment: the value tables for
2, 4, 5 and 8 bits are an iterative Lloyd-Max fit on a unit-normal sample,
500 iterations. The page gives neither the sample size, the initial
centroids nor the handling of an empty cell; the readings taken here:
  - the sample x and the initial centroids are inputs (the sample's random
    numbers are drawn by the caller);
  - one iteration: boundaries are the fp32 midpoints of adjacent centroids,
    RN(c_k + c_{k+1}) / 2 (the printed tables' boundaries are those
    midpoints); each sample goes to cell count(boundaries < x), the codec's
    searchsorted; each centroid becomes the mean of its cell's samples: the
    exact sum over the exact count, rounded once to fp32 (round to nearest,
    ties to even); a cell with no samples keeps its centroid;
  - the result is the centroids after the last iteration and their
    midpoints.
Exact sums: every sample is an integer multiple of 2^-64 when it is 0 or
|x| >= 2^-41 (an fp32 value's last bit is then worth at least 2^-64), so each
sample splits into integer parts of 2^-32 and 2^-64 units and the cell sums
are integer sums; samples outside that range (or with |x| >= 2^8) are
refused. Library steps used: numpy's searchsorted (side="left" counts the
boundaries strictly below x) and bincount (per-cell counts, and per-cell sums
of integer pieces below 2^21, which float64 adds exactly).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def midpoints(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.float32)
    return ((c[:-1] + c[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)


def cells(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """Cell of every sample: count(boundaries < x)."""
    return np.searchsorted(midpoints(c), x, side="left")


def _check_domain(x: np.ndarray) -> None:
    a = np.abs(x.astype(np.float64))
    if not np.all(np.isfinite(a)) or np.any(a >= 256.0) or np.any((a > 0) & (a < 2.0 ** -41)):
        raise ValueError("lloyd oracle: samples must be 0 or 2^-41 <= |x| < 2^8 (exact in 2^-64 units)")


def _bincount_exact(idx: np.ndarray, v: np.ndarray, K: int) -> list[int]:
    """Per-cell sums of the non-negative int64 values v < 2^41, as Python ints:
    two pieces below 2^21 each, summed by bincount in float64 (exact: every
    partial sum of at most 2^31 pieces stays below 2^52)."""
    hi = (v >> 20).astype(np.float64)
    lo = (v & ((1 << 20) - 1)).astype(np.float64)
    sh = np.bincount(idx, weights=hi, minlength=K)
    sl = np.bincount(idx, weights=lo, minlength=K)
    return [(int(a) << 20) + int(b) for a, b in zip(sh, sl)]


def cell_sums(x: np.ndarray, idx: np.ndarray, K: int, chunk: int = 1 << 24) -> list[Fraction]:
    """Exact per-cell sums of the fp32 samples x (cell idx), as Fractions
    (computed in chunks of `chunk` samples to bound the memory)."""
    x = np.asarray(x, np.float32)
    if x.size > (1 << 31):
        raise ValueError("lloyd oracle: at most 2^31 samples")
    total = [0] * K  # in units of 2^-64
    for a in range(0, x.size, chunk):
        x64 = x[a:a + chunk].astype(np.float64)
        ix = idx[a:a + chunk]
        t = x64 * 2.0 ** 32  # exact (a power-of-two scaling)
        whole = np.floor(t)  # multiples of 2^-32 (|x| < 2^8: |whole| < 2^40)
        frac = (t - whole) * 2.0 ** 32  # exact: the integer count of 2^-64 units left, in [0, 2^32)
        w = whole.astype(np.int64) + (1 << 40)  # made non-negative for the split
        f = frac.astype(np.int64)
        sw = _bincount_exact(ix, w, K)
        sf = _bincount_exact(ix, f, K)
        cnt = np.bincount(ix, minlength=K)
        for k in range(K):
            total[k] += ((sw[k] - int(cnt[k]) * (1 << 40)) << 32) + sf[k]
    return [Fraction(t_, 1 << 64) for t_ in total]


def round_f32(q: Fraction) -> np.float32:
    """The fp32 value nearest to the rational q (ties to even), |q| < 2^128."""
    if q == 0:
        return np.float32(0.0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^e <= a < 2^(e+2)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # below the normal range the last bit is worth 2^-149
    scaled = a * Fraction(2) ** (23 - e)  # the 24-bit significand, with a fraction
    m, r = divmod(scaled.numerator, scaled.denominator)
    twice = 2 * r
    if twice > scaled.denominator or (twice == scaled.denominator and (m & 1)):
        m += 1
    return np.float32(s * float(m) * 2.0 ** (e - 23))  # exact: m <= 2^24


def lloyd_step(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """One Lloyd iteration: the new centroids."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    _check_domain(x)
    K = c.shape[0]
    idx = cells(x, c)
    cnt = np.bincount(idx, minlength=K)
    sums = cell_sums(x, idx, K)
    out = np.array(c, np.float32).copy()
    for k in range(K):
        if cnt[k] > 0:
            out[k] = round_f32(sums[k] / int(cnt[k]))
    return out


class SortedSample:
    """A sample sorted once, with exact prefix sums, so that the exact cell
    sums and counts of any centroids take a binary search per boundary (a sum
    does not depend on the order of its terms). Cell k holds the samples with
    b_{k-1} < x <= b_k, i.e. count(boundaries < x) = k. At most 2^22 samples
    (the prefix sums stay below 2^62)."""

    def __init__(self, x):
        xs = np.sort(np.asarray(x, np.float32))
        _check_domain(xs)
        if xs.size > (1 << 22):
            raise ValueError("SortedSample: at most 2^22 samples")
        t = xs.astype(np.float64) * 2.0 ** 32
        whole = np.floor(t)
        frac = (t - whole) * 2.0 ** 32
        z = np.zeros(1, np.int64)
        self.xs = xs
        self.pw = np.concatenate([z, np.cumsum(whole.astype(np.int64))])  # 2^-32 units
        self.pf = np.concatenate([z, np.cumsum(frac.astype(np.int64))])   # 2^-64 units
        self.off_grid = np.concatenate([z, np.cumsum((t != np.rint(t)).astype(np.int64))])

    def cells(self, c: np.ndarray):
        """(start, end) index ranges of every cell in the sorted sample."""
        cut = np.searchsorted(self.xs, midpoints(c), side="right")
        edges = np.concatenate([[0], cut, [self.xs.size]])
        return edges[:-1], edges[1:]

    def sums(self, c: np.ndarray):
        """Exact cell sums (Fractions), counts and counts of samples that are
        not multiples of 2^-32."""
        a, b = self.cells(c)
        sums = [Fraction((int(self.pw[e] - self.pw[s]) << 32) + int(self.pf[e] - self.pf[s]), 1 << 64)
                for s, e in zip(a, b)]
        return sums, (b - a), self.off_grid[b] - self.off_grid[a]

    def step(self, c: np.ndarray) -> np.ndarray:
        """lloyd_step on this sample."""
        sums, cnt, _ = self.sums(c)
        out = np.array(c, np.float32).copy()
        for k in range(out.shape[0]):
            if cnt[k] > 0:
                out[k] = round_f32(sums[k] / int(cnt[k]))
        return out


def lloyd_max_fit(x, init, iters: int):
    """Lloyd-Max fit of len(init) levels to the fp32 sample x, `iters`
    iterations from the centroids `init` -> (centroids, boundaries), fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    c = np.array(init, dtype=np.float32)
    for _ in range(iters):
        c = lloyd_step(x, c)
    return c, midpoints(c)


def distortion(x, c) -> float:
    """Mean squared error of quantising x to the centroids c (float64)."""
    x = np.asarray(x, np.float32)
    idx = cells(x, c)
    d = x.astype(np.float64) - np.asarray(c, np.float64)[idx]
    return float(np.mean(d * d))
