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
    searchsorted; each centroid becomes the mean of its cell's samples, the
    sum and the division in float64 and the quotient rounded to fp32 once;
    a cell with no samples keeps its centroid;
  - the result is the centroids after the last iteration and their
    midpoints.
Library steps used: numpy's searchsorted (side="left" counts the boundaries
strictly below x) and bincount (per-cell counts and float64 sums, added in
sample order).
"""
from __future__ import annotations

import numpy as np


def midpoints(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, np.float32)
    return ((c[:-1] + c[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)


def lloyd_step(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """One Lloyd iteration: the new centroids."""
    K = c.shape[0]
    idx = np.searchsorted(midpoints(c), x, side="left")
    cnt = np.bincount(idx, minlength=K)
    s = np.bincount(idx, weights=x.astype(np.float64), minlength=K)
    out = c.copy()
    nz = cnt > 0
    out[nz] = (s[nz] / cnt[nz]).astype(np.float32)
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
    idx = np.searchsorted(midpoints(c), x, side="left")
    d = x.astype(np.float64) - np.asarray(c, np.float64)[idx]
    return float(np.mean(d * d))
