"""GPU parity of the Lloyd-Max table fit (tq_lloyd_max_fit) against the
oracle's lloyd_max_fit on the same seeded samples and initial centroids.

Page "mlx-bun 0.0.9 -> 0.0.11", file turboquant-tables.ts (header: the value
tables are an iterative Lloyd-Max fit on a unit-normal sample).

Tolerance: both sides sum each cell exactly enough that the float64 mean
rounds to the same fp32 value except when it falls within about 2^-40 of a
rounding midpoint; such a one-ulp step moves a boundary by one ulp and can
move a sample lying exactly there, so results are compared to 4 ulp of each
centroid (measured: identical in the cases below).
"""
import numpy as np
import pytest
import torch

import turboquant_kv_cache_tq_gb300 as tq
from oracle import lloyd_fit as lf
from tests.gpu_common import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fit(x, init, iters):
    c, b = tq.tq_lloyd_max_fit(torch.from_numpy(np.asarray(x, np.float32)).cuda(),
                               torch.from_numpy(np.asarray(init, np.float32)).cuda(), iters)
    torch.cuda.synchronize()
    return c.cpu().numpy(), b.cpu().numpy()


def _ulps(a, b):
    return np.abs(a.astype(np.float64) - b.astype(np.float64)) / np.spacing(np.abs(b).astype(np.float32)).astype(np.float64)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_matches_oracle(bits):
    K = 1 << bits
    x = np.random.default_rng(bits).standard_normal(1 << 16).astype(np.float32)
    init = np.linspace(-2.5, 2.5, K).astype(np.float32)
    c, b = _fit(x, init, 60)
    rc, rb = lf.lloyd_max_fit(x, init, 60)
    assert np.max(_ulps(c, rc)) <= 4, (bits, np.max(_ulps(c, rc)))
    assert np.max(_ulps(b, rb)) <= 4


def test_worked_example_and_empty_cells():
    c, b = _fit([-3.0, -1.0, 0.0, 2.0, 4.0], [-1.0, 1.0], 3)
    assert c[0] == np.float32(-4.0 / 3.0) and c[1] == np.float32(3.0)
    c, _ = _fit([1.0, 2.0, 3.0], [-10.0, 1.0, 5.0, 10.0], 1)
    assert np.array_equal(c, np.array([-10.0, 2.0, 5.0, 10.0], np.float32))


def test_zero_iterations_and_empty_sample():
    init = np.array([-1.5, -0.5, 0.25, 2.0], np.float32)
    c, b = _fit(np.zeros(0, np.float32), init, 0)
    assert np.array_equal(c, init) and np.array_equal(b, lf.midpoints(init))
    c, b = _fit(np.zeros(0, np.float32), init, 5)  # no samples: every cell keeps its centroid
    assert np.array_equal(c, init)


def test_large_sample_reaches_the_printed_table_neighbourhood(oracle_mod=None):
    import oracle

    x = np.random.default_rng(9).standard_normal(1 << 20).astype(np.float32)
    printed, _ = oracle.lloyd_max(2)
    c, _ = _fit(x, np.linspace(-2.0, 2.0, 4), 200)
    rc, _ = lf.lloyd_max_fit(x, np.linspace(-2.0, 2.0, 4), 200)
    assert np.max(_ulps(c, rc)) <= 4
    assert np.max(np.abs(c - printed)) < 0.02  # the page's own fit, on its own sample


def test_host_checks():
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError):
        tq.tq_lloyd_max_fit(x, torch.zeros(3, dtype=torch.float32, device="cuda"), 1)  # not a power of two
    with pytest.raises(tq.TQError):
        tq.tq_lloyd_max_fit(x, torch.zeros(512, dtype=torch.float32, device="cuda"), 1)


def test_bench_size_fit():
    """The bench's fit: 2^20 N(0,1) samples, 500 iterations, 16 levels."""
    x = np.random.default_rng(7).standard_normal(1 << 20).astype(np.float32)
    init = np.linspace(-3.0, 3.0, 16).astype(np.float32)
    c, b = _fit(x, init, 500)
    rc, rb = lf.lloyd_max_fit(x, init, 500)
    assert np.max(_ulps(c, rc)) <= 4 and np.max(_ulps(b, rb)) <= 4


def test_large_sample_takes_the_int64_sums():
    """A warp keeps its cell sums in split 32-bit words while it bins at most
    65536 samples per iteration; 170 M samples (more than 65536 per warp at
    two blocks of eight warps on each of 152 SMs) take the int64 sums.
    Two iterations against the oracle."""
    n = 170_000_000
    x = np.random.default_rng(11).standard_normal(n).astype(np.float32)
    init = np.linspace(-2.5, 2.5, 16).astype(np.float32)
    c, b = _fit(x, init, 2)
    rc, rb = lf.lloyd_max_fit(x, init, 2)
    assert np.max(_ulps(c, rc)) <= 4 and np.max(_ulps(b, rb)) <= 4
