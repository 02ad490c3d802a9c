"""GPU parity of the Lloyd-Max table fit (tq_lloyd_max_fit) against the
oracle's lloyd_max_fit on the same seeded samples and initial centroids.

Page "mlx-bun 0.0.9 -> 0.0.11", file turboquant-tables.ts (header: the value
tables are an iterative Lloyd-Max fit on a unit-normal sample).

Tolerance, derived from the kernel's arithmetic. The oracle's cell mean is
the exact sum over the count, rounded once to fp32. The kernel sums every
sample as rint(x * 2^32) in int64 (exact for |x| >= 2^-9, where x is a
multiple of 2^-32; a smaller sample moves by at most 2^-33), so a cell with
m samples off that grid has a sum within m * 2^-33 of the exact one; it then
converts the integer sum to float64 and divides by the count in float64 (two
roundings, at most 2^-52 relative together) and rounds to fp32. As fp32
rounding is monotone, each GPU centroid of one iteration lies between the fp32
roundings of (S - m 2^-33) / n (1 - 2^-51) and (S + m 2^-33) / n (1 + 2^-51),
S the oracle's exact sum and n the count, from the same input centroids
(hence the same boundaries and cells). When those two roundings agree - the
common case - the centroid must equal the oracle's exactly. The tests check
this bound on every iteration of the GPU's own trajectory (single-iteration
launches chained), that a multi-iteration launch equals that chain bit for
bit, and that the whole fit equals the oracle's whole fit whenever every step
of the chain was unambiguous.
"""
from fractions import Fraction

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


def _fit_dev(xd, init, iters, **kw):
    c, b = tq.tq_lloyd_max_fit(xd, torch.from_numpy(np.asarray(init, np.float32)).cuda(), iters, **kw)
    torch.cuda.synchronize()
    return c.cpu().numpy(), b.cpu().numpy()


def _fit(x, init, iters):
    return _fit_dev(torch.from_numpy(np.asarray(x, np.float32)).cuda(), init, iters)


def step_bounds(sample, x: np.ndarray, c_in: np.ndarray):
    """fp32 bounds of every GPU centroid after one iteration from c_in, and
    the oracle's own step; empty cells keep their centroid exactly. `sample`
    is the oracle's SortedSample of x, or None for the per-sample form."""
    K = c_in.shape[0]
    if sample is not None:
        sums, cnt, off = sample.sums(c_in)
    else:
        idx = lf.cells(x, c_in)
        cnt = np.bincount(idx, minlength=K)
        sums = lf.cell_sums(x, idx, K)
        t = x.astype(np.float64) * 2.0 ** 32
        off = np.bincount(idx, weights=(t != np.rint(t)).astype(np.float64), minlength=K)
    lo = c_in.astype(np.float32).copy()
    hi = lo.copy()
    ref = lo.copy()
    slack = Fraction(1, 1 << 51)
    for k in range(K):
        if cnt[k] == 0:
            continue
        n = int(cnt[k])
        e = Fraction(int(off[k]), 1 << 33)
        ref[k] = lf.round_f32(sums[k] / n)
        m_lo, m_hi = (sums[k] - e) / n, (sums[k] + e) / n
        lo[k] = lf.round_f32(m_lo - abs(m_lo) * slack)
        hi[k] = lf.round_f32(m_hi + abs(m_hi) * slack)
    return lo, hi, ref


def check_chain(x: np.ndarray, init, iters: int):
    """Run the fit as `iters` chained single-iteration launches, checking each
    step against its derived bounds; then the multi-iteration launch against
    the chain, and against the oracle's fit when no step was ambiguous.
    Returns the number of ambiguous steps."""
    xd = torch.from_numpy(x).cuda()
    sample = lf.SortedSample(x) if x.size <= (1 << 22) else None
    c = np.asarray(init, np.float32)
    ambiguous = 0
    for it in range(iters):
        lo, hi, ref = step_bounds(sample, x, c)
        g, gb = _fit_dev(xd, c, 1)
        assert np.all((g >= lo) & (g <= hi)), (it, np.argwhere((g < lo) | (g > hi))[:4].tolist())
        assert np.array_equal(gb, lf.midpoints(g))
        ambiguous += int(np.any(lo != hi))
        if not np.any(lo != hi):
            assert np.array_equal(g, ref), it
        c = g
    full, fb = _fit_dev(xd, init, iters)
    assert np.array_equal(full, c) and np.array_equal(fb, lf.midpoints(c))
    if ambiguous == 0:
        rc = np.asarray(init, np.float32)
        for _ in range(iters):
            rc = sample.step(rc) if sample is not None else lf.lloyd_step(x, rc)
        assert np.array_equal(full, rc)
    return ambiguous


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_matches_oracle(bits):
    K = 1 << bits
    x = np.random.default_rng(bits).standard_normal(1 << 16).astype(np.float32)
    check_chain(x, np.linspace(-2.5, 2.5, K), 30)


def test_samples_off_the_fixed_point_grid():
    """Half of the samples are below 2^-9 in magnitude (not multiples of
    2^-32): the bound widens by their rounding and the GPU stays inside it."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal(1 << 16)
    small = rng.random(1 << 16) < 0.5
    x[small] = np.sign(x[small]) * np.exp2(rng.uniform(-40, -9, small.sum()))
    x = x.astype(np.float32)
    check_chain(x, np.linspace(-1.5, 1.5, 8), 10)


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


def test_large_sample_reaches_the_printed_table_neighbourhood():
    import oracle

    x = np.random.default_rng(9).standard_normal(1 << 20).astype(np.float32)
    printed, _ = oracle.lloyd_max(2)
    c, _ = _fit(x, np.linspace(-2.0, 2.0, 4), 200)
    rc, _ = lf.lloyd_max_fit(x, np.linspace(-2.0, 2.0, 4), 200)
    assert np.array_equal(c, rc)
    assert np.max(np.abs(c - printed)) < 0.02  # the page's own fit, on its own sample


def test_host_checks():
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError):
        tq.tq_lloyd_max_fit(x, torch.zeros(3, dtype=torch.float32, device="cuda"), 1)  # not a power of two
    with pytest.raises(tq.TQError):
        tq.tq_lloyd_max_fit(x, torch.zeros(512, dtype=torch.float32, device="cuda"), 1)


def test_bench_size_fit():
    """The bench's fit: 2^20 N(0,1) samples, 500 iterations, 16 levels, every
    iteration checked."""
    x = np.random.default_rng(7).standard_normal(1 << 20).astype(np.float32)
    check_chain(x, np.linspace(-3.0, 3.0, 16), 500)


def test_large_sample_takes_the_int64_sums():
    """A warp keeps its cell sums in split 32-bit words while it bins at most
    65536 samples per iteration; 170 M samples (more than 65536 per warp at
    two blocks of eight warps on each of 152 SMs) take the int64 sums.
    Two iterations, each checked."""
    n = 170_000_000
    x = np.random.default_rng(11).standard_normal(n).astype(np.float32)
    check_chain(x, np.linspace(-2.5, 2.5, 16), 2)


def test_barrier_give_up_is_reported():
    """Failure detection in a form that faults nothing: one block of the
    cooperative fit leaves without arriving at its first grid barrier
    (absent_block), every other block's bounded wait (spin_limit polls) runs
    out, the fit's error word is set and read back through the C ABI as
    TQ_ERR_TIMEOUT, and the results are NaN. The same workspace then serves a
    normal fit, whose status is TQ_OK again."""
    x = torch.from_numpy(np.random.default_rng(3).standard_normal(1 << 16).astype(np.float32)).cuda()
    init = torch.linspace(-2.0, 2.0, 16, device="cuda")
    work = torch.empty(tq.lib().tq_lloyd_max_fit_workspace_size(16), dtype=torch.uint8, device="cuda")
    c, b = tq.tq_lloyd_max_fit(x, init, 5, workspace=work, spin_limit=20000, absent_block=3)
    assert tq.tq_lloyd_max_fit_status(work) == 7  # TQ_ERR_TIMEOUT
    assert torch.isnan(c).all() and torch.isnan(b).all()
    c, b = tq.tq_lloyd_max_fit(x, init, 5, workspace=work)
    assert tq.tq_lloyd_max_fit_status(work) == 0
    assert not torch.isnan(c).any()
    check_chain(x.cpu().numpy(), init.cpu().numpy(), 5)
