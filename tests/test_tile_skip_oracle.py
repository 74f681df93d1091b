"""Pins of the oracle's tile-skip rule (tile_pair_bound, tile_span) against
what the mathematics fixes: the bound is never below the exact quantity it
bounds (brute force over the full fp64 logits), it is attained exactly when
the scores vanish (the bias alone, which the foxwindow README's monotone decay
makes largest at the pair's nearest corner), a constant gate gives a closed
form for the span, an open gate skips nothing, and the span arrays describe
the same set of pairs from both sides."""
import math

import numpy as np
import pytest

from oracle import fox_oracle as ora


def _inputs(N, d, seed, gate_mean, gate_sd=0.5, score_sd=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, d)) * score_sd
    k = rng.standard_normal((N, d)) * score_sd
    z = gate_mean + gate_sd * rng.standard_normal(N)
    return q, k, z


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("N,d,gate_mean,scale", [(700, 64, 0.0, None), (513, 32, -1.0, None),
                                                 (640, 16, 2.0, -0.3), (390, 8, -4.0, 0.9)])
def test_bound_never_below_exact_excess(N, d, gate_mean, scale, from_j):
    q, k, z = _inputs(N, d, seed=N + d, gate_mean=gate_mean)
    U = ora.tile_pair_bound(q, k, z, scale, from_j)
    E = ora.tile_pair_excess(q, k, z, scale, from_j)
    lower = np.tril(np.ones_like(U, dtype=bool), k=-1)
    assert np.all(E[lower] <= U[lower] + 1e-9)
    assert np.all(np.isinf(U[~lower]))


@pytest.mark.parametrize("from_j", [False, True])
def test_bound_is_attained_with_zero_scores(from_j):
    """q = 0: x_ij - M_i = (colterm_i - colterm_j) log2 e, largest at (i0, j1)."""
    N, d = 600, 16
    _, k, z = _inputs(N, d, seed=5, gate_mean=0.5, gate_sd=1.0)
    q = np.zeros((N, d))
    U = ora.tile_pair_bound(q, k, z, None, from_j)
    E = ora.tile_pair_excess(q, k, z, None, from_j)
    lower = np.tril(np.ones_like(U, dtype=bool), k=-1)
    np.testing.assert_allclose(E[lower], U[lower], rtol=1e-12, atol=1e-9)


def test_bound_is_attained_by_the_scores():
    """d = 1, q = 1, keys +1 in tile 0 and -1 after it, a steep constant gate: for a row i0
    of tile I >= 1 the diagonal (-scale) is the row maximum and key j1 = 127 sits at
    +scale + (c_i0 - c_127), so the excess of pair (I, 0) is exactly
    scale log2e (kmax_0 + kmax_I) + (c_i0 - c_127) log2e: both score terms of the bound count."""
    N = 128 * 4
    q = np.ones((N, 1))
    k = np.where(np.arange(N) < 128, 1.0, -1.0)[:, None]
    z = np.full(N, -5.0)
    U = ora.tile_pair_bound(q, k, z, scale=1.0)
    E = ora.tile_pair_excess(q, k, z, scale=1.0)
    np.testing.assert_allclose(E[1:, 0], U[1:, 0], rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("from_j", [False, True])
@pytest.mark.parametrize("zc", [-0.5, 1.0, 3.0])
def test_constant_gate_span_closed_form(zc, from_j):
    """Constant gate a and zero scores: U(I, J) = a log2e (128 (I - J) - 127); pair (I, J)
    is negligible iff 128 (I - J) - 127 > thr / (|a| log2 e), so
    jmin(I) = max(0, I - g + 1) with g the smallest integer gap satisfying it."""
    N, d = 128 * 24 + 17, 8
    q = np.zeros((N, d))
    k = np.ones((N, d))
    z = np.full(N, zc)
    a = ora.log_forget_gate(np.array([zc]))[0]
    reach = ora.SKIP_THRESHOLD_LOG2 / (abs(a) * ora.LOG2E)
    g = math.floor((reach + 127) / 128) + 1  # smallest gap with 128 g - 127 > reach
    nT = (N + 127) // 128
    jmin, imax = ora.tile_span(q, k, z, None, from_j)
    expect = np.array([max(0, I - g + 1) for I in range(nT)])
    np.testing.assert_array_equal(jmin, expect)
    np.testing.assert_array_equal(imax, [min(nT - 1, J + g - 1) for J in range(nT)])


def test_open_gate_skips_nothing():
    q, k, _ = _inputs(900, 32, seed=3, gate_mean=0.0)
    z = np.full(900, np.inf)
    jmin, imax = ora.tile_span(q, k, z)
    assert np.all(jmin == 0) and np.all(imax == len(imax) - 1)


@pytest.mark.parametrize("gate_mean", [-2.0, 0.0, 1.5])
def test_span_arrays_agree(gate_mean):
    """jmin non-decreasing with jmin(I) <= I; imax(J) >= J; and the pair (I, J) is visited
    from the query side (jmin(I) <= J <= I) exactly when it is from the key side
    (J <= I <= imax(J)). Every pair left out is negligible under the bound."""
    N, d = 128 * 20 + 5, 32
    q, k, z = _inputs(N, d, seed=11, gate_mean=gate_mean)
    jmin, imax = ora.tile_span(q, k, z)
    nT = len(jmin)
    assert np.all(np.diff(jmin) >= 0) and np.all(jmin <= np.arange(nT)) and np.all(imax >= np.arange(nT))
    U = ora.tile_pair_bound(q, k, z)
    for I in range(nT):
        for J in range(I + 1):
            assert (jmin[I] <= J) == (I <= imax[J])
            if J < jmin[I]:
                assert U[I, J] < -ora.SKIP_THRESHOLD_LOG2
