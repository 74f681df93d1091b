"""Pins of the oracle's epsilon-effective window (foxwindow README) against
what the page prints and what renewal theory fixes."""
import math
import os

import numpy as np
import pytest

from oracle import fox_oracle as ora

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "foxwindow_alibi_limit.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            m, eps, printed = line.split()
            rows.append((float(m), float(eps), float(printed)))
    return rows


@pytest.mark.parametrize("m,eps,printed", _golden())
def test_alibi_limit_matches_printed_values(m, eps, printed):
    """Constant gate e^{-m}: every increment is m, so the first passage over L is
    floor(L/m) + 1 for every row with enough history; L/m is the page's printed value."""
    L = math.log(1.0 / eps)
    assert round(L / m, 1) == printed
    N = 400
    z = np.full(N, -math.log(math.expm1(m)))
    w = ora.effective_window(z, eps)
    expect = math.floor(L / m) + 1
    hist = np.arange(N) + 1  # increments available to row i
    np.testing.assert_array_equal(w[hist >= expect], expect)
    np.testing.assert_array_equal(w[hist < expect], -1)


def test_open_gate_never_passes():
    assert np.all(ora.effective_window(np.full(50, np.inf), 1e-3) == -1)


def test_window_brute_force_on_tiny_input():
    z = np.array([0.3, -1.0, 2.0, 0.5, -0.2, 4.0])
    X = np.log1p(np.exp(-z))  # -log sigmoid(z)
    L = math.log(1 / 0.2)
    w = ora.effective_window(z, 0.2)
    for i in range(len(z)):
        sums = np.cumsum(X[: i + 1][::-1])
        hit = np.nonzero(sums > L)[0]
        assert w[i] == (hit[0] + 1 if hit.size else -1)


def test_window_grows_with_smaller_epsilon():
    r = np.random.default_rng(3)
    z = r.normal(2.0, 1.0, 3000)
    inf = lambda w: np.where(w < 0, np.inf, w)  # -1: not reached inside the sequence
    prev = inf(ora.effective_window(z, 0.5))
    for eps in (0.1, 1e-2, 1e-3):
        cur = inf(ora.effective_window(z, eps))
        assert np.all(cur >= prev)
        prev = cur


def test_renewal_laws_for_exponential_increments():
    """Exponential increments (rate lam) make the walk a Poisson process, where the page's
    two-moment law E[N] = L/k + E[X^2]/(2 k^2) and Var[N] = s^2 L / k^3 are exact:
    E[N] = lam L + 1, Var[N] = lam L. Checked on independent walks (one row per walk)."""
    lam, eps = 3.0, 1e-3
    L = math.log(1 / eps)
    kappa, s2 = 1 / lam, 1 / lam**2
    mean_law = L / kappa + (s2 + kappa**2) / (2 * kappa**2)
    var_law = s2 * L / kappa**3
    assert mean_law == pytest.approx(lam * L + 1) and var_law == pytest.approx(lam * L)
    r = np.random.default_rng(11)
    walks, length = 20000, 64
    X = r.exponential(1 / lam, size=(walks, length))
    z = -np.log(np.expm1(X))  # sigmoid(z) = e^{-X}
    N = np.array([ora.effective_window(z[w], eps)[-1] for w in range(walks)])
    assert np.all(N > 0)
    se = math.sqrt(var_law / walks)
    assert abs(N.mean() - mean_law) < 5 * se
    assert abs(N.var() - var_law) < 0.05 * var_law


def test_rows_subset_matches_full():
    r = np.random.default_rng(5)
    z = r.normal(1.0, 2.0, 500)
    full = ora.effective_window(z, 1e-2)
    rows = [0, 3, 250, 499]
    np.testing.assert_array_equal(ora.effective_window(z, 1e-2, rows=rows), full[rows])
