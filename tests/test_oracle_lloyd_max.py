"""Pins of the oracle's Lloyd-Max tables (CPU only).

The tables are pinned to things other than the iteration that produced them:
the optimality conditions with conditional means re-derived by numerical
quadrature (scipy), J. Max's 1960 published table, the MSE by quadrature and by
Monte Carlo, and exact antisymmetry.
"""

import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import lloyd_max

pytestmark = pytest.mark.filterwarnings("ignore::scipy.integrate.IntegrationWarning")


def _phi(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _read_max(golden_dir):
    table = {}
    with open(os.path.join(golden_dir, "lloyd_max_max1960.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            table[(int(parts[0]), parts[1])] = [float(v) for v in parts[2:]]
    return table


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_centroid_condition_by_quadrature(levels):
    c, m = lloyd_max.lloyd_max_normal(levels)
    edges = [-np.inf] + list(m) + [np.inf]
    for k in range(levels):
        a, b = edges[k], edges[k + 1]
        num = integrate.quad(lambda x: x * _phi(x), a, b, epsabs=1e-15, epsrel=1e-13)[0]
        den = integrate.quad(_phi, a, b, epsabs=1e-15, epsrel=1e-13)[0]
        assert abs(num / den - c[k]) < 1e-12, (levels, k)


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_midpoint_condition_and_order(levels):
    c, m = lloyd_max.lloyd_max_normal(levels)
    assert np.all(np.diff(c) > 0)
    np.testing.assert_allclose(m, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    assert np.all(c[:-1] < m) and np.all(m < c[1:])


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_exact_antisymmetry(levels):
    c, m = lloyd_max.lloyd_max_normal(levels)
    assert np.array_equal(c, -c[::-1])
    assert m[levels // 2 - 1] == 0.0
    for bits in (2, 3, 4):
        cf, mf = lloyd_max.tables_f32(bits)
        assert np.array_equal(cf, -cf[::-1]) and mf[len(mf) // 2] == 0.0


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_against_max_1960_table(levels, golden_dir):
    table = _read_max(golden_dir)
    c, m = lloyd_max.lloyd_max_normal(levels)
    half = levels // 2
    # Max prints 4 significant digits
    np.testing.assert_allclose(c[half:], table[(levels, "output")], rtol=6e-4, atol=1e-4)
    if (levels, "threshold") in table:
        np.testing.assert_allclose(m[half - 1:], table[(levels, "threshold")], rtol=6e-4, atol=1e-4)
    mse = lloyd_max.mse_normal(c, m)
    assert abs(mse - table[(levels, "mse")][0]) / table[(levels, "mse")][0] < 1e-3


@pytest.mark.parametrize("levels", [4, 8, 16])
def test_mse_by_quadrature(levels):
    c, m = lloyd_max.lloyd_max_normal(levels)
    edges = [-np.inf] + list(m) + [np.inf]
    q = sum(integrate.quad(lambda x: (x - c[k]) ** 2 * _phi(x), edges[k], edges[k + 1],
                           epsabs=1e-15, epsrel=1e-12)[0] for k in range(levels))
    assert abs(q - lloyd_max.mse_normal(c, m)) < 1e-12


def test_mse_monte_carlo_8_levels():
    """8 levels: MSE ~ 0.0345 on N(0,1) samples, within 4 standard errors."""
    c, m = lloyd_max.lloyd_max_normal(8)
    x = np.random.default_rng(12345).standard_normal(4_000_000)
    err = (x - c[np.searchsorted(m, x)]) ** 2
    mse = lloyd_max.mse_normal(c, m)
    assert abs(err.mean() - mse) < 4 * err.std() / math.sqrt(len(x))
    assert abs(mse - 0.0345) < 1e-4


def test_lloyd_max_is_a_local_minimum():
    """Moving any output or threshold increases the MSE (a dropped term or a
    wrong sign in the update formula would not survive this)."""
    c, m = lloyd_max.lloyd_max_normal(8)
    base = lloyd_max.mse_normal(c, m)
    for k in range(8):
        for eps in (1e-3, -1e-3):
            c2 = c.copy()
            c2[k] += eps
            assert lloyd_max.mse_normal(c2, m) > base
    for k in range(7):
        for eps in (1e-3, -1e-3):
            m2 = m.copy()
            m2[k] += eps
            assert lloyd_max.mse_normal(c, m2) > base


def test_float32_tables_are_single_roundings():
    for bits in (2, 3, 4):
        c, m = lloyd_max.lloyd_max_normal(1 << bits)
        cf, mf = lloyd_max.tables_f32(bits)
        assert cf.dtype == np.float32 and mf.dtype == np.float32
        assert np.array_equal(cf, c.astype(np.float32))
        assert np.array_equal(mf, (0.5 * (c[:-1] + c[1:])).astype(np.float32))
