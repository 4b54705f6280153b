"""Lloyd-Max scalar quantiser for the standard normal density.

Source: PolyKV summary, section 2.B -- rotated V coordinates are mapped to
"pre-computed Lloyd-Max centroids optimised for N(0, 1)"; 3 bits (8 levels).
CoMixKV article: 2 to 4 bits per layer, hence 4 and 16 levels as well.

The quantiser is the textbook one (J. Max, "Quantizing for minimum distortion",
IRE Trans. Information Theory, 1960): thresholds are midpoints of adjacent
outputs, and every output is the conditional mean of N(0, 1) over its cell.
N(0, 1) is symmetric, so for an even number of levels the middle threshold is 0
and only the positive half is iterated (Max computed his tables the same way);
this also makes the table exactly antisymmetric, so a zero coordinate falls on
the threshold 0 on every machine.

Pinned by tests/test_oracle_lloyd_max.py: the centroid and midpoint conditions
(with the conditional means re-derived by numerical quadrature), Max's
published values, the MSE by quadrature and by Monte Carlo.
"""

from __future__ import annotations

import functools
import math

import numpy as np

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def _phi(x: float) -> float:
    """N(0,1) density."""
    if math.isinf(x):
        return 0.0
    return _INV_SQRT_2PI * math.exp(-0.5 * x * x)


def _upper_tail(x: float) -> float:
    """P(X > x) for X ~ N(0,1), accurate in the upper tail."""
    if math.isinf(x):
        return 0.0 if x > 0 else 1.0
    return 0.5 * math.erfc(x / _SQRT2)


def lloyd_max_normal(levels: int, tol: float = 1e-16, max_iter: int = 20000):
    """Return (centroids, thresholds) in float64 for ``levels`` in {2, 4, 8, 16}.

    ``centroids`` is ascending, length ``levels``; ``thresholds`` has the
    ``levels - 1`` interior cell boundaries (midpoints of adjacent centroids).

    Positive half: outputs y_1 < ... < y_K (K = levels/2) over cells
    [x_{k-1}, x_k) with x_0 = 0 and x_K = +inf. Lloyd's iteration alternates
      y_k = E[X | x_{k-1} <= X < x_k] = (phi(x_{k-1}) - phi(x_k)) / (Q(x_{k-1}) - Q(x_k))
      x_k = (y_k + y_{k+1}) / 2
    where Q is the upper-tail probability, until no value moves by more than
    ``tol`` (relative), starting from cells of equal probability.
    """
    if levels not in (2, 4, 8, 16):
        raise ValueError("levels must be 2, 4, 8 or 16")
    K = levels // 2
    # start: equal-probability cells on the positive half
    x = [0.0]
    for k in range(1, K):
        p = 0.5 - 0.5 * k / K  # upper tail mass above x_k
        lo, hi = 0.0, 10.0
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            if _upper_tail(mid) > p:
                lo = mid
            else:
                hi = mid
        x.append(0.5 * (lo + hi))
    x.append(math.inf)
    y = [0.0] * K
    for _ in range(max_iter):
        y_new = [(_phi(x[k]) - _phi(x[k + 1])) / (_upper_tail(x[k]) - _upper_tail(x[k + 1]))
                 for k in range(K)]
        x_new = [0.0] + [0.5 * (y_new[k] + y_new[k + 1]) for k in range(K - 1)] + [math.inf]
        delta = max(abs(a - b) / max(abs(a), 1e-300) for a, b in zip(y_new, y))
        y, x = y_new, x_new
        if delta <= tol:
            break
    pos = np.array(y, dtype=np.float64)
    centroids = np.concatenate([-pos[::-1], pos])
    thresholds = 0.5 * (centroids[:-1] + centroids[1:])
    return centroids, thresholds


def mse_normal(centroids: np.ndarray, thresholds: np.ndarray) -> float:
    """Mean squared error of the quantiser on N(0,1), in closed form per cell:
    E[(X - c)^2; a<X<b] = P(cell)(1 + c^2) - 2c(phi(a)-phi(b)) + (a phi(a) - b phi(b))."""
    edges = [-math.inf] + list(map(float, thresholds)) + [math.inf]
    total = 0.0
    for k, c in enumerate(map(float, centroids)):
        a, b = edges[k], edges[k + 1]
        p = _upper_tail(a) - _upper_tail(b)
        pa, pb = _phi(a), _phi(b)
        apa = 0.0 if math.isinf(a) else a * pa
        bpb = 0.0 if math.isinf(b) else b * pb
        total += p * (1.0 + c * c) - 2.0 * c * (pa - pb) + (apa - bpb)
    return total


@functools.lru_cache(maxsize=None)
def _tables_f32(bits: int):
    c, m = lloyd_max_normal(1 << bits)
    return c.astype(np.float32), m.astype(np.float32)


def tables_f32(bits: int):
    """The stored tables of a ``bits``-bit V code: float32 centroids (ascending,
    2**bits values) and float32 midpoints (2**bits - 1 values), each midpoint
    being (c_k + c_{k+1}) / 2 computed in float64 and then rounded once."""
    c, m = _tables_f32(bits)
    return c.copy(), m.copy()
