"""Pins of oracle/allocator.py (the local attention-error estimate and the
per-layer bit allocation; the pages print no formula, so these pin the
reading against mathematics: published Lloyd-Max distortions, closed forms,
a Monte-Carlo check of the error prediction against the oracle's own codec,
and brute force for the allocation)."""

import math

import numpy as np
import pytest

from oracle import allocator, attention, codec


def test_distortions_match_max_1960():
    # J. Max (1960), minimum mean squared error for N(0,1) at 4, 8 and 16
    # levels, to the precision of his table (his 16-level entry 0.009497 is
    # 4e-6 below the converged value; the output levels agree to every digit)
    assert allocator.distortion(2) == pytest.approx(0.1175, abs=1e-4)
    assert allocator.distortion(3) == pytest.approx(0.03454, abs=1e-5)
    assert allocator.distortion(4) == pytest.approx(0.009497, abs=1e-5)


def test_row_ratio_closed_forms():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(64)
    q = rng.standard_normal(64)
    # one token: p = 1, o = v
    assert allocator.row_ratio(q, v[None], v[None], 0.125) == pytest.approx(1.0)
    # T equal logits (q orthogonal to every key) on one repeated vector: 1/sqrt(T)
    K = np.zeros((16, 64))
    assert allocator.row_ratio(q, K, np.tile(v, (16, 1)), 0.125) == pytest.approx(1 / 4)
    # two equal-weight orthogonal values of equal norm: |o|^2 = sum p^2 |v|^2
    e1, e2 = np.eye(64)[0] * 3, np.eye(64)[1] * 3
    assert allocator.row_ratio(q, np.zeros((2, 64)), np.stack([e1, e2]), 0.125) == pytest.approx(1.0)
    assert allocator.row_ratio(q, np.zeros((0, 64)), np.zeros((0, 64)), 0.125) == 0.0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_error_prediction_tracks_quantised_v(bits):
    # E|o - o_hat| / |o| against sqrt(D_b) * r, with V coded by the pool's own
    # V codec (FWHT, norm, Lloyd-Max) over many random rows
    rng = np.random.default_rng(bits)
    d, T = 64, 48
    meas, pred = [], []
    for _ in range(200):
        q = rng.standard_normal(d)
        K = rng.standard_normal((T, d))
        V = codec.f32_to_bf16(rng.standard_normal((1, T, d)).astype(np.float32))
        codes, norms = codec.v_codes(V, bits)
        Vh = attention.dequantise_f64(dict(bits=bits, codes=codes, norms=norms, kq=np.zeros((1, T, d), np.int8),
                                           scale=np.float32(1)))[1][0]
        v = codec.bf16_to_f32(V)[0].astype(np.float64)
        lg = 0.3 * (K @ q)
        p = np.exp(lg - lg.max())
        p /= p.sum()
        o, oh = p @ v, p @ Vh
        meas.append(np.sum((o - oh) ** 2) / np.sum(o ** 2))
        pred.append((allocator.layer_error(allocator.row_ratio(q, K, v, 0.3), bits)) ** 2)
    ratio = math.sqrt(np.mean(meas) / np.mean(pred))
    assert 0.8 < ratio < 1.25, ratio


def test_allocation_equals_brute_force():
    rng = np.random.default_rng(7)
    for _ in range(40):
        L = int(rng.integers(1, 6))
        sens = list(rng.uniform(0.05, 1.0, L))
        cost = list(rng.integers(1, 5, L))
        budget = int(rng.integers(2 * sum(cost), 4 * sum(cost) + 1))
        assert allocator.allocate(sens, cost, budget) == allocator.allocate_brute_force(sens, cost, budget)


def test_allocation_extremes_and_monotonicity():
    sens = [0.9, 0.1, 0.5, 0.3]
    cost = [3, 3, 3, 3]
    assert allocator.allocate(sens, cost, 4 * 12) == (4, 4, 4, 4)
    assert allocator.allocate(sens, cost, 2 * 12) == (2, 2, 2, 2)
    assert allocator.allocate(sens, cost, 2 * 12 - 1) is None
    # average 3 bits with equal costs: the more sensitive layers get more bits
    bits = allocator.allocate(sens, cost, 3 * 12)
    order = np.argsort(sens)
    assert all(bits[order[i]] <= bits[order[i + 1]] for i in range(3))
    assert sum(bits) == 12


def test_layer_sensitivity_mean_over_rows():
    rng = np.random.default_rng(3)
    A, Hk, Hq, T, d = 2, 2, 4, 10, 64
    Q = codec.f32_to_bf16(rng.standard_normal((A, Hq, d)).astype(np.float32))
    K = codec.f32_to_bf16(rng.standard_normal((A, Hk, T, d)).astype(np.float32))
    V = codec.f32_to_bf16(rng.standard_normal((A, Hk, T, d)).astype(np.float32))
    lens = np.array([T, 4])
    s = allocator.layer_sensitivity(Q, K, V, lens)
    q, k, v = (codec.bf16_to_f32(x).astype(np.float64) for x in (Q, K, V))
    rows = [allocator.row_ratio(q[a, h], k[a, h // 2, :lens[a]], v[a, h // 2, :lens[a]], 1 / 8)
            for a in range(A) for h in range(Hq)]
    assert s == pytest.approx(np.mean(rows))
    assert s > 0
    # values that cancel in o raise r above 1 (errors do not cancel)
    w = np.ones(64)
    assert allocator.row_ratio(np.zeros(64), np.zeros((2, 64)), np.stack([w, -0.9 * w]), 1.0) > 5
