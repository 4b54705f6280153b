"""The library's bit allocator (host code of the C-ABI, no GPU): the same
allocations as the oracle's exact dynamic programme, and its argument
checks."""

import numpy as np
import pytest

from oracle import allocator


@pytest.fixture(scope="module")
def kp():
    from shared_quantized_kv_gb300 import build, kvpool

    build.build()
    return kvpool


def test_library_distortions_equal_oracle(kp):
    # the widths are chosen from the library's own Lloyd-Max distortions:
    # equal layer costs and sensitivities whose ratio crosses D_2/D_3 decide
    # the upgrade order exactly as the oracle's distortions do
    rng = np.random.default_rng(11)
    for _ in range(200):
        L = int(rng.integers(1, 9))
        sens = rng.uniform(0.01, 2.0, L)
        cost = rng.integers(1, 7, L)
        budget = int(rng.integers(2 * cost.sum(), 4 * cost.sum() + 3))
        assert kp.allocate_bits(sens, cost, budget) == list(allocator.allocate(list(sens), list(cost), budget))


def test_large_pools_and_units(kp):
    # 64 layers with byte costs (the greatest common divisor becomes the unit)
    rng = np.random.default_rng(12)
    sens = rng.lognormal(0, 0.7, 64)
    cost = np.full(64, 8 * 4096 * 128 // 8, dtype=np.int64)  # V bytes per bit of a Llama-4K layer
    budget = int(3 * cost.sum())
    bits = kp.allocate_bits(sens, cost, budget)
    assert bits == list(allocator.allocate(list(sens), [1] * 64, 3 * 64))
    assert sum(b * c for b, c in zip(bits, cost)) <= budget


def test_argument_checks(kp):
    with pytest.raises(kp.KVPoolError):
        kp.allocate_bits([0.5, 0.5], [4, 4], 15)  # below 2 bits everywhere
    with pytest.raises(kp.KVPoolError):
        kp.allocate_bits([0.5, -1.0], [4, 4], 24)
    with pytest.raises(kp.KVPoolError):
        kp.allocate_bits([0.5, 0.5], [0, 4], 24)
    assert kp.allocate_bits([0.5, 0.5], [4, 4], 16) == [2, 2]
    assert kp.allocate_bits([0.5, 0.5], [4, 4], 10 ** 9) == [4, 4]
