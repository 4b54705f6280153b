"""The numbers the PolyKV summary prints, reproduced from the oracle's storage
formula (CPU only): the 16/5.5 compression ratio of section 2.B and the 97.7%
memory reduction for 15 agents of section 4."""

import os

import pytest

from oracle import codec


def _golden(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "polykv_printed_numbers.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_theoretical_ratio(golden_dir):
    g = _golden(golden_dir)
    ratio = g["ratio_baseline_bits"] / ((g["ratio_k_bits"] + g["ratio_v_bits"]) / 2)
    assert round(ratio, 2) == g["ratio_printed"]
    # the oracle's payload bytes per (token, head) without the per-vector norm
    # give exactly 16 / 5.5 against bf16 K + V
    d = 128
    payload = d + d * 3 // 8
    assert 4 * d / payload == pytest.approx(16 / 5.5, rel=1e-12)


@pytest.mark.parametrize("d,ratio", [(128, 512 / 180), (64, 256 / 92)])
def test_ratio_with_norm_overhead(d, ratio):
    """A float32 norm per head-vector is the scale overhead of the V code."""
    hk, t = 8, 4096
    full = 2 * hk * t * d * 2
    stored = codec.layer_bytes(hk, t, d, 3)
    assert full / stored == pytest.approx(ratio, rel=1e-5)


def test_reduction_for_fifteen_agents(golden_dir):
    g = _golden(golden_dir)
    n = g["agents"]
    # one shared pool against n private full-precision caches: 1 - 1/(n * ratio)
    for ratio in (16 / 5.5, 512 / 180):
        assert round(100 * (1 - 1 / (n * ratio)), 1) == g["reduction_printed_pct"]
    # the printed sizes are consistent with the same arithmetic
    assert round(100 * (1 - g["pool_gb"] / g["full_gb"]), 1) == g["reduction_printed_pct"]
    assert g["full_gb"] / g["pool_gb"] / n == pytest.approx(16 / 5.5, rel=0.02)


def test_pool_size_independent_of_agents(golden_dir):
    g = _golden(golden_dir)
    assert g["pool_2k_gb_3_agents"] == g["pool_2k_gb_10_agents"]
    # the oracle's stored bytes take no agent count at all
    assert codec.layer_bytes.__code__.co_varnames[:4] == ("kv_heads", "ctx", "head_dim", "bits")
