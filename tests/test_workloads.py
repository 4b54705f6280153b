"""Seeded input generators (CPU only): determinism, shapes, bf16 rounding and
the stated channel statistics."""

import struct

import numpy as np

from shared_quantized_kv_gb300 import workloads as wl


def test_configs_shapes():
    W = wl.WORKLOADS
    assert [w.index for w in W.values()] == [0, 1, 2, 3, 4]
    assert W["llama3_8b_4k"].rows == 60 and W["qwen3_32b_32k"].rows == 256
    assert W["smollm2_2k"].rows == 10 and W["tiny"].rows == 6
    b = W["qwen3_32b_32k"].bits_list()
    assert len(b) == 64 and sum(b) == 3 * 64 and {b.count(2), b.count(3), b.count(4)} == {21, 22}
    lw = W["llama3_8b_long"]
    assert [lw.tail_len(s) for s in range(4)] == [129, 130, 131, 132] and lw.tail_max == 132


def test_bf16_rounding_by_hand():
    for v in (1.0, 3.14159265, -0.1, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1e30):
        b = struct.unpack("<I", struct.pack("<f", v))[0]
        lo, hi = b & 0xFFFF, b >> 16
        if lo > 0x8000 or (lo == 0x8000 and hi & 1):
            hi += 1
        assert wl.f32_to_bf16_bits(np.array([v], np.float32))[0] == hi


def test_deterministic_and_distinct():
    w = wl.WORKLOADS["tiny"]
    K1, V1 = wl.layer_kv(w, 0)
    K2, V2 = wl.layer_kv(w, 0)
    assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
    assert not np.array_equal(K1, V1)
    assert not np.array_equal(wl.layer_q(w, 0, 0), wl.layer_q(w, 0, 1))
    assert K1.shape == (2, 256, 64) and K1.dtype == np.uint16


def test_tiny_outlier_channels():
    w = wl.WORKLOADS["tiny"]
    K, _ = wl.layer_kv(w, 0)
    k = wl.bf16_bits_to_f32(K)
    std = k.std(axis=1)  # [head, channel]
    for h in range(2):
        assert (std[h] > 4).sum() == 2


def test_lognormal_statistics():
    w = wl.custom(kv_heads=4, head_dim=64, ctx=2048)
    K, _ = wl.layer_kv(w, 0)
    k = wl.bf16_bits_to_f32(K)
    std = k.std(axis=1)
    n_out = int(round(0.01 * 4 * 64))
    assert n_out == 3
    logs = np.log(np.sort(std.ravel())[:-n_out])
    assert abs(logs.mean()) < 0.15 and abs(logs.std() - 0.5) < 0.1
