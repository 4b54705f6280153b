"""Pins of the oracle's per-group V widths (layers grown by appends whose
blocks take the width the allocator chose when they were quantised; CoMixKV
article, section on the incremental quantisation strategy).

Checked against what the pages and the mathematics fix, not against the
oracle's own formulas: hand-derived layout bytes, the float64 nearest
centroid of each token's own table, the uniform layout as the special case
of equal widths, and the decompressed values of a group against those of a
layer made of that group alone."""

import os

import numpy as np
import pytest

from oracle import codec, lloyd_max
from oracle.attention import dequantise_f64, hadamard


def _golden(golden_dir):
    cases, cur = [], None
    with open(os.path.join(golden_dir, "pool_v_groups_layout.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "case":
                cur = dict(widths=[int(x) for x in t[1].split(",")], H=int(t[2]), ctx=int(t[3]), d=int(t[4]),
                           codes=[], bytes=[])
            elif t[0] == "code":
                cur["codes"].append(tuple(int(x) for x in t[1:]))
            elif t[0] == "byte":
                cur["bytes"].append(tuple(int(x, 0) for x in t[1:]))
            elif t[0] == "end":
                cases.append(cur)
    return cases


def test_group_layout_golden(golden_dir):
    cases = _golden(golden_dir)
    assert len(cases) == 2
    for c in cases:
        W, H, T, d = c["widths"], c["H"], c["ctx"], c["d"]
        codes = np.zeros((H, T, d), np.uint8)
        for h, t, i, v in c["codes"]:
            codes[h, t, i] = v
        want = np.zeros((H, d * 4 * sum(W)), np.uint8)
        for h, off, v in c["bytes"]:
            want[h, off] = v
        got = codec.pack_pool_v_groups(codes, W)
        assert got.shape == want.shape
        assert np.array_equal(got, want), np.argwhere(got != want)
        assert np.array_equal(codec.unpack_pool_v_groups(got, W, T, d), codes)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_equal_widths_are_the_uniform_layout(bits):
    """A layer whose groups all have width b stores exactly the uniform layer
    of width b (so appends at the create width change nothing)."""
    rng = np.random.default_rng(70 + bits)
    T, d = 100, 64
    K = codec.f32_to_bf16(rng.standard_normal((2, T, d)).astype(np.float32))
    V = codec.f32_to_bf16(rng.standard_normal((2, T, d)).astype(np.float32))
    mixed = codec.encode_layer_groups(K, V, [bits] * 4)
    uni = codec.encode_layer(K, V, bits, k_block=32)
    assert np.array_equal(mixed["packed"], uni["packed"].reshape(2, -1))
    for key in ("codes", "norms", "kq", "kscales"):
        assert np.array_equal(mixed[key], uni[key]), key


def test_group_codes_are_nearest_centroid_of_their_width():
    """Each token's codes are the float64 nearest centroid of y = Hv/|v| in
    the table of its own group's width (except within float32 rounding of a
    midpoint)."""
    widths = [2, 4, 3, 3, 2, 4]
    rng = np.random.default_rng(77)
    T, d = 6 * 32, 64
    V = codec.f32_to_bf16(rng.standard_normal((1, T, d)).astype(np.float32))
    K = codec.f32_to_bf16(rng.standard_normal((1, T, d)).astype(np.float32))
    enc = codec.encode_layer_groups(K, V, widths)
    v = codec.bf16_to_f32(V[0]).astype(np.float64)
    y = (v @ hadamard(d)) / np.linalg.norm(v, axis=1, keepdims=True)
    for g, b in enumerate(widths):
        c64, m64 = lloyd_max.lloyd_max_normal(1 << b)
        yy = y[g * 32:(g + 1) * 32]
        nearest = np.argmin(np.abs(yy[..., None] - c64), axis=-1)
        close = np.min(np.abs(yy[..., None] - m64), axis=-1) < 1e-5
        got = enc["codes"][0, g * 32:(g + 1) * 32]
        assert np.array_equal(got[~close], nearest[~close]), g
        assert got.max() < (1 << b)


def test_group_byte_count_and_offsets():
    """Per KV head, group g starts at byte sum_{g' < g} d * 4 * b_g' and the
    head holds exactly sum_g d * 4 * b_g bytes (no gap, no padding)."""
    widths = [3, 2, 4, 2]
    rng = np.random.default_rng(78)
    H, T, d = 2, 110, 128
    codes = np.zeros((H, T, d), np.uint8)
    for g, b in enumerate(widths):
        sl = slice(g * 32, min(T, g * 32 + 32))
        codes[:, sl] = rng.integers(0, 1 << b, size=codes[:, sl].shape)
    p = codec.pack_pool_v_groups(codes, widths)
    assert p.shape == (H, d * 4 * sum(widths))
    off = 0
    for g, b in enumerate(widths):
        n = d * 4 * b
        blk = p[:, off:off + n].reshape(H, 1, d, 4 * b)
        T_g = min(32, T - g * 32)
        assert np.array_equal(codec.unpack_pool_v(blk, b, T_g), codes[:, g * 32:g * 32 + T_g])
        off += n
    with pytest.raises(ValueError):
        codec.pack_pool_v_groups(codes, widths[:-1])


def test_mixed_dequantise_and_decompress_per_group():
    """Dequantised values and bf16 decompress of every group equal those of a
    layer made of that group's tokens alone at its width (block-scaled K
    depends on each token only)."""
    widths = [4, 2, 3]
    rng = np.random.default_rng(79)
    H, T, d = 2, 90, 64
    K = codec.f32_to_bf16(rng.standard_normal((H, T, d)).astype(np.float32))
    V = codec.f32_to_bf16((rng.standard_normal((H, T, d)) * rng.uniform(0.5, 3, (H, T, 1))).astype(np.float32))
    enc = codec.encode_layer_groups(K, V, widths)
    Kh, Vh = dequantise_f64(enc)
    Kd, Vd = codec.decompress_layer(enc)
    for g, b in enumerate(widths):
        sl = slice(g * 32, min(T, g * 32 + 32))
        one = codec.encode_layer(K[:, sl], V[:, sl], b, k_block=32)
        k1, v1 = dequantise_f64(one)
        kd1, vd1 = codec.decompress_layer(one)
        assert np.array_equal(Kh[:, sl], k1) and np.array_equal(Vh[:, sl], v1), g
        assert np.array_equal(Kd[:, sl], kd1) and np.array_equal(Vd[:, sl], vd1), g
    # coarser groups carry larger errors: the relative V error of each group
    # is near sqrt(D_b), the Lloyd-Max distortion of its width
    v = codec.bf16_to_f32(V).astype(np.float64)
    for g, b in enumerate(widths):
        sl = slice(g * 32, min(T, g * 32 + 32))
        rel = np.sum((Vh[:, sl] - v[:, sl]) ** 2) / np.sum(v[:, sl] ** 2)
        c, m = lloyd_max.lloyd_max_normal(1 << b)
        assert 0.6 < rel / lloyd_max.mse_normal(c, m) < 1.5, (b, rel)
