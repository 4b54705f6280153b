"""Pins of the oracle's encode / decompress (CPU only).

Independent checks: an exact rational model of IEEE float32 (round to nearest,
ties to even, written here from the definition with ``fractions.Fraction``) run
over the stated operation order on tiny inputs; closed forms of the
Walsh-Hadamard transform; spike vectors with a known decoded value;
hand-derived packing bytes; the quantisation error bound of the int8 K code;
agreement of the codes with the float64 nearest centroid of y = Hv / |v|.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codec, lloyd_max
from oracle.attention import dequantise_f64, hadamard


# ------------------------------------------------- exact float32 model (pin)

def rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest float32 (ties to even)."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * n * ulp


def F(x) -> Fraction:
    return Fraction(float(x))


def rational_fwht(v):
    x = [F(t) for t in v]
    d = len(x)
    h = 1
    while h < d:
        for i in range(d):
            if i & h == 0:
                a, b = x[i], x[i + h]
                x[i], x[i + h] = rn32(a + b), rn32(a - b)
        h *= 2
    return x


def rational_norm(v):
    sq = [rn32(F(t) * F(t)) for t in v]
    w = len(sq) // 2
    while w >= 1:
        for i in range(w):
            sq[i] = rn32(sq[i] + sq[i + w])
        w //= 2
    return float(rn32(Fraction(math.sqrt(float(sq[0])))))  # sqrt of a float32 is correctly rounded in float64 then to 32


def _wide_range_f32(rng, shape):
    mant = rng.uniform(-1, 1, size=shape)
    expo = rng.integers(-20, 20, size=shape)
    return (mant * np.exp2(expo)).astype(np.float32)


# ---------------------------------------------------------------- transforms

@pytest.mark.parametrize("d", [2, 4, 8, 16, 32])
def test_fwht_matches_exact_float32_model(d):
    rng = np.random.default_rng(d)
    for _ in range(20):
        v = _wide_range_f32(rng, d)
        got = codec.fwht_f32(v)
        want = np.array([float(t) for t in rational_fwht(v)], dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_fwht_stage_order_is_observable():
    """The stated order (h = 1 first) and the reverse order round differently
    on some inputs, so the exact-model test above does pin the order."""
    rng = np.random.default_rng(7)
    differs = 0
    for _ in range(200):
        v = _wide_range_f32(rng, 8)
        fwd = codec.fwht_f32(v)
        x = v.astype(np.float32).copy()
        h = 4
        while h >= 1:
            y = x.reshape(8 // (2 * h), 2, h)
            a, b = y[:, 0, :].copy(), y[:, 1, :].copy()
            y[:, 0, :], y[:, 1, :] = a + b, a - b
            x = y.reshape(8)
            h //= 2
        differs += int(not np.array_equal(fwd, x))
    assert differs > 0


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_closed_forms(d):
    H = hadamard(d)
    eye = np.eye(d, dtype=np.float32)
    # H e_k is row k of H, exactly; applying twice gives d e_k exactly
    np.testing.assert_array_equal(codec.fwht_f32(eye), H.astype(np.float32))
    np.testing.assert_array_equal(codec.fwht_f32(codec.fwht_f32(eye)), d * eye)
    # H_ij = (-1)^popcount(i & j)
    for i in range(0, d, 7):
        for j in range(0, d, 5):
            assert H[i, j] == (-1) ** bin(i & j).count("1")
    # orthogonality on random vectors
    v = np.random.default_rng(1).standard_normal((100, d)).astype(np.float32)
    u = codec.fwht_f32(v).astype(np.float64)
    np.testing.assert_allclose((u ** 2).sum(1), d * (v.astype(np.float64) ** 2).sum(1), rtol=1e-5)


@pytest.mark.parametrize("d", [8, 16, 64])
def test_norm_matches_exact_float32_model(d):
    rng = np.random.default_rng(100 + d)
    for _ in range(20):
        v = _wide_range_f32(rng, d)
        got = codec.norm_f32(v)
        assert got == np.float32(rational_norm(v))


def test_norm_exact_on_integers():
    v = np.arange(-32, 32, dtype=np.float32)
    assert codec.norm_f32(v) == np.float32(math.sqrt(float((v.astype(np.float64) ** 2).sum())))


# ---------------------------------------------------------------------- bf16

def test_bf16_round_trip_and_rounding():
    import struct
    vals = [1.0, -2.5, 3.14159, 1e-3, 65504.0, 1.00390625, 1.0078125 + 2 ** -9]
    for v in vals:
        b32 = struct.unpack("<I", struct.pack("<f", v))[0]
        # ties-to-even rounding of the low 16 bits, written out by hand
        lo, hi = b32 & 0xFFFF, b32 >> 16
        if lo > 0x8000 or (lo == 0x8000 and hi & 1):
            hi += 1
        assert int(codec.f32_to_bf16(np.float32(v))) == hi
        assert codec.bf16_to_f32(np.uint16(hi)) == struct.unpack("<f", struct.pack("<I", hi << 16))[0]


# --------------------------------------------------------------------- K codec

def test_k_codec_brute_force_tiny():
    rng = np.random.default_rng(3)
    K = codec.f32_to_bf16(rng.standard_normal((2, 5, 8)).astype(np.float32) * 3)
    absmax, s = codec.k_scale(K)
    q = codec.k_quantize(K, s)
    k = codec.bf16_to_f32(K).astype(np.float64).ravel()
    am = max(abs(t) for t in k)
    assert absmax == am
    s_exact = rn32(Fraction(am) / 127)
    assert Fraction(float(s)) == s_exact
    for t, qt in zip(k, q.ravel()):
        quot = float(rn32(Fraction(t) / s_exact))
        assert qt == max(-127, min(127, round(quot)))  # Python round(): ties to even


def test_k_codec_error_bound_and_extremes():
    rng = np.random.default_rng(4)
    K = codec.f32_to_bf16(rng.standard_normal((4, 64, 32)).astype(np.float32) * 7)
    absmax, s = codec.k_scale(K)
    q = codec.k_quantize(K, s)
    k = codec.bf16_to_f32(K).astype(np.float64)
    err = np.abs(k - q.astype(np.float64) * float(s))
    assert err.max() <= 0.5 * float(s) * (1 + 1e-5)
    i = np.argmax(np.abs(k))
    assert abs(int(q.ravel()[i])) == 127
    assert q.min() >= -127 and q.max() <= 127
    assert np.all(np.sign(q) * np.sign(k) >= 0)


def test_k_codec_zero_and_nonfinite():
    z = np.zeros((1, 3, 8), np.uint16)
    absmax, s = codec.k_scale(z)
    assert absmax == 0 and s == 1
    assert not codec.k_quantize(z, s).any()
    bad = z.copy()
    bad[0, 1, 2] = 0x7F80  # +inf
    with pytest.raises(ValueError):
        codec.k_scale(bad)


def test_k_decompress_definition():
    q = np.array([[-127, -1, 0, 1, 64, 127]], np.int8)
    s = np.float32(0.0123)
    out = codec.bf16_to_f32(codec.k_dequantize_bf16(q, s))
    for qi, o in zip(q.ravel(), out.ravel()):
        p = rn32(Fraction(int(qi)) * F(s))
        assert o == codec.bf16_to_f32(codec.f32_to_bf16(np.float32(float(p))))


# --------------------------------------------------------------------- V codec

def _golden_packing(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "packing_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            left, right = line.split("->")
            nums = [int(t) for t in left.split()]
            rows.append((nums[0], nums[1:], [int(t, 16) for t in right.split()]))
    return rows


def test_packing_golden(golden_dir):
    for bits, codes, want in _golden_packing(golden_dir):
        c = np.array([codes], np.uint8)
        assert codec.pack_codes(c, bits).ravel().tolist() == want
        assert np.array_equal(codec.unpack_codes(codec.pack_codes(c, bits), bits, len(codes)), c)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_packing_round_trip_random(bits):
    rng = np.random.default_rng(bits)
    c = rng.integers(0, 1 << bits, size=(3, 5, 64), dtype=np.uint8)
    p = codec.pack_codes(c, bits)
    assert p.shape == (3, 5, 64 * bits // 8)
    assert np.array_equal(codec.unpack_codes(p, bits, 64), c)


def _golden_pool_layout(golden_dir):
    cases, cur = [], None
    with open(os.path.join(golden_dir, "pool_v_layout.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "case":
                cur = dict(bits=int(t[1]), H=int(t[2]), ctx=int(t[3]), d=int(t[4]), codes=[], bytes=[])
            elif t[0] == "code":
                cur["codes"].append(tuple(int(x) for x in t[1:]))
            elif t[0] == "byte":
                cur["bytes"].append(tuple(int(x, 0) for x in t[1:]))
            elif t[0] == "end":
                cases.append(cur)
    return cases


def test_pool_v_layout_golden(golden_dir):
    cases = _golden_pool_layout(golden_dir)
    assert len(cases) == 4
    for c in cases:
        bits, H, T, d = c["bits"], c["H"], c["ctx"], c["d"]
        codes = np.zeros((H, T, d), np.uint8)
        for h, t, i, v in c["codes"]:
            codes[h, t, i] = v
        want = np.zeros((H, -(-T // 32), d, 4 * bits), np.uint8)
        for h, g, i, b, v in c["bytes"]:
            want[h, g, i, b] = v
        got = codec.pack_pool_v(codes, bits)
        assert got.shape == want.shape
        assert np.array_equal(got, want), np.argwhere(got != want)
        assert np.array_equal(codec.unpack_pool_v(got, bits, T), codes)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pool_v_layout_round_trip_ragged(bits):
    rng = np.random.default_rng(40 + bits)
    for T in (1, 31, 32, 33, 100, 128):
        c = rng.integers(0, 1 << bits, size=(2, T, 64), dtype=np.uint8)
        p = codec.pack_pool_v(c, bits)
        assert p.shape == (2, -(-T // 32), 64, 4 * bits)
        assert np.array_equal(codec.unpack_pool_v(p, bits, T), c)
        # the padded token slots of the last group decode to code 0
        full = codec.unpack_pool_v(p, bits, p.shape[1] * 32)
        assert not full[:, T:].any()


def test_v_codes_match_exact_float32_model():
    rng = np.random.default_rng(9)
    for bits in (2, 3, 4):
        _, mid = lloyd_max.tables_f32(bits)
        for _ in range(5):
            v32 = rng.standard_normal(16).astype(np.float32) * np.float32(rng.uniform(0.1, 10))
            V = codec.f32_to_bf16(v32)
            codes, n = codec.v_codes(V[None], bits)
            vf = codec.bf16_to_f32(V)
            u = rational_fwht(vf)
            nn = rational_norm(vf)
            assert n[0] == np.float32(nn)
            taus = [rn32(F(m) * F(nn)) for m in mid]
            want = [sum(1 for t in taus if ui > t) for ui in u]
            assert codes[0].tolist() == want


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_v_codes_are_nearest_centroid(bits):
    """Codes equal the float64 nearest centroid of y = Hv/|v| except where y is
    within float32 rounding of a midpoint."""
    c64, m64 = lloyd_max.lloyd_max_normal(1 << bits)
    rng = np.random.default_rng(20 + bits)
    V = codec.f32_to_bf16(rng.standard_normal((500, 64)).astype(np.float32))
    codes, n = codec.v_codes(V, bits)
    v = codec.bf16_to_f32(V).astype(np.float64)
    y = (v @ hadamard(64)) / np.linalg.norm(v, axis=1, keepdims=True)
    nearest = np.argmin(np.abs(y[..., None] - c64), axis=-1)
    close = np.min(np.abs(y[..., None] - m64), axis=-1) < 1e-5
    assert np.array_equal(codes[~close], nearest[~close])
    assert close.mean() < 1e-3


def test_v_quantiser_mse_on_gaussian_vectors():
    """Rotated, normalised Gaussian coordinates are close to N(0,1), so the
    per-coordinate distortion is close to the table MSE (3 bits: ~0.0345)."""
    c, m = lloyd_max.lloyd_max_normal(8)
    rng = np.random.default_rng(5)
    V = codec.f32_to_bf16(rng.standard_normal((4000, 128)).astype(np.float32))
    codes, n = codec.v_codes(V, 3)
    v = codec.bf16_to_f32(V).astype(np.float64)
    y = (v @ hadamard(128)) / n[:, None].astype(np.float64)
    cf, _ = lloyd_max.tables_f32(3)
    mse = np.mean((y - cf.astype(np.float64)[codes]) ** 2)
    assert abs(mse - lloyd_max.mse_normal(c, m)) < 1.5e-3


@pytest.mark.parametrize("bits,cpos", [(2, 1.510), (3, 0.7560), (4, 0.9424)])
def test_spike_vector_closed_form(bits, cpos):
    """v = alpha e_k: Hv = alpha * row_k(H) = +-alpha, n = |alpha|, y = +-1,
    so every coordinate takes the centroid c(1) (Max's table, given here to 4
    digits) with the sign of H_kj, and the decoded vector is c(1) alpha e_k."""
    d = 64
    cf, _ = lloyd_max.tables_f32(bits)
    for k in (0, 5, 63):
        for alpha in (1.0, -3.5):
            v = np.zeros((1, d), np.float32)
            v[0, k] = alpha
            enc = codec.encode_layer(np.zeros((1, 1, d), np.uint16), codec.f32_to_bf16(v)[None], bits)
            _, Vh = dequantise_f64(enc)
            c1 = float(cf[np.argmin(np.abs(cf - cpos))])
            want = np.zeros(d)
            want[k] = c1 * alpha
            np.testing.assert_allclose(Vh[0, 0], want, atol=1e-6)
            assert abs(c1 - cpos) < 1e-3


def test_zero_vector_decodes_to_zero():
    enc = codec.encode_layer(np.zeros((1, 2, 64), np.uint16), np.zeros((1, 2, 64), np.uint16), 3)
    Kb, Vb = codec.decompress_layer(enc)
    assert not Kb.any() and not codec.bf16_to_f32(Vb).any()
    assert np.all(enc["norms"] == 0)


def test_v_decompress_agrees_with_float64_dequantisation():
    rng = np.random.default_rng(11)
    V = codec.f32_to_bf16(rng.standard_normal((2, 50, 128)).astype(np.float32) * 4)
    K = codec.f32_to_bf16(rng.standard_normal((2, 50, 128)).astype(np.float32))
    for bits in (2, 3, 4):
        enc = codec.encode_layer(K, V, bits)
        Kb, Vb = codec.decompress_layer(enc)
        Kh, Vh = dequantise_f64(enc)
        vb = codec.bf16_to_f32(Vb).astype(np.float64)
        assert np.all(np.abs(vb - Vh) <= np.abs(Vh) * 2 ** -8 + 1e-6)
        assert np.array_equal(codec.bf16_to_f32(Kb), codec.bf16_to_f32(codec.f32_to_bf16(Kh.astype(np.float32))))


def test_encode_nonfinite_v():
    V = np.zeros((1, 1, 64), np.uint16)
    V[0, 0, 3] = 0x7FC0  # NaN
    with pytest.raises(ValueError):
        codec.v_codes(V, 3)


# ----------------------------------------------------- block-scaled K (option)

def _rand_k(shape, seed):
    rng = np.random.default_rng(seed)
    return codec.f32_to_bf16(rng.standard_normal(shape).astype(np.float32) * np.float32(3))


def test_k_block_max_maps_to_127_and_error_bound():
    K = _rand_k((2, 5, 128), 11)
    s = codec.k_scales_block(K)
    q = codec.k_quantize_block(K, s)
    k = codec.bf16_to_f32(K).reshape(2, 5, 4, 32)
    qb = q.reshape(2, 5, 4, 32).astype(np.int32)
    assert s.shape == (2, 5, 4) and s.dtype == np.float32
    # the largest |k| of every block lands on +-127
    arg = np.abs(k).argmax(axis=-1)
    top = np.take_along_axis(qb, arg[..., None], axis=-1)[..., 0]
    assert np.all(np.abs(top) == 127)
    # nearest-integer error: |k/s - q| <= 1/2 (+ float32 slack)
    assert np.all(np.abs(k / s[..., None] - qb) <= 0.5 + 1e-5)
    assert qb.min() >= -127 and qb.max() <= 127


def test_k_block_zero_block_and_ties_to_even():
    K = np.zeros((1, 1, 64), dtype=np.uint16)
    vals = np.zeros(32, dtype=np.float32)
    vals[0] = 127.0  # s = 1 exactly
    vals[1:6] = [2.5, 3.5, -2.5, -0.5, 0.5]
    K[0, 0, 32:] = codec.f32_to_bf16(vals)
    s = codec.k_scales_block(K)
    q = codec.k_quantize_block(K, s).astype(np.int32)
    assert s[0, 0, 0] == 1.0 and not q[0, 0, :32].any()  # all-zero block
    assert s[0, 0, 1] == 1.0
    assert list(q[0, 0, 32:38]) == [127, 2, 4, -2, 0, 0]


def test_k_block_power_of_two_scaling_is_local_to_its_block():
    K = _rand_k((1, 3, 128), 12)
    s0 = codec.k_scales_block(K)
    q0 = codec.k_quantize_block(K, s0)
    k = codec.bf16_to_f32(K).copy()
    k[0, 1, 64:96] *= np.float32(2.0 ** 7)  # one block of one token
    K2 = codec.f32_to_bf16(k)
    s2 = codec.k_scales_block(K2)
    q2 = codec.k_quantize_block(K2, s2)
    assert np.array_equal(q2, q0)  # codes are scale-invariant per block
    ratio = s2 / s0
    assert ratio[0, 1, 2] == 2.0 ** 7
    ratio[0, 1, 2] = 1.0
    assert np.all(ratio == 1.0)  # no other block (token or coordinate) moved


def test_k_block_equals_per_tensor_when_every_block_holds_the_maximum():
    K = _rand_k((2, 4, 64), 13)
    k = codec.bf16_to_f32(K).copy()
    m = np.float32(np.abs(k).max() * 2)
    k[..., ::32] = m  # the first element of every block is the tensor maximum
    K2 = codec.f32_to_bf16(k)
    _, st = codec.k_scale(K2)
    sb = codec.k_scales_block(K2)
    assert np.all(sb == st)
    assert np.array_equal(codec.k_quantize_block(K2, sb), codec.k_quantize(K2, st))


def test_k_block_layer_round_trip_and_dequantisation():
    K = _rand_k((2, 7, 64), 14)
    V = _rand_k((2, 7, 64), 15)
    enc = codec.encode_layer(K, V, 3, k_block=32)
    assert enc["scale"] == 1.0 and enc["kscales"].shape == (2, 7, 2)
    Kd, _ = codec.decompress_layer(enc)
    want = codec.f32_to_bf16(enc["kq"].astype(np.float32).reshape(2, 7, 2, 32)
                             * enc["kscales"][..., None]).reshape(2, 7, 64)
    assert np.array_equal(Kd, want)
    # block scales never lose to the per-tensor scale on the same K
    err_t = np.abs(codec.bf16_to_f32(codec.decompress_layer(codec.encode_layer(K, V, 3))[0]) - codec.bf16_to_f32(K)).max()
    err_b = np.abs(codec.bf16_to_f32(Kd) - codec.bf16_to_f32(K)).max()
    assert err_b <= err_t
    with pytest.raises(ValueError):
        codec.encode_layer(K, V, 3, k_block=16)


def test_block_k_encoding_concatenates_at_group_boundaries():
    # incremental append reads: with block-scaled K every stored byte depends
    # only on its own token, so encoding a context in parts (split at 32-token
    # group boundaries) gives the bytes of encoding it at once; a per-tensor
    # K scale depends on every token, which is why appends need block scales
    K = _rand_k((2, 100, 64), 21)
    V = _rand_k((2, 100, 64), 22)
    whole = codec.encode_layer(K, V, 3, k_block=32)
    parts = [codec.encode_layer(K[:, a:b], V[:, a:b], 3, k_block=32) for a, b in ((0, 32), (32, 96), (96, 100))]
    for key in ("kq", "kscales", "norms", "codes"):
        assert np.array_equal(np.concatenate([p[key] for p in parts], axis=1), whole[key]), key
    assert np.array_equal(np.concatenate([p["packed"] for p in parts], axis=1), whole["packed"])
    tensor = [codec.encode_layer(K[:, a:b], V[:, a:b], 3) for a, b in ((0, 32), (32, 100))]
    assert not np.array_equal(np.concatenate([p["kq"] for p in tensor], axis=1), codec.encode_layer(K, V, 3)["kq"])
