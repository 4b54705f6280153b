"""Pins of the oracle's float64 attention (CPU only).

Independent checks: a pure-Python double loop (math.exp, Python floats, the
Hadamard matrix from its popcount formula) on tiny inputs; closed forms
(equal logits give the mean value, a dominant logit selects its token, a
masked-out pool leaves plain attention over the tail); invariance to the order
of agents; the GQA head mapping; the sampled-row entry point.
"""

import math

import numpy as np
import pytest

from oracle import attention, codec
from shared_quantized_kv_gb300 import workloads as wl


def _tiny_layer(seed=0, Hk=2, T=5, d=8, bits=3):
    rng = np.random.default_rng(seed)
    K = codec.f32_to_bf16(rng.standard_normal((Hk, T, d)).astype(np.float32))
    V = codec.f32_to_bf16(rng.standard_normal((Hk, T, d)).astype(np.float32))
    return codec.encode_layer(K, V, bits)


def _brute(enc, Q, tail, scale):
    """Pure-Python restatement of the attention definition."""
    A, Hq, d = Q.shape
    Hk, T, _ = enc["kq"].shape
    G = Hq // Hk
    cen, _ = __import__("oracle").lloyd_max.tables_f32(enc["bits"])
    hij = lambda i, j: -1.0 if bin(i & j).count("1") % 2 else 1.0
    s = float(enc["scale"])
    out = np.zeros((A, Hq, d))
    for a in range(A):
        for h in range(Hq):
            g = h // G
            q = [float(codec.bf16_to_f32(Q[a, h, i])) for i in range(d)]
            keys, vals = [], []
            for t in range(T):
                keys.append([int(enc["kq"][g, t, i]) * s for i in range(d)])
                n = float(enc["norms"][g, t])
                c = [float(cen[enc["codes"][g, t, j]]) for j in range(d)]
                vals.append([n * sum(hij(i, j) * c[j] for j in range(d)) / d for i in range(d)])
            if tail is not None:
                for t in range(int(tail[2][a])):
                    keys.append([float(codec.bf16_to_f32(tail[0][a, g, t, i])) for i in range(d)])
                    vals.append([float(codec.bf16_to_f32(tail[1][a, g, t, i])) for i in range(d)])
            logits = [scale * sum(q[i] * k[i] for i in range(d)) for k in keys]
            mx = max(logits)
            w = [math.exp(x - mx) for x in logits]
            tot = sum(w)
            for i in range(d):
                out[a, h, i] = sum(w[t] * vals[t][i] for t in range(len(w))) / tot
    return out


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_matches_pure_python_double_loop(bits):
    enc = _tiny_layer(bits=bits)
    rng = np.random.default_rng(1)
    A, Hq, d = 3, 4, 8
    Q = codec.f32_to_bf16(rng.standard_normal((A, Hq, d)).astype(np.float32))
    Kt = codec.f32_to_bf16(rng.standard_normal((A, 2, 4, d)).astype(np.float32))
    Vt = codec.f32_to_bf16(rng.standard_normal((A, 2, 4, d)).astype(np.float32))
    lens = np.array([0, 3, 4])
    Kh, Vh = attention.dequantise_f64(enc)
    for tail in (None, (Kt, Vt, lens)):
        for scale in (None, 0.7):
            got = attention.attend_f64(Kh, Vh, Q, tail, scale)
            want = _brute(enc, Q, tail, 1 / math.sqrt(d) if scale is None else scale)
            np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_equal_logits_give_mean_value():
    enc = _tiny_layer(T=7)
    Kh, Vh = attention.dequantise_f64(enc)
    Q = np.zeros((2, 4, 8), np.uint16)  # q = 0 -> all logits 0
    out = attention.attend_f64(Kh, Vh, Q)
    for h in range(4):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(Vh[h // 2].mean(0), (2, 8)), atol=1e-14)


def test_dominant_logit_selects_its_token():
    enc = _tiny_layer(T=6)
    Kh, Vh = attention.dequantise_f64(enc)
    for t in range(6):
        K2 = np.zeros_like(Kh)
        K2[:, t, 0] = 1.0
        Q = np.zeros((1, 2, 8), np.float32)
        Q[:, :, 0] = 4096.0
        out = attention.attend_f64(K2, Vh, codec.f32_to_bf16(Q), scale=1.0)
        np.testing.assert_allclose(out[0, 0], Vh[0, t], atol=1e-12)
        np.testing.assert_allclose(out[0, 1], Vh[1, t], atol=1e-12)


def test_masked_pool_leaves_tail_attention():
    enc = _tiny_layer(T=5, Hk=1)
    Kh, Vh = attention.dequantise_f64(enc)
    K2 = np.zeros_like(Kh)
    K2[..., 0] = -1000.0  # pool logits far below the tail's
    rng = np.random.default_rng(2)
    Q = np.zeros((2, 1, 8), np.float32)
    Q[..., 0] = 1.0
    Q[..., 1:] = rng.standard_normal((2, 1, 7))
    Qb = codec.f32_to_bf16(Q)
    Kt = rng.standard_normal((2, 1, 3, 8)).astype(np.float32)
    Kt[..., 0] = 0.0
    Kt = codec.f32_to_bf16(Kt)
    Vt = codec.f32_to_bf16(rng.standard_normal((2, 1, 3, 8)).astype(np.float32))
    out = attention.attend_f64(K2, Vh, Qb, (Kt, Vt, np.array([3, 2])), scale=1.0)
    for a, n in ((0, 3), (1, 2)):
        q = codec.bf16_to_f32(Qb[a, 0]).astype(np.float64)
        k = codec.bf16_to_f32(Kt[a, 0, :n]).astype(np.float64)
        v = codec.bf16_to_f32(Vt[a, 0, :n]).astype(np.float64)
        w = np.exp(k @ q - (k @ q).max())
        np.testing.assert_allclose(out[a, 0], (w / w.sum()) @ v, rtol=1e-12)


def test_agent_order_invariance_and_gqa_mapping():
    w = wl.WORKLOADS["tiny"]
    K, V = wl.layer_kv(w, 0)
    enc = codec.encode_layer(K, V, 3)
    Kh, Vh = attention.dequantise_f64(enc)
    Q = wl.layer_q(w, 0)
    out = attention.attend_f64(Kh, Vh, Q)
    perm = np.array([2, 0, 1])
    np.testing.assert_allclose(attention.attend_f64(Kh, Vh, Q[perm]), out[perm], rtol=1e-13)
    # consecutive grouping: q-head h reads kv-head h // G
    Vc = np.zeros_like(Vh)
    Vc[0], Vc[1] = 1.0, 2.0
    o = attention.attend_f64(Kh, Vc, Q)
    np.testing.assert_allclose(o[:, :2], 1.0)
    np.testing.assert_allclose(o[:, 2:], 2.0)


def test_sampled_rows_agree_with_full():
    w = wl.custom(kv_heads=2, q_heads=8, head_dim=64, ctx=96, agents=4, tail_init=5, decode_steps=2)
    K, V = wl.layer_kv(w, 0)
    enc = codec.encode_layer(K, V, 3)
    Kh, Vh = attention.dequantise_f64(enc)
    Q = wl.layer_q(w, 0)
    Kt, Vt = wl.layer_tail(w, 0)
    lens = np.array([w.tail_len(1)] * 4)
    full = attention.attend_f64(Kh, Vh, Q, (Kt, Vt, lens))
    rows = [(0, 0), (3, 7), (2, 4)]
    part = attention.attend_rows_f64(Kh, Vh, Q, rows, (Kt, Vt, lens))
    for i, (a, h) in enumerate(rows):
        np.testing.assert_allclose(part[i], full[a, h], rtol=1e-12)


def test_row_error_metric():
    ref = np.array([[1.0, -2.0, 0.5], [0.0, 0.0, 4.0]])
    out = ref + np.array([[0.002, 0, 0], [0, 0.004, 0]])
    assert attention.row_rel_error(out, ref) == pytest.approx(1e-3)


# ---------------------------------------------------------------- context split

def _small_layer(seed=3, Hk=2, G=2, d=16, T=40, A=3):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((Hk, T, d)) * 1.5
    V = rng.standard_normal((Hk, T, d))
    Q = codec.f32_to_bf16(rng.standard_normal((A, Hk * G, d)).astype(np.float32))
    return K, V, Q


@pytest.mark.parametrize("cuts", [[20], [1], [39], [7, 19, 33], list(range(1, 40))])
def test_merged_slices_equal_full_attention(cuts):
    # any split of the context, merged by log-sum-exp, is the plain softmax
    # attention over the whole context
    K, V, Q = _small_layer()
    edges = [0] + cuts + [K.shape[1]]
    parts = [attention.attend_slice_f64(K, V, Q, b, e) for b, e in zip(edges[:-1], edges[1:])]
    got = attention.merge_slices_f64(parts)
    want = attention.attend_f64(K, V, Q)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # the order of the parts does not matter
    assert np.allclose(attention.merge_slices_f64(parts[::-1]), want, rtol=1e-12, atol=1e-12)


def test_one_slice_is_the_slice_attention():
    K, V, Q = _small_layer(seed=5)
    lse, o = attention.attend_slice_f64(K, V, Q, 0, K.shape[1])
    assert np.allclose(attention.merge_slices_f64([(lse, o)]), attention.attend_f64(K, V, Q), atol=1e-12)


def test_slice_lse2_brute_force():
    # lse2 = log2 sum_t 2^(x_t), x_t = scale * <q, k_t> / ln 2, by a Python loop
    K, V, Q = _small_layer(seed=7, Hk=1, G=2, d=8, T=9, A=2)
    lse, _ = attention.attend_slice_f64(K, V, Q, 2, 7)
    q = codec.bf16_to_f32(Q).astype(np.float64)
    scale = 1.0 / math.sqrt(8)
    for a in range(2):
        for h in range(2):
            tot = 0.0
            for t in range(2, 7):
                x = scale * sum(q[a, h, i] * K[0, t, i] for i in range(8)) / math.log(2.0)
                tot += 2.0 ** x
            assert abs(lse[a, h] - math.log2(tot)) < 1e-12


def test_slices_with_tail_equal_attention_with_tail():
    K, V, Q = _small_layer(seed=9, Hk=2, G=2, d=16, T=30, A=3)
    rng = np.random.default_rng(11)
    Kt = codec.f32_to_bf16(rng.standard_normal((3, 2, 5, 16)).astype(np.float32))
    Vt = codec.f32_to_bf16(rng.standard_normal((3, 2, 5, 16)).astype(np.float32))
    lens = np.array([0, 5, 2])
    tail = (Kt, Vt, lens)
    parts = [attention.attend_slice_f64(K, V, Q, 0, 13), attention.attend_slice_f64(K, V, Q, 13, 30),
             attention.tail_slice_f64(Q, tail, 2)]
    got = attention.merge_slices_f64(parts)
    want = attention.attend_f64(K, V, Q, tail)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
