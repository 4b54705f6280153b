"""Multi-layer compress and decompress (kvpool_compress_layers,
kvpool_decompress_layers) against the CPU oracle, through the C-ABI: mixed V
widths in one call, block-scaled K, more layers than one launch takes, the
argument and state errors, and all 32 layers of the Llama-3-8B-shaped 4K
workload in the benchmark's launch configuration (sampled layers bit-exact)."""

import ctypes

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_encode, from_dev_bf16, to_dev

pytestmark = pytest.mark.gpu

INVALID_ARG, STATE = -1, -2


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _check_dec(Kd, Vd, enc):
    kb, vb = codec.decompress_layer(enc)
    assert np.array_equal(from_dev_bf16(Kd), kb)
    assert np.array_equal(from_dev_bf16(Vd), vb)


def _sample_rows(w, n=24, seed=1):
    rng = np.random.default_rng(seed)
    return [(int(a), int(h)) for a, h in zip(rng.integers(0, w.agents, n), rng.integers(0, w.q_heads, n))]


def test_mixed_widths_any_order(kp):
    bits = (2, 3, 4, 3, 2)
    w = wl.custom("multi", len(bits), 2, 8, 128, 333, 3, "lognormal", 0, 1, bits)
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, list(bits))
    KV = [wl.layer_kv(w, l) for l in range(w.layers)]
    order = [3, 0, 4, 1, 2]
    pool.compress_layers(order, [to_dev(KV[l][0]) for l in order], [to_dev(KV[l][1]) for l in order])
    assert pool.status() == 0
    encs = [codec.encode_layer(KV[l][0], KV[l][1], bits[l]) for l in range(w.layers)]
    for l in range(w.layers):
        check_encode(pool, l, encs[l])
    Ko, Vo = pool.decompress_layers(list(range(w.layers)))
    for l in range(w.layers):
        _check_dec(Ko[l], Vo[l], encs[l])
    for l in (0, 2):
        Q = wl.layer_q(w, l)
        err = attention_error(pool.attend(l, to_dev(Q)), encs[l], Q)
        assert err <= TOL, (l, err)
    assert pool.status() == 0
    pool.close()


def test_block_scaled_d64(kp):
    bits = (4, 2, 3)
    w = wl.custom("multi_kb", len(bits), 2, 4, 64, 200, 2, "lognormal", 0, 1, bits)
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, list(bits), k_block=32)
    KV = [wl.layer_kv(w, l) for l in range(w.layers)]
    pool.compress_layers([0, 1, 2], [to_dev(k) for k, _ in KV], [to_dev(v) for _, v in KV])
    assert pool.status() == 0
    for l in range(w.layers):
        enc = codec.encode_layer(KV[l][0], KV[l][1], bits[l], k_block=32)
        check_encode(pool, l, enc)
        Ko, Vo = pool.decompress_layers([l])
        _check_dec(Ko[0], Vo[0], enc)
    pool.close()


def test_more_layers_than_one_launch(kp):
    import torch

    n = 35  # one launch takes 32 layers
    bits = tuple(2 + l % 3 for l in range(n))
    w = wl.custom("many", n, 1, 2, 64, 40, 1, "lognormal", 0, 1, bits)
    pool = kp.KVPool(n, w.kv_heads, w.head_dim, w.ctx, list(bits))
    KV = [wl.layer_kv(w, l) for l in range(n)]
    pool.compress_layers(list(range(n)), [to_dev(k) for k, _ in KV], [to_dev(v) for _, v in KV])
    assert pool.status() == 0
    encs = [codec.encode_layer(KV[l][0], KV[l][1], bits[l]) for l in range(n)]
    for l in range(n):
        check_encode(pool, l, encs[l])
    # V only: a NULL array for the K half
    Vo = [torch.empty((w.kv_heads, w.ctx, w.head_dim), dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    lay = (ctypes.c_int * n)(*range(n))
    vp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in Vo])
    rc = kp.lib().kvpool_decompress_layers(pool._h, n, lay, None, vp, None)
    assert rc == 0
    torch.cuda.synchronize()
    for l in range(n):
        _, vb = codec.decompress_layer(encs[l])
        assert np.array_equal(from_dev_bf16(Vo[l]), vb), l
    pool.close()


def test_errors_leave_state_unchanged(kp):
    import torch

    w = wl.custom("errs", 3, 1, 2, 64, 64, 1, "lognormal", 0, 1, (3, 3, 3))
    pool = kp.KVPool(3, 1, 64, 64, [3, 3, 3])
    K, V = wl.layer_kv(w, 0)
    Kd, Vd = to_dev(K), to_dev(V)
    L = kp.lib()

    def call(layers, Ks, Vs, n=None):
        n = len(layers) if n is None else n
        lay = (ctypes.c_int * max(len(layers), 1))(*layers)
        kp_ = (ctypes.c_void_p * max(len(Ks), 1))(*Ks)
        vp_ = (ctypes.c_void_p * max(len(Vs), 1))(*Vs)
        return L.kvpool_compress_layers(pool._h, n, lay, kp_, vp_, None)

    p, q = Kd.data_ptr(), Vd.data_ptr()
    assert call([0, 0], [p, p], [q, q]) == INVALID_ARG   # a layer named twice
    assert call([0, 3], [p, p], [q, q]) == INVALID_ARG   # out of range
    assert call([0], [p], [q], n=0) == INVALID_ARG       # n < 1
    assert call([0], [p + 2], [q]) == INVALID_ARG        # misaligned
    assert call([0], [0], [q]) == INVALID_ARG            # null
    pool.compress(1, Kd, Vd)
    assert call([0, 1], [p, p], [q, q]) == STATE         # layer 1 already compressed
    view = pool.layer_view(0)
    assert view.compressed == 0                          # layer 0 untouched
    lay = (ctypes.c_int * 1)(0)
    out = (ctypes.c_void_p * 1)(Kd.data_ptr())
    assert L.kvpool_decompress_layers(pool._h, 1, lay, out, None, None) == STATE
    assert L.kvpool_decompress_layers(pool._h, 1, lay, None, None, None) == INVALID_ARG
    assert call([0, 2], [p, p], [q, q]) == 0
    torch.cuda.synchronize()
    assert pool.status() == 0
    enc = codec.encode_layer(K, V, 3)
    for l in range(3):
        check_encode(pool, l, enc)
    pool.close()


def test_llama_4k_all_layers_as_benchmarked(kp):
    # the benchmark's compress and decompress phases: all 32 layers in one
    # call each, inputs drawn on the device; sampled layers against the oracle
    w = wl.WORKLOADS["llama3_8b_4k"]
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, w.bits_list())
    KV = [wl.layer_kv_torch(w, l, "cuda") for l in range(w.layers)]
    pool.compress_layers(list(range(w.layers)), [k for k, _ in KV], [v for _, v in KV])
    Ko, Vo = pool.decompress_layers(list(range(w.layers)))
    assert pool.status() == 0
    for l in (0, 17, 31):
        K, V = from_dev_bf16(KV[l][0]), from_dev_bf16(KV[l][1])
        enc = codec.encode_layer(K, V, w.layer_bits(l))
        check_encode(pool, l, enc)
        _check_dec(Ko[l], Vo[l], enc)
        Q = wl.layer_q(w, l)
        rows = _sample_rows(w)
        err = attention_error(pool.attend(l, to_dev(Q)), enc, Q, rows=rows)
        assert err <= TOL, (l, err)
    assert pool.status() == 0
    pool.close()
