"""GPU parity of the whole hot path against the CPU oracle, through the C-ABI.

Encode (int8 K, packed V codes, norms, K scale) and decompress (bf16 K, V) must
be bit-exact; attention within 2e-3 (max over rows of max|o - r| / max|r|)
of the oracle's float64 attention over the same dequantised cache.
"""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_decompress, check_encode, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _run_layer(kp, pool, w, layer, step=0, tail=None, rows=None):
    import torch

    K, V = wl.layer_kv(w, layer)
    pool.compress(layer, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, w.layer_bits(layer))
    Q = wl.layer_q(w, layer, step)
    dev_tail, host_tail = None, None
    if tail is not None:
        Kt, Vt, lens = tail
        dev_tail = (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())
        host_tail = (Kt, Vt, lens)
    out = pool.attend(layer, to_dev(Q), tail=dev_tail)
    assert pool.status() == 0
    check_encode(pool, layer, enc)
    err = attention_error(out, enc, Q, host_tail, rows=rows)
    assert err <= TOL, f"layer {layer}: attention error {err:.3e}"
    return enc, err


SMALL = [
    # name, Hk, Hq, d, ctx, agents, bits, tail_init
    ("tiny_like", 2, 4, 64, 256, 3, 3, 0),
    ("gqa4_ragged_2bit", 4, 16, 128, 300, 5, 2, 0),
    ("gqa8_4bit_tail", 2, 16, 128, 1000, 2, 4, 7),
    ("mha_one_agent", 3, 3, 64, 129, 1, 3, 0),
    ("ctx1_tail", 1, 2, 128, 1, 4, 3, 3),
    ("d64_gqa2_3bit_tail", 2, 4, 64, 700, 6, 3, 20),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(kp, case):
    _, Hk, Hq, d, ctx, A, bits, tail_init = case
    w = wl.custom(case[0], 1, Hk, Hq, d, ctx, A, "lognormal", tail_init, 2, (bits,))
    pool = kp.KVPool(1, Hk, d, ctx, [bits])
    tail = None
    if tail_init:
        Kt, Vt = wl.layer_tail(w, 0)
        lens = np.array([(a * 3) % (w.tail_max + 1) for a in range(A)])  # ragged, includes 0
        tail = (Kt, Vt, lens)
    enc, _ = _run_layer(kp, pool, w, 0, tail=tail)
    check_decompress(pool, 0, enc)
    pool.close()


def test_tiny_workload(kp):
    w = wl.WORKLOADS["tiny"]
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, w.bits_list())
    enc, err = _run_layer(kp, pool, w, 0)
    check_decompress(pool, 0, enc)
    pool.close()


def _sample_rows(w, n=24, seed=0):
    rng = np.random.default_rng(seed)
    return [(int(a), int(h)) for a, h in zip(rng.integers(0, w.agents, n), rng.integers(0, w.q_heads, n))]


@pytest.mark.parametrize("name,layers", [
    ("smollm2_2k", [0, 11, 23]),
    ("llama3_8b_4k", [0, 17, 31]),
])
def test_full_size_layers(kp, name, layers):
    w = wl.WORKLOADS[name]
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, w.bits_list())
    for layer in layers:
        enc, _ = _run_layer(kp, pool, w, layer)
        if layer == layers[0]:
            check_decompress(pool, layer, enc)
    pool.close()


def test_llama_long_with_tails(kp):
    w = wl.WORKLOADS["llama3_8b_long"]
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, w.bits_list())
    for layer in (0, 31):
        Kt, Vt = wl.layer_tail(w, layer)
        enc = None
        for step in range(w.decode_steps):
            lens = np.full(w.agents, w.tail_len(step))
            if enc is None:
                enc, _ = _run_layer(kp, pool, w, layer, step, (Kt, Vt, lens))
            else:
                import torch
                Q = wl.layer_q(w, layer, step)
                out = pool.attend(layer, to_dev(Q), tail=(to_dev(Kt), to_dev(Vt),
                                                          torch.from_numpy(lens.astype(np.int32)).cuda()))
                err = attention_error(out, enc, Q, (Kt, Vt, lens))
                assert err <= TOL, (layer, step, err)
    pool.close()


def test_qwen_mixed_precision_sampled_layers(kp):
    w = wl.WORKLOADS["qwen3_32b_32k"]
    bits = w.bits_list()
    pick = []
    for b in (2, 3, 4):
        pick += [l for l in range(w.layers) if bits[l] == b][:2]
    pool = kp.KVPool(w.layers, w.kv_heads, w.head_dim, w.ctx, bits)
    for layer in pick:
        _run_layer(kp, pool, w, layer, rows=_sample_rows(w))
    pool.close()
