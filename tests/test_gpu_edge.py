"""GPU edge cases of the hot path against the CPU oracle, through the C-ABI:
degenerate data (an all-zero K tensor, zero V vectors, extreme magnitudes),
non-finite inputs (the device status word), and the largest row count a pool
accepts (1024 query rows per KV head, eight row groups)."""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_decompress, check_encode, to_dev

pytestmark = pytest.mark.gpu

KVPOOL_ERR_NONFINITE = -5


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _bf16(x):
    return codec.f32_to_bf16(np.asarray(x, dtype=np.float32))


def _check_layer(kp, pool, K, V, Q, bits, rows=None):
    pool.compress(0, to_dev(K), to_dev(V))
    out = pool.attend(0, to_dev(Q))
    assert pool.status() == 0
    enc = codec.encode_layer(K, V, bits)
    check_encode(pool, 0, enc)
    check_decompress(pool, 0, enc)
    err = attention_error(out, enc, Q, rows=rows)
    assert err <= TOL, err
    return enc


def test_zero_k_and_zero_v_vectors(kp):
    # K all zero: s = 1 and every q = 0, so every logit is 0 and each row is
    # the mean of the dequantised V; every 7th V vector is zero (n = 0)
    w = wl.custom("zeros", 1, 2, 8, 128, 333, 3, "lognormal")
    _, V = wl.layer_kv(w, 0)
    K = np.zeros_like(V)
    V = V.copy()
    V[:, ::7, :] = 0
    Q = wl.layer_q(w, 0)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3])
    enc = _check_layer(kp, pool, K, V, Q, 3)
    assert float(enc["scale"]) == 1.0 and not enc["kq"].any()
    pool.close()


@pytest.mark.parametrize("kexp,vexp", [(40, -40), (-40, 40)])
def test_extreme_magnitudes(kp, kexp, vexp):
    # power-of-two scalings keep the bf16 inputs exact; the squares of the
    # norm tree stay normal float32 numbers
    w = wl.custom("scaled", 1, 2, 4, 64, 200, 2, "lognormal")
    K, V = wl.layer_kv(w, 0)
    K = _bf16(codec.bf16_to_f32(K) * np.float32(2.0 ** kexp))
    V = _bf16(codec.bf16_to_f32(V) * np.float32(2.0 ** vexp))
    Q = wl.layer_q(w, 0)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [4])
    _check_layer(kp, pool, K, V, Q, 4)
    pool.close()


@pytest.mark.parametrize("kexp", [6, 7])
def test_logits_around_the_fused_exponent_bound(kp, kexp):
    # K scaled so that the rows' largest logits (log2 units) lie around
    # 2^10 (about 300 to 1100 for 2^6, 600 to 2200 for 2^7), where the
    # softmax switches between its two exponent forms (one fused
    # multiply-add, or the difference first); several tiles, so the
    # reference moves between tiles of one row; both attention paths
    w = wl.custom("bound", 1, 2, 16, 128, 1500, 6, "lognormal", bits=(3,))
    K, V = wl.layer_kv(w, 0)
    K = _bf16(codec.bf16_to_f32(K) * np.float32(2.0 ** kexp))
    Q = wl.layer_q(w, 0)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3], max_rows=w.rows)
    enc = _check_layer(kp, pool, K, V, Q, 3)
    out = pool.attend_ws(0, to_dev(Q))
    assert pool.status() == 0
    err = attention_error(out, enc, Q)
    assert err <= TOL, err
    pool.close()


@pytest.mark.parametrize("where", ["k_inf", "v_nan"])
def test_nonfinite_input_sets_status(kp, where):
    w = wl.custom("nonfinite", 1, 2, 4, 64, 100, 2, "lognormal")
    K, V = wl.layer_kv(w, 0)
    bad_K, bad_V = K.copy(), V.copy()
    if where == "k_inf":
        bad_K[1, 37, 5] = 0x7F80  # +Inf
    else:
        bad_V[0, 99, 63] = 0x7FC0  # NaN
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3])
    pool.compress(0, to_dev(bad_K), to_dev(bad_V))
    assert pool.status() == KVPOOL_ERR_NONFINITE
    assert pool.status() == 0  # read and cleared
    # the pool stays usable: re-arm the layer and encode finite data
    pool.reset_layer(0)
    _check_layer(kp, pool, K, V, wl.layer_q(w, 0), 3)
    pool.close()


def test_largest_row_count(kp):
    # 128 agents x 8 query heads per KV head = 1024 rows: eight row groups of
    # 128 rows per KV head, each over the same context splits
    w = wl.custom("rows1024", 1, 1, 8, 128, 700, 128, "lognormal")
    K, V = wl.layer_kv(w, 0)
    Q = wl.layer_q(w, 0)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3], max_rows=1024)
    rng = np.random.default_rng(3)
    rows = [(int(a), int(h)) for a, h in zip(rng.integers(0, 128, 48), rng.integers(0, 8, 48))]
    rows += [(0, 0), (127, 7), (64, 3)]
    _check_layer(kp, pool, K, V, Q, 3, rows=rows)
    pool.close()
