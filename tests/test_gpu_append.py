"""GPU parity of incremental appends to block-scaled pools (kvpool_append):
after each append the layer's stored bytes equal the oracle's encode of all
its tokens at once (with block-scaled K every byte depends on its own token),
decompress is bit-exact and attention over the tokens held is within 2e-3."""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_decompress, check_encode, to_dev

pytestmark = pytest.mark.gpu

ERR_INVALID_ARG, ERR_STATE, ERR_UNSUPPORTED = -1, -2, -7


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _check_prefix(pool, K, V, Q, T, bits):
    assert pool.layer_len(0) == T
    enc = codec.encode_layer(K[:, :T], V[:, :T], bits, k_block=32)
    check_encode(pool, 0, enc)
    check_decompress(pool, 0, enc)
    out = pool.attend(0, to_dev(Q))
    assert pool.status() == 0
    err = attention_error(out, enc, Q)
    assert err <= TOL, (T, err)


@pytest.mark.parametrize("d,cuts,bits", [
    (128, (256, 640, 690), 3),       # 32-token items; a ragged last append
    (64, (32, 128, 160, 333), 2),    # 64-token items starting at odd group offsets
    (128, (96, 1000), 4),
    # d 64 encodes 64 tokens per item: an append in the last 32-token group of
    # the padded token axis (96 of 128) must not write the item's second group,
    # which lies past the KV head's codes
    (64, (96, 100), 3),
])
def test_appends_equal_one_encode(kp, d, cuts, bits):
    ctx = cuts[-1] + 24  # capacity above the last length
    w = wl.custom("append", 1, 2, 8, d, ctx, 3, "lognormal", bits=(bits,))
    K, V = wl.layer_kv(w, 0)
    Q = wl.layer_q(w, 0)
    pool = kp.KVPool(1, w.kv_heads, d, ctx, [bits], k_block=32)
    a = 0
    for b in cuts:
        pool.append(0, to_dev(np.ascontiguousarray(K[:, a:b])), to_dev(np.ascontiguousarray(V[:, a:b])))
        _check_prefix(pool, K, V, Q, b, bits)
        a = b
    pool.close()


def test_append_errors_and_reset(kp):
    w = wl.custom("append_err", 1, 2, 4, 64, 200, 2, "lognormal")
    K, V = wl.layer_kv(w, 0)
    dK, dV = to_dev(K), to_dev(V)
    per_tensor = kp.KVPool(1, 2, 64, 200, [3])
    with pytest.raises(kp.KVPoolError) as e:
        per_tensor.append(0, dK[:, :32].contiguous(), dV[:, :32].contiguous())
    assert e.value.code == ERR_UNSUPPORTED
    per_tensor.close()

    pool = kp.KVPool(1, 2, 64, 200, [3], k_block=32)
    assert pool.layer_len(0) == 0
    pool.append(0, dK[:, :64].contiguous(), dV[:, :64].contiguous())
    with pytest.raises(kp.KVPoolError) as e:  # beyond the capacity
        pool.append(0, dK[:, :150].contiguous(), dV[:, :150].contiguous())
    assert e.value.code == ERR_INVALID_ARG
    with pytest.raises(kp.KVPoolError) as e:  # compress needs an empty layer
        pool.compress(0, dK, dV)
    assert e.value.code == ERR_STATE
    pool.append(0, dK[:, 64:100].contiguous(), dV[:, 64:100].contiguous())  # ragged: closes the layer
    with pytest.raises(kp.KVPoolError) as e:
        pool.append(0, dK[:, 100:132].contiguous(), dV[:, 100:132].contiguous())
    assert e.value.code == ERR_STATE
    assert pool.layer_len(0) == 100
    # reset empties the layer; compress then writes all ctx tokens
    pool.reset_layer(0)
    assert pool.layer_len(0) == 0
    pool.compress(0, dK, dV)
    assert pool.status() == 0 and pool.layer_len(0) == 200
    check_encode(pool, 0, codec.encode_layer(K, V, 3, k_block=32))
    pool.close()
