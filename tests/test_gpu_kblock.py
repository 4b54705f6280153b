"""GPU parity of block-scaled K pools (kvpool_create_ex with k_block = 32, the
"q8_0" reading): int8 K codes, their float32 block scales, V codes and norms
bit-exact; decompress bit-exact; attention (the tensor-core kernel, K^ as fp16
hi + lo of each block's codes times its scale) within 2e-3 of the oracle's
float64 attention over the same dequantised cache: row groups of at most 64
rows (spread layout) and of 128, with and without tails."""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_decompress, check_encode, to_dev

pytestmark = pytest.mark.gpu

KVPOOL_ERR_UNSUPPORTED = -7


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _run(kp, w, bits, tail_lens=None, rows=None):
    import torch

    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [bits], k_block=32)
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, bits, k_block=32)
    Q = wl.layer_q(w, 0)
    dev_tail = host_tail = None
    if tail_lens is not None:
        Kt, Vt = wl.layer_tail(w, 0)
        dev_tail = (to_dev(Kt), to_dev(Vt), torch.from_numpy(tail_lens.astype(np.int32)).cuda())
        host_tail = (Kt, Vt, tail_lens)
    out = pool.attend(0, to_dev(Q), tail=dev_tail)
    assert pool.status() == 0
    check_encode(pool, 0, enc)
    check_decompress(pool, 0, enc)
    err = attention_error(out, enc, Q, host_tail, rows=rows)
    assert err <= TOL, err
    return pool


SMALL = [
    # name, Hk, Hq, d, ctx, agents, bits, tail_init
    ("kb_ragged_2bit", 4, 16, 128, 300, 5, 2, 0),
    ("kb_d64_3bit_tail", 2, 4, 64, 700, 6, 3, 20),
    ("kb_4bit_tail", 2, 16, 128, 1000, 2, 4, 7),
    ("kb_ctx1", 1, 2, 128, 1, 4, 3, 3),
    ("kb_128rows_3bit", 2, 16, 128, 600, 16, 3, 0),
    ("kb_200rows_d64_4bit_tail", 2, 16, 64, 900, 25, 4, 9),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(kp, case):
    _, Hk, Hq, d, ctx, A, bits, tail_init = case
    w = wl.custom(case[0], 1, Hk, Hq, d, ctx, A, "lognormal", tail_init, 2, (bits,))
    lens = np.array([(a * 3) % (w.tail_max + 1) for a in range(A)]) if tail_init else None
    _run(kp, w, bits, lens).close()


def test_llama_layer_sampled_rows(kp):
    w = wl.WORKLOADS["llama3_8b_4k"]
    rng = np.random.default_rng(5)
    rows = [(int(a), int(h)) for a, h in zip(rng.integers(0, w.agents, 24), rng.integers(0, w.q_heads, 24))]
    pool = _run(kp, w, 3, rows=rows)
    # block-scaled layers export their bytes and scales but do not import
    kq, vc, vn, ks = pool.export_layer(0)
    assert float(ks.cpu()[0]) == 1.0
    fresh = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3], k_block=32)
    with pytest.raises(kp.KVPoolError) as e:
        fresh.import_layer(0, kq, vc, vn, ks)
    assert e.value.code == KVPOOL_ERR_UNSUPPORTED
    fresh.close()
    pool.close()


def test_per_tensor_pool_has_no_block_scales(kp):
    w = wl.custom("pt", 1, 2, 4, 64, 64, 2, "lognormal")
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3])
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    with pytest.raises(kp.KVPoolError) as e:
        pool.export_kscales(0)
    assert e.value.code == KVPOOL_ERR_UNSUPPORTED
    pool.close()
