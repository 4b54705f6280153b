"""GPU parity of the local attention-error estimate (kvpool_sensitivity)
against the oracle's float64 definition, and the allocation flow it feeds:
estimate every layer from recent tokens, allocate widths under a budget,
build a pool with them."""

import numpy as np
import pytest

from oracle import allocator, codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_encode, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _recent(w, layer, lens):
    import torch

    Kt, Vt = wl.layer_tail(w, layer)
    return (Kt, Vt, lens), (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())


@pytest.mark.parametrize("d,Hk,Hq,A,T", [(128, 2, 8, 5, 40), (64, 3, 6, 4, 130)])
def test_sensitivity_matches_oracle(kp, d, Hk, Hq, A, T):
    w = wl.custom("sens", 1, Hk, Hq, d, 64, A, "lognormal", T, 2)
    lens = np.array([(7 * a + 3) % (T + 1) for a in range(A)])
    lens[1] = 0  # an agent without recent tokens
    host, dev = _recent(w, 0, lens)
    Q = wl.layer_q(w, 0)
    s, rows = kp.sensitivity(to_dev(Q), dev, Hk)
    want = allocator.layer_sensitivity(Q, host[0], host[1], lens)
    assert s == pytest.approx(want, rel=1e-4)
    q, k, v = (codec.bf16_to_f32(x).astype(np.float64) for x in (Q, host[0], host[1]))
    G = Hq // Hk
    ref = [allocator.row_ratio(q[a, h], k[a, h // G, :lens[a]], v[a, h // G, :lens[a]], 1 / np.sqrt(d))
           for a in range(A) for h in range(Hq)]
    np.testing.assert_allclose(rows.cpu().numpy(), ref, rtol=1e-4, atol=1e-7)


def test_allocation_flow(kp):
    w = wl.WORKLOADS["llama3_8b_long"]
    layers = [0, 9, 18, 31]
    lens = np.full(w.agents, w.tail_len(0))
    sens = []
    for l in layers:
        _, dev = _recent(w, l, lens)
        s, _ = kp.sensitivity(to_dev(wl.layer_q(w, l)), dev, w.kv_heads)
        sens.append(s)
    per_bit = w.kv_heads * w.ctx * w.head_dim // 8
    bits = kp.allocate_bits(sens, [per_bit] * 4, 3 * 4 * per_bit)
    assert bits == list(allocator.allocate(sens, [1] * 4, 12)) and sum(bits) <= 12
    pool = kp.KVPool(len(layers), w.kv_heads, w.head_dim, w.ctx, bits)
    for i, l in enumerate(layers):
        K, V = wl.layer_kv(w, l)
        pool.compress(i, to_dev(K), to_dev(V))
        enc = codec.encode_layer(K, V, bits[i])
        Q = wl.layer_q(w, l)
        rng = np.random.default_rng(l)
        rows = [(int(a), int(h)) for a, h in zip(rng.integers(0, w.agents, 12), rng.integers(0, w.q_heads, 12))]
        out = pool.attend(i, to_dev(Q))
        assert pool.status() == 0
        check_encode(pool, i, enc)
        assert attention_error(out, enc, Q, rows=rows) <= TOL
    pool.close()
