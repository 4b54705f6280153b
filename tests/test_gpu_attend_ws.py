"""GPU parity of attention through a caller workspace (kvpool_attend_ws)
against the CPU oracle: the context in slices of one CTA each, partial states
in the workspace, then the log-sum-exp merge with the agents' tails and one
inverse FWHT per row. Within 2e-3 of the oracle's float64 attention on the
workloads' shapes, with tails, on block-scaled and per-group-width layers;
argument errors."""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, to_dev

pytestmark = pytest.mark.gpu

ERR_INVALID_ARG, ERR_UNSUPPORTED = -1, -7


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _dev_tail(tail):
    import torch

    if tail is None:
        return None
    Kt, Vt, lens = tail
    return (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())


def _check(kp, w, layer, k_block=0, tail=None, rows=None, step=0):
    K, V = wl.layer_kv(w, layer)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [w.layer_bits(layer)], max_rows=w.rows, k_block=k_block)
    pool.compress(0, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, w.layer_bits(layer), k_block=k_block)
    Q = wl.layer_q(w, layer, step)
    out = pool.attend_ws(0, to_dev(Q), tail=_dev_tail(tail))
    assert pool.status() == 0
    err = attention_error(out, enc, Q, tail, rows=rows)
    assert err <= TOL, err
    pool.close()
    return err


def _rows(w, n=32, seed=0):
    rng = np.random.default_rng(seed)
    return [(int(a), int(h)) for a, h in zip(rng.integers(0, w.agents, n), rng.integers(0, w.q_heads, n))]


SMALL = [
    # name, Hk, Hq, d, ctx, agents, bits, tail_init
    ("ws_tiny_like", 2, 4, 64, 256, 3, 3, 0),
    ("ws_gqa4_ragged_2bit", 4, 16, 128, 300, 5, 2, 0),
    ("ws_gqa8_4bit_tail", 2, 16, 128, 1000, 2, 4, 7),
    ("ws_one_tile", 3, 3, 64, 100, 1, 3, 0),
    ("ws_d64_many_slices_tail", 2, 4, 64, 5000, 6, 3, 20),
    ("ws_200_rows", 1, 40, 128, 3000, 5, 3, 0),  # two row groups of whole agents
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(kp, case):
    name, Hk, Hq, d, ctx, A, bits, tail_init = case
    w = wl.custom(name, 1, Hk, Hq, d, ctx, A, "lognormal", tail_init, 2, (bits,))
    tail = None
    if tail_init:
        Kt, Vt = wl.layer_tail(w, 0)
        tail = (Kt, Vt, np.array([(a * 3) % (w.tail_max + 1) for a in range(A)]))
    _check(kp, w, 0, tail=tail)


@pytest.mark.parametrize("name,layer", [("llama3_8b_4k", 5), ("smollm2_2k", 7)])
def test_full_size_layer(kp, name, layer):
    _check(kp, wl.WORKLOADS[name], layer)


def test_llama_long_with_tails(kp):
    w = wl.WORKLOADS["llama3_8b_long"]
    Kt, Vt = wl.layer_tail(w, 3)
    _check(kp, w, 3, tail=(Kt, Vt, np.full(w.agents, w.tail_len(2))), step=2)


def test_qwen_shaped_layer_sampled_rows(kp):
    """Qwen3-32B shape (8 KV heads, 64 query heads, 32 agents: 256 rows per
    KV head in two row groups) over 16K tokens, 4-bit V; sampled rows."""
    w = wl.custom("ws_qwen_like", 1, 8, 64, 128, 16384, 32, "lognormal", 0, 1, (4,))
    _check(kp, w, 0, rows=_rows(w))


def test_block_scaled_and_mixed_width(kp):
    import torch

    w = wl.custom("ws_kb", 1, 4, 16, 128, 2100, 5, "lognormal", 9, 2, (3,))
    Kt, Vt = wl.layer_tail(w, 0)
    tail = (Kt, Vt, np.array([(a * 2) % 10 for a in range(w.agents)]))
    _check(kp, w, 0, k_block=32, tail=tail)
    # a layer grown at widths 4, 2, 3
    K, V = wl.layer_kv(w, 0)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [4], max_rows=w.rows, k_block=32)
    widths, a = [], 0
    for b, bw in ((640, 4), (1280, 2), (2100, 3)):
        pool.append(0, to_dev(np.ascontiguousarray(K[:, a:b])), to_dev(np.ascontiguousarray(V[:, a:b])), bits=bw)
        widths += [bw] * ((b - a + 31) // 32)
        a = b
    enc = codec.encode_layer_groups(K, V, widths)
    Q = wl.layer_q(w, 0)
    out = pool.attend_ws(0, to_dev(Q), tail=_dev_tail(tail))
    assert pool.status() == 0
    assert attention_error(out, enc, Q, tail) <= TOL
    ws = torch.empty(pool.attend_ws_bytes(w.agents, w.q_heads), dtype=torch.uint8, device="cuda")
    out2 = pool.attend_ws(0, to_dev(Q), ws, tail=_dev_tail(tail))  # a given workspace, reused
    assert torch.equal(out, out2)
    pool.close()


def test_workspace_errors(kp):
    import torch

    w = wl.custom("ws_err", 1, 2, 8, 64, 1000, 3, "lognormal")
    K, V = wl.layer_kv(w, 0)
    pool = kp.KVPool(1, 2, 64, 1000, [3], max_rows=w.rows)
    pool.compress(0, to_dev(K), to_dev(V))
    Q = to_dev(wl.layer_q(w, 0))
    need = pool.attend_ws_bytes(w.agents, w.q_heads)
    assert need > 0
    assert pool.attend_ws_bytes(0, w.q_heads) == 0 and pool.attend_ws_bytes(w.agents, 3) == 0
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    for bad in (ws[:need - 16], ws[1:need + 1]):  # short, misaligned
        with pytest.raises(kp.KVPoolError) as e:
            pool.attend_ws(0, Q, bad)
        assert e.value.code == ERR_INVALID_ARG
    pool.close()
    # more (KV head, row group) pairs than SMs: no wave of one CTA each
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = kp.KVPool(1, sms + 8, 64, 128, [3])
    assert big.attend_ws_bytes(1, sms + 8) == 0
    wb = wl.custom("ws_many_heads", 1, sms + 8, sms + 8, 64, 128, 1, "lognormal")
    Kb, Vb = wl.layer_kv(wb, 0)
    big.compress(0, to_dev(Kb), to_dev(Vb))
    with pytest.raises(kp.KVPoolError) as e:
        big.attend_ws(0, to_dev(wl.layer_q(wb, 0)), torch.empty(1024, dtype=torch.uint8, device="cuda"))
    assert e.value.code == ERR_UNSUPPORTED
    big.close()


def test_recompress_right_after_attention_same_stream(kp):
    # attend_ws, then the same layer re-armed and compressed with other data,
    # then attend_ws again, all queued on one stream with no host sync: the
    # writers of the layer must not start before the first attention (and
    # the merge that releases its dependents early) is done with it. Full
    # Llama-4K-shaped layer, so the merge takes the spread launch.
    import torch

    w = wl.WORKLOADS["llama3_8b_4k"]
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3], max_rows=w.rows)
    data = [wl.layer_kv(w, l) for l in (0, 1)]
    Q = wl.layer_q(w, 0, 0)
    Qd = to_dev(Q)
    outs = []
    for rep in range(2):
        for K, V in data:
            pool.reset_layer(0)
            pool.compress(0, to_dev(K), to_dev(V))
            outs.append(pool.attend_ws(0, Qd))
    torch.cuda.synchronize()
    assert pool.status() == 0
    rows = _rows(w, 24, seed=3)
    for i, out in enumerate(outs):
        K, V = data[i % 2]
        enc = codec.encode_layer(K, V, 3)
        err = attention_error(out, enc, Q, None, rows=rows)
        assert err <= TOL, (i, err)
    pool.close()
