"""The context split through the C-ABI (kvpool_attend_partial,
kvpool_merge_partials) against the CPU oracle.

One pool; its context is cut into tile-aligned slices (one, two, three and
many parts, uneven, and a slice that neither starts nor ends at the context
ends). For every slice the library's state is checked against the oracle's
state of that slice: the slice's output H acc / (D l) within 2e-3 (the
attention metric) and its log-sum-exp m + log2 l within 1e-3 (log2 units).
The merged parts, with and without the agents' bf16 tails, must give the
oracle's attention over the whole context within 2e-3 and agree with
kvpool_attend. Argument errors are refused. Block-scaled pools take the same
calls."""

import numpy as np
import pytest

from oracle import attention, codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, to_dev

pytestmark = pytest.mark.gpu

INVALID_ARG = -1


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _row_err(a, b):
    return attention.row_rel_error(np.asarray(a), np.asarray(b))


def _setup(kp, w, bits):
    import torch

    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [bits], max_rows=w.rows)
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, bits)
    Kh, Vh = attention.dequantise_f64(enc)
    Qh = wl.layer_q(w, 0)
    return pool, Kh, Vh, Qh, to_dev(Qh)


def _slice_state(ml, acc, d, G):
    """(lse2 [A, Hq], o [A, Hq, d]) of a library partial ([Hk, R, 2], [Hk, R, d])."""
    ml, acc = ml.cpu().numpy().astype(np.float64), acc.cpu().numpy().astype(np.float64)
    Hk, R, _ = ml.shape
    A = R // G
    H = attention.hadamard(d)
    o = (acc @ H) / (d * ml[..., 1:2])
    lse = ml[..., 0] + np.log2(ml[..., 1])
    # rows r = a * G + j of head g -> (a, g * G + j)
    o = o.reshape(Hk, A, G, d).transpose(1, 0, 2, 3).reshape(A, Hk * G, d)
    lse = lse.reshape(Hk, A, G).transpose(1, 0, 2).reshape(A, Hk * G)
    return lse, o


CASES = [
    # name, Hk, Hq, d, ctx, agents, bits, cuts (token offsets, multiples of 128)
    ("llama_like_2", 8, 32, 128, 1500, 15, 3, [768]),
    ("gqa8_3parts_4bit", 2, 16, 128, 1000, 16, 4, [128, 640]),
    ("d64_mha_many", 4, 4, 64, 900, 5, 2, [128, 256, 384, 512, 640, 768]),
    ("one_part", 2, 8, 128, 300, 3, 3, []),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_slices_and_merge(kp, case):
    import torch

    _, Hk, Hq, d, ctx, A, bits, cuts = case
    w = wl.custom(case[0], 1, Hk, Hq, d, ctx, A, "lognormal", 5, 1, (bits,))
    G = Hq // Hk
    pool, Kh, Vh, Qh, Q = _setup(kp, w, bits)
    edges = [0] + cuts + [ctx]
    MLs, ACCs = [], []
    for b, e in zip(edges[:-1], edges[1:]):
        ml, acc = pool.attend_partial(0, Q, b, e)
        lse_g, o_g = _slice_state(ml, acc, d, G)
        lse_r, o_r = attention.attend_slice_f64(Kh, Vh, Qh, b, e)
        assert _row_err(o_g, o_r) <= TOL, ("slice", b, e, _row_err(o_g, o_r))
        assert np.abs(lse_g - lse_r).max() <= 1e-3, ("lse", b, e, np.abs(lse_g - lse_r).max())
        MLs.append(ml)
        ACCs.append(acc)
    ML, ACC = torch.stack(MLs), torch.stack(ACCs)
    # in any order of the parts
    perm = list(range(len(MLs)))[::-1]
    out = kp.merge_partials(ML[perm].contiguous(), ACC[perm].contiguous(), Q, Hk)
    ref = attention.attend_f64(Kh, Vh, Qh)
    assert _row_err(out.cpu().numpy(), ref) <= TOL
    assert _row_err(out.cpu().numpy(), pool.attend(0, Q).cpu().numpy()) <= TOL
    # with the agents' tails
    Kt, Vt = wl.layer_tail(w, 0)
    lens = np.array([(a * 2) % (w.tail_max + 1) for a in range(A)])
    dev_tail = (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())
    out_t = kp.merge_partials(ML, ACC, Q, Hk, dev_tail)
    ref_t = attention.attend_f64(Kh, Vh, Qh, (Kt, Vt, lens))
    assert _row_err(out_t.cpu().numpy(), ref_t) <= TOL
    assert pool.status() == 0
    pool.close()


def test_inner_slice(kp):
    # a slice that starts and ends inside the context
    w = wl.custom("inner", 1, 2, 8, 128, 1000, 4, "lognormal", 0, 1, (3,))
    pool, Kh, Vh, Qh, Q = _setup(kp, w, 3)
    ml, acc = pool.attend_partial(0, Q, 256, 777)
    lse_g, o_g = _slice_state(ml, acc, 128, 4)
    lse_r, o_r = attention.attend_slice_f64(Kh, Vh, Qh, 256, 777)
    assert _row_err(o_g, o_r) <= TOL
    assert np.abs(lse_g - lse_r).max() <= 1e-3
    pool.close()


def test_refusals(kp):
    import torch

    w = wl.custom("cp_err", 1, 2, 4, 64, 300, 2, "lognormal")
    pool, _, _, _, Q = _setup(kp, w, 3)
    for b, e in [(64, 200), (0, 301), (256, 256), (-128, 100)]:  # unaligned, past the end, empty, negative
        with pytest.raises(kp.KVPoolError) as err:
            pool.attend_partial(0, Q, b, e)
        assert err.value.code == INVALID_ARG, (b, e)
    pool.close()


def test_block_scaled_slices(kp):
    # block-scaled K: slice states and their merge against the oracle
    import torch

    w = wl.custom("cp_kb", 1, 4, 16, 128, 1100, 5, "lognormal", 0, 1, (3,))
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3], k_block=32)
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    Kh, Vh = attention.dequantise_f64(codec.encode_layer(K, V, 3, k_block=32))
    Qh = wl.layer_q(w, 0)
    Q = to_dev(Qh)
    MLs, ACCs = [], []
    for b, e in [(0, 384), (384, 1100)]:
        ml, acc = pool.attend_partial(0, Q, b, e)
        lse_g, o_g = _slice_state(ml, acc, 128, 4)
        lse_r, o_r = attention.attend_slice_f64(Kh, Vh, Qh, b, e)
        assert _row_err(o_g, o_r) <= TOL
        assert np.abs(lse_g - lse_r).max() <= 1e-3
        MLs.append(ml)
        ACCs.append(acc)
    out = kp.merge_partials(torch.stack(MLs), torch.stack(ACCs), Q, w.kv_heads)
    assert _row_err(out.cpu().numpy(), attention.attend_f64(Kh, Vh, Qh)) <= TOL
    assert pool.status() == 0
    pool.close()


def test_merge_of_many_slices(kp):
    """40 one-tile slices (more than one warp's lanes hold: the merge reads the
    (m, l) of slices 32.. in its second loop), with some slices repeated as
    empty parts (l = 0), merged with tails, against the oracle."""
    import torch

    Hk, Hq, d, ctx, A = 2, 8, 64, 40 * 128 - 50, 3
    w = wl.custom("many_slices", 1, Hk, Hq, d, ctx, A, "lognormal", 6, 1, (3,))
    pool, Kh, Vh, Qh, Q = _setup(kp, w, 3)
    edges = list(range(0, ctx, 128)) + [ctx]
    MLs, ACCs = [], []
    for b, e in zip(edges[:-1], edges[1:]):
        ml, acc = pool.attend_partial(0, Q, b, e)
        MLs.append(ml)
        ACCs.append(acc)
    assert len(MLs) == 40
    # three empty parts (l = 0) among them, one in the first 16: neither their
    # m nor their accumulator (NaN here) may count
    empty_ml = torch.zeros_like(MLs[0])
    empty_ml[..., 0] = 1e30
    for at in (5, 17, 36):
        MLs.insert(at, empty_ml)
        ACCs.insert(at, torch.full_like(ACCs[0], float("nan")))
    ML, ACC = torch.stack(MLs), torch.stack(ACCs)
    Kt, Vt = wl.layer_tail(w, 0)
    lens = np.array([(a * 2) % (w.tail_max + 1) for a in range(A)])
    dev_tail = (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())
    out = kp.merge_partials(ML, ACC, Q, Hk, dev_tail)
    assert pool.status() == 0
    ref = attention.attend_f64(Kh, Vh, Qh, (Kt, Vt, lens))
    assert _row_err(out.cpu().numpy(), ref) <= TOL
    pool.close()
