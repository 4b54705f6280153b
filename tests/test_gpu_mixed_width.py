"""GPU parity of appends at new V widths (kvpool_append_bits): a block-scaled
layer grows by groups whose widths the allocator chose when they were
quantised (CoMixKV article, incremental quantisation strategy: a new width
applies only to blocks quantised afterwards; old blocks are never
rewritten). After each append the stored bytes equal the oracle's per-group
encode, bytes written earlier are unchanged, decompress is bit-exact, and
attention (whole layer, tails, context slices) is within 2e-3."""

import numpy as np
import pytest

from oracle import allocator, attention, codec
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


def _widths_of(cuts, bws):
    """Per-group widths of a layer built by appends [cuts[i-1], cuts[i]) at bws[i]."""
    out, a = [], 0
    for b, w in zip(cuts, bws):
        out += [w] * ((b - a + 31) // 32)
        a = b
    return out


def _grow(kp, w, cuts, bws, create_bits, tail_lens=None, rows=None):
    import torch

    K, V = wl.layer_kv(w, 0)
    Q = wl.layer_q(w, 0)
    dev_tail = host_tail = None
    if tail_lens is not None:
        Kt, Vt = wl.layer_tail(w, 0)
        dev_tail = (to_dev(Kt), to_dev(Vt), torch.from_numpy(tail_lens.astype(np.int32)).cuda())
        host_tail = (Kt, Vt, tail_lens)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [create_bits], max_rows=w.rows, k_block=32)
    prev, a = None, 0
    for b, bw in zip(cuts, bws):
        pool.append(0, to_dev(np.ascontiguousarray(K[:, a:b])), to_dev(np.ascontiguousarray(V[:, a:b])), bits=bw)
        a = b
        widths = _widths_of(cuts[:cuts.index(b) + 1], bws)
        assert pool.layer_widths(0) == widths
        assert pool.layer_view(0).mixed == int(any(x != create_bits for x in widths))
        enc = codec.encode_layer_groups(K[:, :b], V[:, :b], widths)
        check_encode(pool, 0, enc)
        got = pool.read_layer(0)["vcodes"].reshape(w.kv_heads, -1)
        if prev is not None:  # the bytes of earlier groups never change
            assert np.array_equal(got[:, :prev.shape[1]], prev)
        prev = got
        check_decompress(pool, 0, enc)
        out = pool.attend(0, to_dev(Q), tail=dev_tail)
        assert pool.status() == 0
        err = attention_error(out, enc, Q, host_tail, rows=rows)
        assert err <= TOL, (b, err)
    return pool, K, V, Q, enc


@pytest.mark.parametrize("d,create_bits,cuts,bws", [
    (128, 4, (64, 160, 230), (2, 4, 3)),          # 2, then 4, then 3 bits; a ragged last append
    (64, 4, (32, 96, 128, 300), (3, 2, 4, 2)),   # group widths changing inside tiles
    (128, 3, (128, 256, 384, 500), (2, 3, 2, 3)),
    (64, 3, (96, 416), (3, 2)),                  # the create width first (uniform), then mixed
])
def test_appends_at_new_widths(kp, d, create_bits, cuts, bws):
    w = wl.custom("mixw", 1, 2, 8, d, cuts[-1] + 40, 3, "lognormal")
    pool, *_ = _grow(kp, w, list(cuts), list(bws), create_bits)
    pool.close()


def test_mixed_layer_llama_shape_with_tails(kp):
    """Llama-3-8B-shaped layer (8 KV heads, 32 query heads, 15 agents, d 128)
    grown to 1,400 tokens in blocks of 2, 4, 3 and 2 bits, with the agents'
    bf16 tails; sampled rows."""
    w = wl.custom("mixw_llama", 1, 8, 32, 128, 1400, 15, "lognormal", 24)
    tail_lens = np.array([(5 * a) % 25 for a in range(15)])
    rng = np.random.default_rng(5)
    rows = [(int(a), int(h)) for a, h in zip(rng.integers(0, 15, 40), rng.integers(0, 32, 40))]
    pool, *_ = _grow(kp, w, [256, 640, 1152, 1400], [2, 4, 3, 2], 4, tail_lens, rows)
    pool.close()


def test_mixed_layer_context_slices(kp):
    """Partial attention over slices of a mixed layer merges to the oracle's
    attention over all its tokens."""
    import torch

    w = wl.custom("mixw_split", 1, 2, 8, 128, 700, 4, "lognormal")
    pool, K, V, Q, enc = _grow(kp, w, [192, 416, 700], [4, 2, 3], 4)
    Kh, Vh = attention.dequantise_f64(enc)
    ref = attention.attend_f64(Kh, Vh, Q)
    dQ = to_dev(Q)
    mls, accs = [], []
    for t0, t1 in ((0, 256), (256, 384), (384, 700)):
        ml, acc = pool.attend_partial(0, dQ, t0, t1)
        mls.append(ml)
        accs.append(acc)
    out = kp.merge_partials(torch.stack(mls), torch.stack(accs), dQ, w.kv_heads)
    assert pool.status() == 0
    assert attention.row_rel_error(out.cpu().numpy().astype(np.float64), ref) <= TOL
    pool.close()


def test_allocator_refresh_sets_new_block_widths(kp):
    """The controller loop: new observations -> sensitivity -> joint
    allocation under a byte budget -> the next blocks of every layer appended
    at their new widths; the first blocks keep the widths of the first
    allocation."""
    import torch

    w = wl.custom("mixw_alloc", 3, 2, 8, 64, 512, 4, "lognormal", 48, 2)
    pool = kp.KVPool(3, w.kv_heads, w.head_dim, w.ctx, [4, 4, 4], max_rows=w.rows, k_block=32)
    per_bit = w.kv_heads * 256 * w.head_dim // 8
    chosen = []
    for step, (a, b) in enumerate(((0, 256), (256, 512))):
        lens = np.full(w.agents, 16 + 16 * step)
        sens = []
        for l in range(3):
            Kt, Vt = wl.layer_tail(w, l, seed=step)
            s, _ = kp.sensitivity(to_dev(wl.layer_q(w, l, step)), (to_dev(Kt), to_dev(Vt),
                                  torch.from_numpy(lens.astype(np.int32)).cuda()), w.kv_heads)
            sens.append(s)
        bits = kp.allocate_bits(sens, [per_bit] * 3, (8 + step) * per_bit)
        assert bits == list(allocator.allocate(sens, [1] * 3, 8 + step))
        chosen.append(bits)
        for l in range(3):
            K, V = wl.layer_kv(w, l)
            pool.append(l, to_dev(np.ascontiguousarray(K[:, a:b])), to_dev(np.ascontiguousarray(V[:, a:b])),
                        bits=bits[l])
    for l in range(3):
        widths = [chosen[0][l]] * 8 + [chosen[1][l]] * 8
        assert pool.layer_widths(l) == widths
        K, V = wl.layer_kv(w, l)
        enc = codec.encode_layer_groups(K, V, widths)
        check_encode(pool, l, enc)
        Q = wl.layer_q(w, l)
        out = pool.attend(l, to_dev(Q))
        assert pool.status() == 0
        assert attention_error(out, enc, Q) <= TOL
    pool.close()


def test_append_width_errors(kp):
    w = wl.custom("mixw_err", 1, 2, 4, 64, 200, 2, "lognormal")
    K, V = wl.layer_kv(w, 0)
    dK, dV = to_dev(K), to_dev(V)
    pool = kp.KVPool(1, 2, 64, 200, [3], k_block=32)
    for bad in (1, 4, 5):  # outside [2, create width 3]
        with pytest.raises(kp.KVPoolError) as e:
            pool.append(0, dK[:, :32].contiguous(), dV[:, :32].contiguous(), bits=bad)
        assert e.value.code == ERR_INVALID_ARG
    assert pool.layer_len(0) == 0 and pool.layer_widths(0) == []
    pool.append(0, dK[:, :64].contiguous(), dV[:, :64].contiguous(), bits=2)
    assert pool.layer_widths(0) == [2, 2]
    # reset forgets the widths; compress writes every group at the create width
    pool.reset_layer(0)
    assert pool.layer_widths(0) == []
    pool.compress(0, dK, dV)
    assert pool.status() == 0 and pool.layer_widths(0) == [3] * 7 and not pool.layer_view(0).mixed
    check_encode(pool, 0, codec.encode_layer(K, V, 3, k_block=32))
    pool.close()
    per_tensor = kp.KVPool(1, 2, 64, 200, [3])
    with pytest.raises(kp.KVPoolError) as e:
        per_tensor.append(0, dK[:, :32].contiguous(), dV[:, :32].contiguous(), bits=2)
    assert e.value.code == ERR_UNSUPPORTED
    per_tensor.close()


@pytest.mark.parametrize("host", [False, True])
def test_handoff_of_a_grown_layer(kp, host):
    """A block-scaled layer grown at widths 2, 4, 3 is exported (bytes, block
    scales, widths) and loaded into a fresh pool (QKVShare blog, section 3.1:
    the quantised cache travels with its scales): the same bytes, decompress
    and attention against the oracle; the loaded layer then takes a further
    append."""
    import torch

    w = wl.custom("mixw_handoff", 1, 2, 8, 128, 600, 3, "lognormal")
    pool, K, V, Q, enc = _grow(kp, w, [128, 320, 416], [2, 4, 3], 4)
    kq, vc, vn, _ = pool.export_layer(0)
    ks = pool.export_kscales(0)
    widths = pool.layer_widths(0)
    if host:  # pinned host buffers
        kq, vc, vn, ks = (t.cpu().pin_memory() for t in (kq, vc, vn, ks))
    dst = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [4], max_rows=w.rows, k_block=32)
    dst.import_layer_blocks(0, kq, vc, vn, ks, widths)
    torch.cuda.synchronize()
    assert dst.layer_len(0) == 416 and dst.layer_widths(0) == widths and dst.layer_view(0).mixed
    check_encode(dst, 0, enc)
    check_decompress(dst, 0, enc)
    out = dst.attend(0, to_dev(Q))
    assert dst.status() == 0
    assert attention_error(out, enc, Q) <= TOL
    with pytest.raises(kp.KVPoolError) as e:  # write-once
        dst.import_layer_blocks(0, kq, vc, vn, ks, widths)
    assert e.value.code == ERR_STATE
    # the loaded layer grows on
    dst.append(0, to_dev(np.ascontiguousarray(K[:, 416:600])), to_dev(np.ascontiguousarray(V[:, 416:600])), bits=2)
    widths2 = widths + [2] * 6
    enc2 = codec.encode_layer_groups(K[:, :600], V[:, :600], widths2)
    check_encode(dst, 0, enc2)
    out = dst.attend(0, to_dev(Q))
    assert dst.status() == 0
    assert attention_error(out, enc2, Q) <= TOL
    dst.close()
    pool.close()


def test_import_blocks_errors(kp):
    import torch

    w = wl.custom("mixw_imp_err", 1, 2, 4, 64, 200, 2, "lognormal")
    pool = kp.KVPool(1, 2, 64, 200, [3], k_block=32)
    kq = torch.zeros((2, 64, 64), dtype=torch.int8, device="cuda")
    vc = torch.zeros((2, 2 * 64 * 12), dtype=torch.uint8, device="cuda")
    vn = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    ks = torch.ones((2, 64, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(kp.KVPoolError) as e:  # a width above the create width
        pool.import_layer_blocks(0, kq, vc, vn, ks, [3, 4])
    assert e.value.code == ERR_INVALID_ARG
    assert pool.layer_len(0) == 0
    per_tensor = kp.KVPool(1, 2, 64, 200, [3])
    with pytest.raises(kp.KVPoolError) as e:
        per_tensor.import_layer_blocks(0, kq, vc, vn, ks, [3, 3])
    assert e.value.code == ERR_UNSUPPORTED
    per_tensor.close()
    # all-zero codes and norms with unit scales: a layer of zeros, attended to zero output
    pool.import_layer_blocks(0, kq, vc, vn, ks, [3, 3])
    Q = to_dev(wl.layer_q(w, 0))
    out = pool.attend(0, Q)
    assert pool.status() == 0 and float(out.abs().max()) == 0.0
    pool.close()
