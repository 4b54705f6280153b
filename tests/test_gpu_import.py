"""The quantised-cache handoff (QKVShare blog, section 3.1: the sender packs
the quantised cache with its scales, the receiver loads it instead of
recomputing): a per-tensor layer exported from one pool and imported into a
fresh pool must hold the oracle's bytes bit for bit, decompress bit-exactly,
and attend within 2e-3 of the oracle. Exports to host memory and to device
memory are both covered, and a second import into the same layer is refused
(write-once)."""

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, check_decompress, check_encode, to_dev

pytestmark = pytest.mark.gpu

STATE = -2


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


@pytest.mark.parametrize("to_host", [False, True], ids=["device", "host"])
@pytest.mark.parametrize("case", [
    # name, Hk, Hq, d, ctx, agents, bits, tail_init
    ("import_llama_like", 8, 32, 128, 1000, 15, 3, 0),
    ("import_d64_2bit_tail", 4, 8, 64, 333, 3, 2, 6),
    ("import_4bit", 2, 16, 128, 257, 2, 4, 0),
], ids=lambda c: c[0] if isinstance(c, tuple) else None)
def test_export_import_round_trip(kp, case, to_host):
    import torch

    _, Hk, Hq, d, ctx, A, bits, tail_init = case
    w = wl.custom(case[0], 2, Hk, Hq, d, ctx, A, "lognormal", tail_init, 1, (bits, bits))
    src = kp.KVPool(2, Hk, d, ctx, [bits, bits])
    K, V = wl.layer_kv(w, 1)
    src.compress(1, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, bits)
    kq, vc, vn, ks = src.export_layer(1)
    if to_host:
        kq, vc, vn, ks = (t.cpu().pin_memory() for t in (kq, vc, vn, ks))
    torch.cuda.synchronize()
    src.close()  # the receiver holds its own copy

    dst = kp.KVPool(2, Hk, d, ctx, [bits, bits])
    dst.import_layer(0, kq, vc, vn, ks)
    torch.cuda.synchronize()
    assert dst.status() == 0
    assert dst.layer_view(0).compressed == 1 and dst.layer_len(0) == ctx
    check_encode(dst, 0, enc)
    check_decompress(dst, 0, enc)
    Q = wl.layer_q(w, 1)
    tail_dev = host_tail = None
    if tail_init:
        Kt, Vt = wl.layer_tail(w, 1)
        lens = np.array([(a * 5) % (w.tail_max + 1) for a in range(A)])
        tail_dev = (to_dev(Kt), to_dev(Vt), torch.from_numpy(lens.astype(np.int32)).cuda())
        host_tail = (Kt, Vt, lens)
    out = dst.attend(0, to_dev(Q), tail=tail_dev)
    assert dst.status() == 0
    err = attention_error(out, enc, Q, host_tail)
    assert err <= TOL, err
    with pytest.raises(kp.KVPoolError) as e:  # write-once
        dst.import_layer(0, kq, vc, vn, ks)
    assert e.value.code == STATE
    dst.close()
