"""The context split of one shared pool across ranks, on CPU: two and three
gloo ranks (127.0.0.1) each hold a tile-aligned slice of one layer's
context, compute their slice's softmax state with the oracle, exchange the
states through the module's all-gather, and merge; every rank must get the
oracle's attention over the whole context (with the agents' tails) to 1e-10.
The library's own partial and merge calls are checked against the oracle on
the GPU (test_gpu_context_split.py); this test covers the host side: the
slice bounds, the exchange and its rank order."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer():
    from oracle import attention, codec
    from shared_quantized_kv_gb300 import workloads as wl

    w = wl.custom("cp", 1, 2, 8, 64, 700, 3, "lognormal", 6, 1, (3,))
    K, V = wl.layer_kv(w, 0)
    enc = codec.encode_layer(K, V, 3)
    Kh, Vh = attention.dequantise_f64(enc)
    Q = wl.layer_q(w, 0)
    Kt, Vt = wl.layer_tail(w, 0)
    tail = (Kt, Vt, np.array([6, 0, 3]))
    return w, Kh, Vh, Q, tail


def _rank_main(rank, world, port, out):
    import sys

    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    from oracle import attention
    from shared_quantized_kv_gb300 import context_parallel as cp

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, Kh, Vh, Q, tail = _layer()
    b, e = cp.slice_bounds(w.ctx, rank, world)

    def partial(layer, Q_):
        lse, o = attention.attend_slice_f64(Kh, Vh, Q_, b, e)
        return torch.from_numpy(lse), torch.from_numpy(o)

    def merge(ML, ACC, Q_, tail_):
        parts = [(ML[s].numpy(), ACC[s].numpy()) for s in range(ML.shape[0])]
        parts.append(attention.tail_slice_f64(Q_, tail_, w.kv_heads))
        return attention.merge_slices_f64(parts)

    got = cp.attend(None, 0, Q, tail, partial=partial, merge=merge)
    want = attention.attend_f64(Kh, Vh, Q, tail)
    out[rank] = (float(np.abs(got - want).max()), (b, e))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_merge_to_full_attention(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    spans = [res[r][1] for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == 700
    assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))  # contiguous, in rank order
    assert all(s[0] % 128 == 0 for s in spans)
    for r in range(world):
        assert res[r][0] < 1e-10, (r, res[r])


def test_slice_bounds():
    import sys

    sys.path.insert(0, ROOT)
    from shared_quantized_kv_gb300 import context_parallel as cp

    assert cp.slice_bounds(4096, 0, 2) == (0, 2048) and cp.slice_bounds(4096, 1, 2) == (2048, 4096)
    assert [cp.slice_bounds(700, r, 3) for r in range(3)] == [(0, 256), (256, 512), (512, 700)]
    # more ranks than tiles: the last ranks hold nothing
    assert [cp.slice_bounds(200, r, 4) for r in range(4)] == [(0, 128), (128, 200), (200, 200), (200, 200)]
    with pytest.raises(ValueError):
        cp.slice_bounds(100, 2, 2)
