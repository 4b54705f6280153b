"""kvpool_attend_noalloc, the allocation-free attention entry point, called
through the C-ABI and compared with kvpool_attend on the same layer.

The entry point serves callers that cannot call cudaMalloc (an engine that
reserved all device memory itself, or a caller that cannot afford the
synchronisation cudaMalloc implies): its scratch is a fixed array inside the
library that every call reuses. Two calls in a row, the second with other
queries, must each match the regular entry point -- the second call reads no
stale partials of the first. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, to_dev

pytestmark = pytest.mark.gpu


def _row_err(a, b):
    a = a.reshape(-1, a.shape[-1]).double()
    b = b.reshape(-1, b.shape[-1]).double()
    return float(((a - b).abs().amax(1) / b.abs().amax(1).clamp_min(1e-30)).max())


def test_noalloc_matches_attend_on_two_calls():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    build.build()
    lib = kvpool.lib()
    w = wl.custom("noalloc", 1, 4, 16, 128, 1500, 5, "lognormal", 9, 2, (3,))
    pool = kvpool.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3])
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    Kt, Vt = wl.layer_tail(w, 0)
    lens = torch.tensor([0, 3, 10, 7, 1], dtype=torch.int32, device="cuda")
    tail_dev = (to_dev(Kt), to_dev(Vt), lens)
    tail = kvpool.Tail(tail_dev[0].data_ptr(), tail_dev[1].data_ptr(), lens.data_ptr(), Kt.shape[2])
    view = pool.layer_view(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    for step in range(2):
        Q = to_dev(wl.layer_q(w, 0, step))
        ref = pool.attend(0, Q, tail=tail_dev)
        out = torch.full((w.agents, w.q_heads, w.head_dim), float("nan"), device="cuda")
        rc = lib.kvpool_attend_noalloc(view.kq, view.vcodes, view.vnorm, view.kscale, w.kv_heads,
                                       w.head_dim, w.ctx, 3, Q.data_ptr(), w.agents, w.q_heads,
                                       ctypes.byref(tail), out.data_ptr(), 0.0, stream)
        assert rc == 0, kvpool.ERRORS.get(rc, rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err = _row_err(out, ref)
        assert err <= TOL, (step, err)

    # a shape whose split partials cannot fit the fixed scratch is refused
    too_many = 1 << 20
    rc = lib.kvpool_attend_noalloc(view.kq, view.vcodes, view.vnorm, view.kscale, 64, 128, w.ctx,
                                   3, Q.data_ptr(), too_many // 64, 64 * 4, None, out.data_ptr(),
                                   0.0, stream)
    assert rc == -1
    assert pool.status() == 0
    pool.close()
