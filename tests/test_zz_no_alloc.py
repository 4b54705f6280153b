"""kvpool_attend_noalloc, the allocation-free attention entry point, called
through the C-ABI and checked against the CPU oracle and against
kvpool_attend on the same layer.

The entry point serves callers that cannot call cudaMalloc (an engine that
reserved all device memory itself, or a caller that cannot afford the
synchronisation cudaMalloc implies): its scratch is a fixed array inside the
library that every call reuses. Each output is compared with the oracle's
float64 attention over the same dequantised layer (the parity bar) and with
kvpool_attend's output. Two calls in a row, the second with other queries,
must each pass: the second reads no stale partials of the first. The shapes
cover a per-tensor layer with tails, a block-scaled layer (its scales passed
in), a call whose splits are cut down to fit the fixed array, and the two
refusals (too many rows; partials of one split larger than the array). This
file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

from oracle import codec
from shared_quantized_kv_gb300 import workloads as wl

from parity_util import TOL, attention_error, to_dev

pytestmark = pytest.mark.gpu

INVALID_ARG = -1
SCRATCH_BYTES = 8 << 20  # the library's fixed split scratch


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _row_err(a, b):
    a = a.reshape(-1, a.shape[-1]).double()
    b = b.reshape(-1, b.shape[-1]).double()
    return float(((a - b).abs().amax(1) / b.abs().amax(1).clamp_min(1e-30)).max())


def _noalloc(kp, view, w, bits, Q, out, tail=None, kscales=None):
    import torch

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return kp.lib().kvpool_attend_noalloc(view.kq, view.vcodes, view.vnorm, view.kscale, kscales,
                                          w.kv_heads, w.head_dim, w.ctx, bits, Q.data_ptr(), w.agents,
                                          w.q_heads, tail, out.data_ptr(), 0.0, stream)


def _two_calls(kp, w, bits, k_block=0, tail_lens=None, max_rows=0):
    """Compress one layer, then run the allocation-free entry point twice
    (decode steps 0 and 1) and check each output against the oracle and
    against kvpool_attend."""
    import torch

    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [bits], max_rows=max_rows, k_block=k_block)
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    enc = codec.encode_layer(K, V, bits, k_block=k_block)
    tail_dev = host_tail = tail = None
    if tail_lens is not None:
        Kt, Vt = wl.layer_tail(w, 0)
        lens = torch.from_numpy(tail_lens.astype(np.int32)).cuda()
        tail_dev = (to_dev(Kt), to_dev(Vt), lens)
        host_tail = (Kt, Vt, tail_lens)
        tail = kp.Tail(tail_dev[0].data_ptr(), tail_dev[1].data_ptr(), lens.data_ptr(), Kt.shape[2])
    view = pool.layer_view(0)
    assert (view.kscales is not None) == bool(k_block)
    for step in range(2):
        Qh = wl.layer_q(w, 0, step)
        Q = to_dev(Qh)
        ref = pool.attend(0, Q, tail=tail_dev)
        out = torch.full((w.agents, w.q_heads, w.head_dim), float("nan"), device="cuda")
        rc = _noalloc(kp, view, w, bits, Q, out, ctypes.byref(tail) if tail else None, view.kscales)
        assert rc == 0, kp.ERRORS.get(rc, rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err_oracle = attention_error(out, enc, Qh, host_tail)
        assert err_oracle <= TOL, ("oracle", step, err_oracle)
        err_attend = _row_err(out, ref)
        assert err_attend <= TOL, ("kvpool_attend", step, err_attend)
    assert pool.status() == 0
    return pool


def test_per_tensor_layer_with_tails_two_calls(kp):
    w = wl.custom("noalloc", 1, 4, 16, 128, 1500, 5, "lognormal", 9, 2, (3,))
    _two_calls(kp, w, 3, tail_lens=np.array([0, 3, 10, 7, 1])).close()


def test_block_scaled_layer_two_calls(kp):
    # the block scales come in through the kscales argument (a block-scaled
    # layer's view holds 1 in *kscale)
    w = wl.custom("noalloc_kb", 1, 2, 8, 64, 700, 3, "lognormal", 5, 1, (2,))
    _two_calls(kp, w, 2, k_block=32, tail_lens=np.array([5, 0, 2])).close()


def test_splits_cut_down_to_fit_the_array(kp):
    # 8 KV heads x 1024 rows x (128 + 2) floats: one split's partials take
    # 4.26 MB, so only one split fits the 8 MiB array (the call would take
    # 22 otherwise)
    w = wl.custom("noalloc_fit", 1, 8, 32, 128, 700, 256, "lognormal", 0, 1, (4,))
    per_split = w.kv_heads * w.rows * (w.head_dim + 2) * 4 + 512
    assert SCRATCH_BYTES // per_split == 1
    _two_calls(kp, w, 4, max_rows=w.rows).close()


def test_refusals(kp):
    import torch

    w = wl.custom("noalloc_ref", 1, 8, 32, 128, 256, 2, "lognormal", 0, 1, (3,))
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [3])
    K, V = wl.layer_kv(w, 0)
    pool.compress(0, to_dev(K), to_dev(V))
    view = pool.layer_view(0)
    out = torch.empty((4096, w.head_dim), dtype=torch.float32, device="cuda")
    Q = torch.zeros((4096, w.head_dim), dtype=torch.bfloat16, device="cuda")
    # 512 agents x 4 query heads per KV head = 2048 rows (within the row
    # limit), but one split's partials, 8 x 2048 x 130 x 4 B, exceed the array
    big = wl.custom("noalloc_big", 1, 8, 32, 128, 256, 512, "lognormal", 0, 1, (3,))
    assert big.rows <= 4096
    assert big.kv_heads * big.rows * (big.head_dim + 2) * 4 > SCRATCH_BYTES
    assert _noalloc(kp, view, big, 3, Q, out) == INVALID_ARG
    # more than 4096 rows per KV head
    many = wl.custom("noalloc_many", 1, 1, 2, 128, 256, 2049, "lognormal", 0, 1, (3,))
    assert many.rows > 4096
    assert _noalloc(kp, view, many, 3, Q, out) == INVALID_ARG
    assert pool.status() == 0
    pool.close()
