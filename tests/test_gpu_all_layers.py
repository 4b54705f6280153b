"""Every layer of the SmolLM2-, Llama-3-8B- and Llama-3-8B-long-shaped
workloads, encoded and decompressed by the library in the benchmark's launch
configuration (all layers in one compress call and one decompress call) and
compared with the CPU oracle bit for bit: int8 K, K scale, V norms, packed V
codes, decompressed bf16 K and V. Attention of every layer (every decode step
of the long workload, with its bf16 tails) within 2e-3 of the oracle's
float64 attention over the same dequantised layer.

The oracle runs in a pool of spawned worker processes (one layer per task);
the comparison of stored bytes goes through SHA-256 digests of the arrays, and
a mismatch is re-derived in this process to name the first differing
element."""

import hashlib
import multiprocessing as mp
import os

import numpy as np
import pytest

from oracle import attention, codec
from shared_quantized_kv_gb300 import workloads as wl

import oracle_layers
from parity_util import TOL, check_encode, from_dev_bf16, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kp():
    import torch

    from shared_quantized_kv_gb300 import build, kvpool

    assert torch.cuda.is_available()
    build.build()
    return kvpool


def _dig(t) -> str:
    a = t.cpu().numpy() if hasattr(t, "cpu") else np.asarray(t)
    return hashlib.sha256(np.ascontiguousarray(a).view(np.uint8).reshape(-1).tobytes()).hexdigest()


def _oracle_results(name, layers):
    """Ordered oracle results of `layers`, computed by spawned workers."""
    n = max(1, min(8, (os.cpu_count() or 2) - 1, len(layers)))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")  # workers inherit these
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(n) as pool:
            for r in pool.imap(oracle_layers.job, [(name, l) for l in layers]):
                yield r
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("name", ["smollm2_2k", "llama3_8b_4k", "llama3_8b_long"])
def test_every_layer_bit_exact(kp, name):
    import torch

    w = wl.WORKLOADS[name]
    L = w.layers
    pool = kp.KVPool(L, w.kv_heads, w.head_dim, w.ctx, w.bits_list(), max_rows=w.rows)
    refs, Ks, Vs = {}, [], []
    for r in _oracle_results(name, list(range(L))):
        Ks.append(to_dev(r.pop("K")))
        Vs.append(to_dev(r.pop("V")))
        refs[r["layer"]] = r
    pool.compress_layers(list(range(L)), Ks, Vs)
    Ko, Vo = pool.decompress_layers(list(range(L)))
    assert pool.status() == 0
    worst = 0.0
    for l in range(L):
        r = refs[l]
        kq, vc, vn, ks = pool.export_layer(l)
        got = {"kscale": _dig(ks), "kq": _dig(kq), "vnorm": _dig(vn), "vcodes": _dig(vc)}
        bad = [f for f in got if got[f] != r["enc"][f]]
        if bad:  # name the first differing element
            K, V = wl.layer_kv(w, l)
            check_encode(pool, l, codec.encode_layer(K, V, w.layer_bits(l)))
            raise AssertionError(f"layer {l}: {bad} differ")
        assert _dig(from_dev_bf16(Ko[l])) == r["Kd"], f"layer {l}: decompressed K differs"
        assert _dig(from_dev_bf16(Vo[l])) == r["Vd"], f"layer {l}: decompressed V differs"
        tail = None
        if w.tail_max:
            tail_k, tail_v = to_dev(r["Kt"]), to_dev(r["Vt"])
        for step, (Q, ref) in enumerate(r["attn"]):
            if w.tail_max:
                lens = torch.full((w.agents,), w.tail_len(step), dtype=torch.int32, device="cuda")
                tail = (tail_k, tail_v, lens)
            out = pool.attend(l, to_dev(Q), tail=tail)
            err = attention.row_rel_error(out.cpu().numpy(), ref)
            worst = max(worst, err)
            assert err <= TOL, f"layer {l} step {step}: attention error {err:.3e}"
        Ko[l] = Vo[l] = None
    assert pool.status() == 0
    print(f"{name}: {L} layers bit-exact, worst attention row error {worst:.2e}")
    pool.close()
