"""Oracle work for one layer of a named workload, run in worker processes of
the all-layers GPU parity test: draw the layer's seeded inputs, encode and
decompress them with the oracle, and compute the oracle's float64 attention
for every decode step. Returns the inputs (for upload), SHA-256 digests of
every stored and decompressed array (compared bit for bit with the library's)
and the attention references."""

from __future__ import annotations

import hashlib

import numpy as np

from oracle import attention, codec
from shared_quantized_kv_gb300 import workloads as wl


def digest(a) -> str:
    a = np.ascontiguousarray(a)
    return hashlib.sha256(a.view(np.uint8).reshape(-1).tobytes()).hexdigest()


def encode_digests(enc: dict) -> dict:
    """Digests of the stored bytes in the library's export layout."""
    return {"kscale": digest(np.float32(enc["scale"]).reshape(1)), "kq": digest(enc["kq"]),
            "vnorm": digest(enc["norms"]), "vcodes": digest(enc["packed"])}


def layer_reference(name: str, layer: int) -> dict:
    w = wl.WORKLOADS[name]
    K, V = wl.layer_kv(w, layer)
    enc = codec.encode_layer(K, V, w.layer_bits(layer))
    kb, vb = codec.decompress_layer(enc)
    Kh, Vh = attention.dequantise_f64(enc)
    refs = []
    Kt = Vt = None
    if w.tail_max:
        Kt, Vt = wl.layer_tail(w, layer)
    for step in range(w.decode_steps):
        Q = wl.layer_q(w, layer, step)
        tail = None
        if w.tail_max:
            tail = (Kt, Vt, np.full(w.agents, w.tail_len(step)))
        refs.append((Q, attention.attend_f64(Kh, Vh, Q, tail)))
    return {"layer": layer, "K": K, "V": V, "Kt": Kt, "Vt": Vt, "enc": encode_digests(enc),
            "Kd": digest(kb), "Vd": digest(vb), "attn": refs}


def job(arg):
    """Pool task: layer_reference(name, layer) of the pair `arg`."""
    return layer_reference(*arg)
