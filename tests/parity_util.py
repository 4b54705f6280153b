"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the library through its C-ABI binding, run the oracle on the same bytes,
and compare."""

import numpy as np

from oracle import attention, codec

TOL = 2e-3  # attention: max over rows of max|o - r| / max|r|


def to_dev(a, dtype="bf16"):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return t.view(torch.bfloat16)


def from_dev_bf16(t):
    import torch

    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check_encode(pool, layer, enc):
    """Stored bytes of `layer` equal the oracle's encode bit for bit."""
    got = pool.read_layer(layer)
    assert got["kscale"].view(np.uint32) == np.float32(enc["scale"]).view(np.uint32), \
        (got["kscale"], enc["scale"])
    assert np.array_equal(got["kq"], enc["kq"]), _first_diff(got["kq"], enc["kq"])
    assert np.array_equal(got["vnorm"].view(np.uint32), enc["norms"].view(np.uint32)), \
        _first_diff(got["vnorm"], enc["norms"])
    H = enc["kq"].shape[0]
    gv, ev = got["vcodes"].reshape(H, -1), enc["packed"].reshape(H, -1)  # both layouts: per head, bytes in order
    assert np.array_equal(gv, ev), _first_diff(gv, ev)
    if enc.get("k_block"):
        assert np.array_equal(got["kscales"].view(np.uint32), enc["kscales"].view(np.uint32)), \
            _first_diff(got["kscales"], enc["kscales"])


def check_decompress(pool, layer, enc):
    Kd, Vd = pool.decompress(layer)
    kb, vb = codec.decompress_layer(enc)
    gk, gv = from_dev_bf16(Kd), from_dev_bf16(Vd)
    assert np.array_equal(gk, kb), _first_diff(gk, kb)
    assert np.array_equal(gv, vb), _first_diff(gv, vb)


def attention_error(out, enc, Q, tail=None, scale=None, rows=None):
    Kh, Vh = attention.dequantise_f64(enc)
    o = out.cpu().numpy().astype(np.float64)
    if rows is None:
        ref = attention.attend_f64(Kh, Vh, Q, tail, scale)
        return attention.row_rel_error(o, ref)
    ref = attention.attend_rows_f64(Kh, Vh, Q, rows, tail, scale)
    got = np.stack([o[a, h] for a, h in rows])
    return attention.row_rel_error(got, ref)


def _first_diff(a, b):
    a, b = np.asarray(a), np.asarray(b)
    if a.shape != b.shape:
        return f"shape {a.shape} vs {b.shape}"
    idx = np.argwhere(a != b)
    if len(idx) == 0:
        return "equal"
    i = tuple(idx[0])
    return f"{len(idx)} differ; first at {i}: {a[i]!r} vs {b[i]!r}"
