"""The C-ABI library on a machine without a GPU: it loads, exports every
function include/kvpool.h declares, derives the same float32 Lloyd-Max table as
the oracle, and rejects bad arguments before touching a device."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import lloyd_max

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kp():
    from shared_quantized_kv_gb300 import build, kvpool

    build.build()
    kvpool.lib()
    return kvpool


def _declared():
    with open(os.path.join(ROOT, "include", "kvpool.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"\b(kvpool_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(kp):
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(kp.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(kp._SIGS)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_library_codebook_equals_oracle(kp, bits):
    c, m = kp.codebook(bits)
    oc, om = lloyd_max.tables_f32(bits)
    assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(m.view(np.uint32), om.view(np.uint32))


def test_strerror_and_bad_codebook(kp):
    lib = kp.lib()
    for code in range(-7, 1):
        assert lib.kvpool_strerror(code)
    assert lib.kvpool_codebook(5, None, None) == -1


def test_create_rejects_bad_arguments_without_a_device(kp):
    lib = kp.lib()
    h = ctypes.c_void_p()
    for args in [(1, 2, 96, 256, None, 0), (0, 2, 64, 256, None, 0), (1, 0, 64, 256, None, 0),
                 (1, 2, 64, 0, None, 0), (1, 2, 64, 256, None, 5000)]:
        assert lib.kvpool_create(ctypes.byref(h), *args) == -1
    bad_bits = (ctypes.c_uint8 * 2)(3, 5)
    assert lib.kvpool_create(ctypes.byref(h), 2, 2, 64, 256, ctypes.cast(bad_bits, ctypes.c_void_p), 0) == -1
    assert lib.kvpool_create(None, 1, 2, 64, 256, None, 0) == -1
    for kb in (1, 16, 64, -32):  # only 0 and 32 are K block sizes
        assert lib.kvpool_create_ex(ctypes.byref(h), 1, 2, 64, 256, None, 0, kb) == -1
    assert lib.kvpool_export_kscales(None, 0, None, None) == -1


def test_null_pool_calls(kp):
    lib = kp.lib()
    assert lib.kvpool_pool_bytes(None) == 0
    assert lib.kvpool_compress(None, 0, None, None, None) == -1
    assert lib.kvpool_attend(None, 0, None, 1, 1, None, None, 0.0, None) == -1
    assert lib.kvpool_decompress(None, 0, None, None, None) == -1
    lay = (ctypes.c_int * 2)(0, 1)
    ptrs = (ctypes.c_void_p * 2)(16, 32)
    assert lib.kvpool_compress_layers(None, 2, lay, ptrs, ptrs, None) == -1
    assert lib.kvpool_decompress_layers(None, 2, lay, ptrs, ptrs, None) == -1
    assert lib.kvpool_append(None, 0, None, None, 1, None) == -1
    assert lib.kvpool_append_bits(None, 0, None, None, 1, 3, None) == -1
    assert lib.kvpool_layer_widths(None, 0, None, 0) == -1
    assert lib.kvpool_import_layer_blocks(None, 0, None, None, None, None, None, 1, None) == -1
    assert lib.kvpool_attend_ws(None, 0, None, 1, 1, None, None, 0.0, None, 0, None) == -1
    assert lib.kvpool_attend_ws_bytes(None, 1, 1) == 0
    assert lib.kvpool_layer_len(None, 0) == -1
    lib.kvpool_destroy(None)
