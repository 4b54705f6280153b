"""Shared, asymmetrically quantized KV-cache pool for multi-agent decode on
GB300 (sm_103a).

The compute path is the C-ABI library ``libkvpool.so`` (hand-written CUDA
kernels); :mod:`shared_quantized_kv_gb300.kvpool` is a thin ctypes binding of
it. :mod:`shared_quantized_kv_gb300.workloads` holds the seeded synthetic
inputs. The binding is imported on first use so the input generators stay
usable on machines without the library.
"""


def __getattr__(name):
    if name in ("kvpool",):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
