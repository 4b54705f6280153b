"""Error against bytes of the two K scalings of the pool (test
infrastructure: CPU only, oracle functions on the seeded synthetic
workloads; no part of the library).

    python -m oracle.compare_k_modes --workload llama3_8b_4k --layers 0 17 31

Per layer: the relative RMS error of the dequantised K, and the attention
error (max over rows of max|o - r| / max|r|) of float64 attention over the
dequantised K with the exact V, against float64 attention over the exact bf16
K and V; both for one scale per layer's K tensor (1 byte per element) and for
one float32 scale per 32 elements (1.125 bytes per element). PolyKV summary,
section 2.B names a per-tensor scale and q8_0; this measures what separates
the two readings on these inputs.
"""

import argparse
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import attention, codec  # noqa: E402
from shared_quantized_kv_gb300 import workloads as wl  # noqa: E402


def compare(w, layer):
    K, V = wl.layer_kv(w, layer)
    Q = wl.layer_q(w, layer)
    k = codec.bf16_to_f32(K).astype(np.float64)
    v = codec.bf16_to_f32(V).astype(np.float64)
    ref = attention.attend_f64(k, v, Q)
    res = {}
    for name, kb in (("per-tensor", 0), ("block-32", 32)):
        enc = codec.encode_layer(K, V, w.layer_bits(layer), k_block=kb)
        kh, _ = attention.dequantise_f64(enc)
        rms = float(np.sqrt(np.mean((kh - k) ** 2) / np.mean(k ** 2)))
        err = attention.row_rel_error(attention.attend_f64(kh, v, Q), ref)
        res[name] = (rms, err, 1.0 + (4.0 / kb if kb else 0.0))
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3_8b_4k")
    ap.add_argument("--layers", type=int, nargs="+", default=[0])
    a = ap.parse_args()
    w = wl.WORKLOADS[a.workload]
    print(f"{a.workload}: K relative RMS error / attention error (exact V) / bytes per K element")
    for layer in a.layers:
        r = compare(w, layer)
        line = "  ".join(f"{n}: {rms:.3e} / {err:.3e} / {b:.3f} B" for n, (rms, err, b) in r.items())
        print(f"  layer {layer:2d}  {line}")


if __name__ == "__main__":
    main()
