"""Run the three calls of the hot path on one layer of a named workload, a few
times, for profilers (ncu captures one kernel of one repetition).

    python -m shared_quantized_kv_gb300.profile_layer --workload llama3_8b_4k --reps 4
    python -m shared_quantized_kv_gb300.profile_layer --workload llama3_8b_4k --layers 8
    python -m shared_quantized_kv_gb300.profile_layer --workload llama3_8b_4k --k-block 32

Every repetition re-arms the layer (kvpool_reset_layer), compresses it,
attends all agents and decompresses it; the script exits non-zero if the
device status word reports an error. Inputs are the seeded synthetic layer of
the workload (layer 0 unless --layer is given). With --layers N (N > 1) the
first N layers of the workload go through the multi-layer calls: one
compress and one decompress call for all N, attend per layer. --k-block 32
builds the pool with block-scaled K. --ws attends through a workspace
(kvpool_attend_ws: one-CTA context slices, then the merge kernel).
"""

import argparse
import sys

import numpy as np
import torch

from . import kvpool as kp
from . import workloads as wl


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3_8b_4k")
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--layers", type=int, default=1)
    ap.add_argument("--k-block", type=int, default=0, choices=[0, 32])
    ap.add_argument("--ws", action="store_true", help="attend through kvpool_attend_ws")
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    if args.layers > 1:
        return multi(w, args)
    bits = w.layer_bits(args.layer)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [bits], max_rows=max(w.rows, 1), k_block=args.k_block)
    ws = torch.empty(max(pool.attend_ws_bytes(w.agents, w.q_heads), 16), dtype=torch.uint8, device="cuda")
    K, V = wl.layer_kv_torch(w, args.layer, "cuda")
    Q = torch.from_numpy(wl.layer_q(w, args.layer).view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((w.agents, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    Kd, Vd = torch.empty_like(K), torch.empty_like(V)
    for _ in range(args.reps):
        pool.reset_layer(0)
        pool.compress(0, K, V)
        if args.ws:
            pool.attend_ws(0, Q, ws, out)
        else:
            pool.attend(0, Q, out)
        pool.decompress(0, Kd, Vd)
    torch.cuda.synchronize()
    st = pool.status()
    print(f"{args.workload} layer {args.layer} ({bits}-bit): {args.reps} repetitions, status {st}")
    pool.close()
    return 0 if st == 0 else 1


def multi(w, args) -> int:
    n = min(args.layers, w.layers)
    bits = [w.layer_bits(l) for l in range(n)]
    pool = kp.KVPool(n, w.kv_heads, w.head_dim, w.ctx, bits, max_rows=max(w.rows, 1), k_block=args.k_block)
    ws = torch.empty(max(pool.attend_ws_bytes(w.agents, w.q_heads), 16), dtype=torch.uint8, device="cuda")
    KV = [wl.layer_kv_torch(w, l, "cuda") for l in range(n)]
    Ks, Vs = [k for k, _ in KV], [v for _, v in KV]
    Q = [torch.from_numpy(wl.layer_q(w, l).view(np.int16)).cuda().view(torch.bfloat16) for l in range(n)]
    out = torch.empty((w.agents, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    Kd = [torch.empty_like(k) for k in Ks]
    Vd = [torch.empty_like(v) for v in Vs]
    layers = list(range(n))
    for _ in range(args.reps):
        for l in layers:
            pool.reset_layer(l)
        pool.compress_layers(layers, Ks, Vs)
        for l in layers:
            if args.ws:
                pool.attend_ws(l, Q[l], ws, out)
            else:
                pool.attend(l, Q[l], out)
        pool.decompress_layers(layers, Kd, Vd)
    torch.cuda.synchronize()
    st = pool.status()
    print(f"{args.workload} layers 0..{n - 1} (multi-layer calls): {args.reps} repetitions, status {st}")
    pool.close()
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
