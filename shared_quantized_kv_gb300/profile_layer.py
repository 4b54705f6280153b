"""Run the three calls of the hot path on one layer of a named workload, a few
times, for profilers (ncu captures one kernel of one repetition).

    python -m shared_quantized_kv_gb300.profile_layer --workload llama3_8b_4k --reps 4

Every repetition re-arms the layer (kvpool_reset_layer), compresses it,
attends all agents and decompresses it; the script exits non-zero if the
device status word reports an error. Inputs are the seeded synthetic layer of
the workload (layer 0 unless --layer is given).
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
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    bits = w.layer_bits(args.layer)
    pool = kp.KVPool(1, w.kv_heads, w.head_dim, w.ctx, [bits])
    K, V = wl.layer_kv_torch(w, args.layer, "cuda")
    Q = torch.from_numpy(wl.layer_q(w, args.layer).view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((w.agents, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    Kd, Vd = torch.empty_like(K), torch.empty_like(V)
    for _ in range(args.reps):
        pool.reset_layer(0)
        pool.compress(0, K, V)
        pool.attend(0, Q, out)
        pool.decompress(0, Kd, Vd)
    torch.cuda.synchronize()
    st = pool.status()
    print(f"{args.workload} layer {args.layer} ({bits}-bit): {args.reps} repetitions, status {st}")
    pool.close()
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
