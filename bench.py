"""Benchmark of the shared quantized KV pool hot path on GB300.

The headline is the decode step of the method: every agent's queries attend
over the resident compressed pool, layer after layer (one attention call per
layer: a layer's queries depend on the layer before). The step calls
kvpool_attend_ws (the context in one-CTA slices over every SM, partial states
in a workspace allocated once before timing, one merge kernel); the
cluster-merged kvpool_attend is timed beside it as the phase "attend". Workload: the
Llama-3-8B-shaped pool (32 layers, 8 KV heads, 32 query heads, head_dim 128,
4096 shared-context tokens, 15 agents x 1 decode query, int8 K, 3-bit V).

value = agents x ranks / (max over ranks of the time of one decode step, all
layers of kvpool_attend_ws): agent-decode steps per second. Each attention
phase is captured as one CUDA graph and replayed; CUDA events around each replay give
its device time, and L2 is flushed (a 512 MiB write) before every replay,
outside the events. The write-once encode (kvpool_compress_layers, all layers
in one call) and the per-agent materialisation baseline (kvpool_decompress_
layers) are timed the same way and reported under "phases".

e2e: the decode step through the C-ABI with the pool resident and every
step's queries (and new tail tokens) copied up from pinned host memory and
its attention outputs copied back, inside the timed region. e2e_full_path:
compress + attend + decompress with the bf16 K, V uploaded and the outputs
and decompressed K, V downloaded every step.

With N ranks (torchrun) the ranks share one pool: rank r holds KV heads
[r*Hk/N, (r+1)*Hk/N) of every layer and serves the query heads that read
them, so attention needs no exchange and the total work is fixed ("strong"
scaling); value is still every agent's step over the whole pool.

cpu_baseline: the CPU oracle's decode step (dequantise the pool in float64,
float64 attention for every agent, every layer) on all host cores (one
process per core, layers spread over them) and on one core, median of 3.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on the host
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "agent-decode steps/s over shared int8-K/3-bit-V pool; % of HBM roofline"
UNIT = "agent-steps/s"
FALLBACK_HBM = 6800.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM, "fallback"


def workload_config(w, ws, k_block):
    """The workload part of both arms' `config` (identical for the GPU arm and
    the reference arm)."""
    return {"workload": w.name, "k_scales": "per 32 elements" if k_block else "per layer",
            "layers": w.layers, "kv_heads": w.kv_heads, "q_heads": w.q_heads, "head_dim": w.head_dim,
            "ctx": w.ctx, "agents": w.agents, "v_bits": sorted(set(w.bits_list())), "tail": w.tail_max,
            "step": "decode: kvpool_attend_ws of every layer for every agent (workspace allocated once)",
            "parallelism": "one GPU" if ws == 1 else
                           f"one pool, its KV heads split over {ws} ranks (no data-path collective)"}


def launches_per_step(w, k_block, per_layer_calls, batch=32):
    """The library's kernel launches in one step, by phase. Compress: a max|K|
    kernel and an encode kernel per layer, or, for all layers in one call, one
    max|K| kernel and one encode kernel per V width per 32 layers. Attend: the
    tensor-core kernel per layer (per-tensor and block-scaled K alike);
    attend_ws: that kernel in workspace mode and the merge kernel per layer.
    Decompress: one kernel per layer, or one per V width per 32 layers."""
    bits = w.bits_list()
    chunks = [bits[i:i + batch] for i in range(0, len(bits), batch)]
    widths = sum(len(set(c)) for c in chunks)
    if per_layer_calls:
        comp, dec = 2 * len(bits), len(bits)
    else:
        comp, dec = len(chunks) + widths, widths
    return {"compress": comp, "attend": len(bits), "attend_ws": 2 * len(bits), "decompress": dec}


def max_over_ranks(step_ms, ph_ms, phases, device=None):
    """(step time, per-phase times) as the maximum over the ranks of the
    default process group (unchanged when no group is initialised). Ranks hold
    shares of one pool (its KV heads): a step takes as long as its slowest
    rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return step_ms, dict(ph_ms)
    t = torch.tensor([step_ms] + [ph_ms[p] for p in phases], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), {p: float(t[i + 1]) for i, p in enumerate(phases)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms (the
    caller keeps the GPU busy with the timed work while it runs)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "shared_quantized_kv_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_file):
    """ncu DRAM bytes per launch recorded for `kernel_file`, if the source has
    not changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    r = rec.get(kernel_file)
    if r and r.get("source_sha") == _source_sha([kernel_file]):
        return r.get("bytes_per_launch")
    return None


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import numpy as np
    import torch

    from shared_quantized_kv_gb300 import build, kvpool
    from shared_quantized_kv_gb300 import workloads as wl

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        build.build()
    if ws > 1:
        dist.barrier()
    kvpool.lib()

    w = wl.WORKLOADS[args.workload]
    L, A = w.layers, w.agents
    # N ranks share one pool: rank r holds KV heads [h0, h1) of every layer
    # and serves the query heads that read them (no exchange in attention)
    if w.kv_heads % ws:
        raise SystemExit(f"{w.kv_heads} KV heads do not split over {ws} ranks")
    hk = w.kv_heads // ws
    h0, h1 = rank * hk, (rank + 1) * hk
    G = w.group
    pool = kvpool.KVPool(L, hk, w.head_dim, w.ctx, w.bits_list(), max_rows=max(w.rows, 1),
                         k_block=args.k_block)
    K, V = [], []
    for l in range(L):
        k, v = wl.layer_kv_torch(w, l, dev)
        K.append(k[h0:h1].contiguous())
        V.append(v[h0:h1].contiguous())
        del k, v
    Q = [torch.from_numpy(wl.layer_q(w, l, 0).view(np.int16)).to(dev).view(torch.bfloat16)[:, h0 * G:h1 * G]
         .contiguous() for l in range(L)]
    tail = None
    if w.tail_max:
        tail = []
        for l in range(L):
            kt, vt = wl.layer_tail(w, l)
            lens = torch.full((A,), w.tail_len(w.decode_steps - 1), dtype=torch.int32, device=dev)
            tail.append((torch.from_numpy(kt.view(np.int16)).to(dev).view(torch.bfloat16)[:, h0:h1].contiguous(),
                         torch.from_numpy(vt.view(np.int16)).to(dev).view(torch.bfloat16)[:, h0:h1].contiguous(),
                         lens))
    out = [torch.empty((A, hk * G, w.head_dim), dtype=torch.float32, device=dev) for _ in range(L)]
    Kd = [torch.empty_like(K[0]) for _ in range(L)]
    Vd = [torch.empty_like(V[0]) for _ in range(L)]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    layers = list(range(L))

    def compress():
        for l in layers:
            pool.reset_layer(l)
        if args.per_layer_calls:
            for l in layers:
                pool.compress(l, K[l], V[l])
        else:  # the whole shared context in one call
            pool.compress_layers(layers, K, V)

    # the decode step's workspace, allocated once (like the pool)
    wsbuf = torch.empty(max(pool.attend_ws_bytes(A, hk * G), 16), dtype=torch.uint8, device=dev)

    def attend_ws():  # the decode step: layer l + 1's queries come from layer l's output
        for l in layers:
            pool.attend_ws(l, Q[l], wsbuf, out[l], tail[l] if tail else None)

    def attend():  # the same step through the cluster-merged kvpool_attend
        for l in layers:
            pool.attend(l, Q[l], out[l], tail[l] if tail else None)

    def decompress():
        if args.per_layer_calls:
            for l in layers:
                pool.decompress(l, Kd[l], Vd[l])
        else:
            pool.decompress_layers(layers, Kd, Vd)

    # eager once (state + correctness of the calls), then capture each phase
    compress(); attend(); attend_ws(); decompress()
    assert pool.status() == 0
    graphs = {}
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    for name, fn in (("compress", compress), ("attend_ws", attend_ws), ("attend", attend),
                     ("decompress", decompress)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        graphs[name] = g
    torch.cuda.synchronize()

    phases = ("attend_ws", "attend", "compress", "decompress")

    def one_step(record):
        ev = []
        for ph in phases:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            graphs[ph].replay()
            e1.record()
            ev.append((ph, e0, e1))
        record.append(ev)

    for _ in range(args.warmup):
        one_step([])
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    # clocks: sampled every 200 ms while the same step runs untimed for about
    # 0.6 s and then through the K timed steps (a timed region of a few ms
    # alone would catch no sample under load)
    sampler = ClockSampler(local)
    sampler.start()
    t_load = time.perf_counter()
    while time.perf_counter() - t_load < 0.6:
        one_step([])
        torch.cuda.synchronize()
    rec = []
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        one_step(rec)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = dict(sampler.stop(), window="0.6 s of the same phases untimed, then the timed steps")
    assert pool.status() == 0

    ph_ms = {ph: 0.0 for ph in phases}
    for ev in rec:
        for ph, e0, e1 in ev:
            ph_ms[ph] += e0.elapsed_time(e1)
    ph_ms = {ph: v / args.steps for ph, v in ph_ms.items()}
    _, ph_ms = max_over_ranks(0.0, ph_ms, phases, dev if ws > 1 else None)
    step_ms = ph_ms["attend_ws"]  # the decode step: all layers of kvpool_attend_ws

    launches = launches_per_step(w, args.k_block, args.per_layer_calls)
    # algorithmic bytes per layer (this rank's share of the heads)
    nvec = hk * w.ctx
    kv_in = 2 * nvec * w.head_dim * 2
    pool_layer = pool.pool_bytes() / L
    tail_bytes = 2 * A * hk * w.tail_len(w.decode_steps - 1) * w.head_dim * 2 if tail else 0
    algo = {"compress": kv_in + pool_layer, "attend": pool_layer + tail_bytes,
            "attend_ws": pool_layer + tail_bytes, "decompress": pool_layer + kv_in}
    peak, peak_kind = _peaks()
    ph_info = {}
    for ph in phases:
        per_call_s = ph_ms[ph] / 1e3 / L
        gbs = algo[ph] / per_call_s / 1e9
        ph_info[ph] = {"ms_per_step": round(ph_ms[ph], 4), "us_per_layer": round(per_call_s * 1e6, 3),
                       "algo_bytes_per_layer": int(algo[ph]), "GB_per_s": round(gbs, 1),
                       "hbm_frac": round(gbs / peak, 4), "launches_per_step": launches[ph]}
    ph_info["attend"]["agent_steps_per_s"] = round(A / (ph_ms["attend"] / 1e3), 1)
    ph_info["attend_ws"]["agent_steps_per_s"] = round(A / (ph_ms["attend_ws"] / 1e3), 1)
    ph_info["attend"]["note"] = "kvpool_attend: clusters merge the context splits in distributed shared memory"
    ph_info["attend_ws"]["note"] = ("kvpool_attend_ws (the decode step): one-CTA context slices, partial states "
                                    "in the workspace, a merge kernel per layer")
    ph_info["compress"]["note"] = "write-once encode of the shared context (once per pool, not per step)"
    ph_info["decompress"]["note"] = "per-agent materialisation baseline of the pages (not on the decode path)"
    att_file = "attend_rows.cuh"

    e2e = e2e_full = None
    if not args.no_e2e:
        e2e = run_e2e_decode(args, pool, w, Q, tail, out, wsbuf)
        e2e_full = run_e2e_full(args, pool, w, K, V, Q, tail, out, Kd, Vd, wsbuf)

    value = A / (step_ms / 1e3)  # every agent's step over the whole (split) pool
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "int8/u3+f32",
        "data": "synthetic (seeded; bf16 K/V with LogNormal(0,0.5) channel std and 1% x10 outlier "
                "channels, Q ~ N(0,1))",
        "config": dict(workload_config(w, ws, args.k_block),
                       calls="attend_ws (the step) and attend: one call per layer; compress and decompress: "
                             "all layers per call" + (" (one call per layer)" if args.per_layer_calls else ""),
                       l2="flushed (512 MiB write) before every timed graph replay, outside the events"),
        "phases": ph_info,
        "roofline": {"bound": "hbm", "kernel": "attend_ws", "achieved": ph_info["attend_ws"]["GB_per_s"],
                     "peak": peak, "unit": "GB/s", "frac": ph_info["attend_ws"]["hbm_frac"],
                     "traffic": _traffic(att_file), "peak_source": peak_kind,
                     "algo_bytes_per_launch": int(algo["attend_ws"]),
                     "how": "algorithmic bytes per layer (pool layer + tails) / (attend_ws graph time / layers: "
                            "the attention kernel and its merge kernel)"},
        "gpu_launches": args.steps * launches["attend_ws"],
        "gpu_launches_all_phases": args.steps * sum(launches.values()),
        "clocks": clocks,
        "wall_s_timed": round(t_wall, 3),
        "e2e": e2e,
        "e2e_full_path": e2e_full,
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, k_block=args.k_block)
    if rank == 0:
        print(json.dumps(line), flush=True)
    pool.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def e2e_download_sizes(L: int) -> list:
    """Layers per download chunk of the end-to-end decode step: eight at a
    time, then halving, so that little is left to copy after the last layer
    (32 layers: 8, 8, 8, 4, 2, 1, 1)."""
    sizes, left = [], L
    while left > 0:
        n = 8 if left > 16 else max(1, left // 2)
        sizes.append(n)
        left -= n
    return sizes


def e2e_upload_pieces(L: int) -> list:
    """Layer ranges [a, b) uploaded as one copy each: layer 0, layers 1-3,
    the rest; each is waited for before its first layer attends."""
    return [p for p in ((0, 1), (1, min(4, L)), (min(4, L), L)) if p[0] < p[1]]


def run_e2e_decode(args, pool, w, Q, tail, out, wsbuf):
    """The decode step end to end: the pool stays resident; every step the
    queries of all layers (and, with tails, each agent's new tail token of
    every layer) are copied up from pinned host memory on an input stream in
    three pieces (layer 0, layers 1-3, the rest), so that layer 0 starts once
    its own inputs are up. With tails, one copy kernel per piece writes the
    new tokens of its layers into the agents' tails (the tails of all layers
    live in one buffer). The layers attend in order, and the attention outputs
    come back on a second stream in chunks that shrink towards the last layer
    (8, 8, 8, 4, 2, 1, 1 layers for 32), overlapping the later layers. One
    step is captured as a CUDA graph and replayed."""
    import torch

    L, A = w.layers, w.agents
    dev = Q[0].device
    q_bytes = Q[0].numel() * Q[0].element_size()
    nt_bytes = 0
    if tail:
        # every layer's tails in one buffer [L][2][A][Hk][T_max][d], so that one
        # copy kernel appends the step's tokens of several layers
        tshape = tuple(tail[0][0].shape)  # [A, Hk, T_max, d]
        tail_all = torch.empty((L, 2) + tshape, dtype=torch.bfloat16, device=dev)
        for l in range(L):
            tail_all[l, 0].copy_(tail[l][0])
            tail_all[l, 1].copy_(tail[l][1])
        t_e2e = [(tail_all[l, 0], tail_all[l, 1], tail[l][2]) for l in range(L)]
        pos = w.tail_len(w.decode_steps - 1) - 1  # the step's token
        nt_shape = (L, 2, tshape[0], tshape[1], tshape[3])  # one new token per agent and KV head
        nt_bytes = 2 * tshape[0] * tshape[1] * tshape[3] * 2
    d_in = torch.empty(L * (q_bytes + nt_bytes), dtype=torch.uint8, device=dev)
    h_in = torch.empty(L * (q_bytes + nt_bytes), dtype=torch.uint8).pin_memory()
    q_dev = [d_in[l * q_bytes:(l + 1) * q_bytes].view(torch.bfloat16).view(Q[l].shape) for l in range(L)]
    for l in range(L):
        q_dev[l].copy_(Q[l])
    if tail:
        nt_all = d_in[L * q_bytes:].view(torch.bfloat16).view(nt_shape)
        for l in range(L):
            nt_all[l, 0].copy_(tail[l][0][:, :, pos])
            nt_all[l, 1].copy_(tail[l][1][:, :, pos])
    h_in.copy_(d_in.cpu())
    o_bytes = out[0].numel() * out[0].element_size()
    d_out = torch.empty(L * o_bytes, dtype=torch.uint8, device=dev)
    o_dev = [d_out[l * o_bytes:(l + 1) * o_bytes].view(torch.float32).view(out[l].shape) for l in range(L)]
    h_out = torch.empty(L * o_bytes, dtype=torch.uint8).pin_memory()
    sizes = e2e_download_sizes(L)
    chunks, c0 = [], 0
    for n in sizes:
        chunks.append(list(range(c0, c0 + n)))
        c0 += n
    pieces = e2e_upload_pieces(L)
    s_main, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_done = [torch.cuda.Event() for _ in chunks]
    ev_in = [torch.cuda.Event() for _ in pieces]
    piece_of = {p[0]: i for i, p in enumerate(pieces)}

    def step():
        s_in.wait_stream(s_main)
        s_out.wait_stream(s_main)
        with torch.cuda.stream(s_in):
            for i, (a, b) in enumerate(pieces):
                d_in[a * q_bytes:b * q_bytes].copy_(h_in[a * q_bytes:b * q_bytes], non_blocking=True)
                if tail:
                    o0 = L * q_bytes
                    d_in[o0 + a * nt_bytes:o0 + b * nt_bytes].copy_(h_in[o0 + a * nt_bytes:o0 + b * nt_bytes],
                                                                    non_blocking=True)
                ev_in[i].record(s_in)
        for c, ls in enumerate(chunks):
            for l in ls:
                if l in piece_of:
                    s_main.wait_event(ev_in[piece_of[l]])
                    if tail:  # the piece's new tokens into the tails
                        a, b = pieces[piece_of[l]]
                        tail_all[a:b, :, :, :, pos].copy_(nt_all[a:b])
                pool.attend_ws(l, q_dev[l], wsbuf, o_dev[l], t_e2e[l] if tail else None, stream=s_main)
            ev_done[c].record(s_main)
        with torch.cuda.stream(s_out):
            for c, ls in enumerate(chunks):
                s_out.wait_event(ev_done[c])
                a, b = ls[0] * o_bytes, (ls[-1] + 1) * o_bytes
                h_out[a:b].copy_(d_out[a:b], non_blocking=True)
        s_main.wait_stream(s_out)
        s_main.wait_stream(s_in)

    s_main.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_main):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_main):
        step()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # the downloaded outputs are the device's
    assert torch.equal(h_out.view(torch.float32)[:out[0].numel()].view(out[0].shape).to(dev), o_dev[0])
    return {"value": round(w.agents / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h_in.numel()), "d2h_bytes_per_step": int(h_out.numel()),
            "how": "decode step through the C-ABI, pool resident: every layer's queries"
                   + (" and new tail tokens (appended by one copy kernel per piece)" if tail else "")
                   + f" uploaded in {len(pieces)} pieces on an input stream (layer 0 first), attend layer by "
                   "layer, outputs "
                   f"downloaded on a second stream in chunks of {sizes} layers; one CUDA graph per step"}


def run_e2e_full(args, pool, w, K, V, Q, tail, out, Kd, Vd, wsbuf):
    """The same step with inputs copied from pinned host memory and the results
    (attention outputs and the decompressed K/V) copied back, inside the timed
    region. Layers are independent, so the step is pipelined over three
    streams: the inputs of layer l go up while layer l-1 computes and the
    results of layer l-2 come down. The inputs (K, V, Q) of each chunk of
    --e2e-chunk consecutive layers sit in one pinned host buffer and one
    device buffer, and so do its results, so a chunk moves with one copy
    each way. One step (copies included) is
    captured as a CUDA graph and replayed, as a serving loop would."""
    import torch

    L = w.layers
    dev = K[0].device

    def packed(parts):
        # one byte buffer per layer holding `parts` back to back (16-byte aligned
        # offsets), and a view of each part in it
        sizes = [t.numel() * t.element_size() for t in parts]
        buf = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
        views, off = [], 0
        for t, n in zip(parts, sizes):
            views.append(buf[off:off + n].view(t.dtype).view(t.shape))
            off += n
        return buf, views

    # copy chunks of `per` consecutive layers
    per = max(1, args.e2e_chunk)
    chunks = [list(range(c, min(L, c + per))) for c in range(0, L, per)]
    dIn, dOut, kv_in, kv_out = [], [], {}, {}
    for ls in chunks:
        b_in, vin = packed([t for l in ls for t in (K[l], V[l], Q[l])])
        b_out, vout = packed([t for l in ls for t in (out[l], Kd[l], Vd[l])])
        for i, l in enumerate(ls):
            k, v, q = vin[3 * i:3 * i + 3]
            k.copy_(K[l]); v.copy_(V[l]); q.copy_(Q[l])
            kv_in[l] = (k, v, q)
            kv_out[l] = tuple(vout[3 * i:3 * i + 3])
        dIn.append(b_in); dOut.append(b_out)
    hIn = [b.cpu().pin_memory() for b in dIn]
    hOut = [torch.empty(b.shape, dtype=b.dtype, pin_memory=True) for b in dOut]
    s_main, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_done = [torch.cuda.Event() for _ in chunks]

    def step():
        # runs on s_main (the capturing stream); s_in and s_out fork from it and join it
        s_in.wait_stream(s_main)
        s_out.wait_stream(s_main)
        with torch.cuda.stream(s_in):
            for c in range(len(chunks)):
                dIn[c].copy_(hIn[c], non_blocking=True)
                ev_in[c].record(s_in)
        for c, ls in enumerate(chunks):
            s_main.wait_event(ev_in[c])
            for l in ls:
                k, v, q = kv_in[l]
                o, kd, vd = kv_out[l]
                pool.reset_layer(l)
                pool.compress(l, k, v, stream=s_main)
                pool.attend_ws(l, q, wsbuf, o, tail[l] if tail else None, stream=s_main)
                pool.decompress(l, kd, vd, stream=s_main)
            ev_done[c].record(s_main)
        with torch.cuda.stream(s_out):
            for c in range(len(chunks)):
                s_out.wait_event(ev_done[c])
                hOut[c].copy_(dOut[c], non_blocking=True)
        s_main.wait_stream(s_in)
        s_main.wait_stream(s_out)

    s_main.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_main):
        step()  # warm-up outside the graph
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_main):
        step()
    for _ in range(max(1, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in hIn)
    d2h = sum(t.numel() * t.element_size() for t in hOut)
    return {"value": round(w.agents / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "how": "one CUDA graph per step: three streams pipelined over layers (upload, compute, download), "
                   f"one copy per {per} layer(s) each way"}


# ------------------------------------------------------------------ CPU legs

def _oracle_worker(name, layers, k_block, reps, barrier, results):
    """One oracle process: encode its layers (set-up, untimed: the pool is
    resident before decode starts), then for each of `reps` rounds wait at
    the barrier with the other workers and time one decode step over its
    layers: dequantise the stored codes in float64 and run float64 attention
    for every agent (with the agents' tails, if any)."""
    import numpy as np

    from oracle import attention, codec, lloyd_max
    from shared_quantized_kv_gb300 import workloads as wl

    w = wl.WORKLOADS[name]
    for b in set(w.bits_list()):
        lloyd_max.tables_f32(b)
    work = []
    for l in layers:
        K, V = wl.layer_kv(w, l)
        enc = codec.encode_layer(K, V, w.layer_bits(l), k_block=k_block)
        tail = None
        if w.tail_max:
            Kt, Vt = wl.layer_tail(w, l)
            tail = (Kt, Vt, np.full(w.agents, w.tail_len(w.decode_steps - 1)))
        work.append((enc, wl.layer_q(w, l), tail))
    for r in range(reps):
        barrier.wait()
        t0 = time.perf_counter()
        for enc, Q, tail in work:
            Kh, Vh = attention.dequantise_f64(enc)
            attention.attend_f64(Kh, Vh, Q, tail)
        results.put((r, time.perf_counter() - t0))


def oracle_decode_times(name, k_block, workers, layers, reps):
    """Seconds of `reps` oracle decode steps over `layers`, spread round-robin
    over `workers` single-threaded processes that start each step together;
    a step takes as long as its slowest worker."""
    import multiprocessing as mp

    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "CUDA_VISIBLE_DEVICES")
    saved = {k: os.environ.get(k) for k in env_keys}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                      CUDA_VISIBLE_DEVICES="")  # inherited by the spawned workers
    try:
        ctx = mp.get_context("spawn")
        workers = max(1, min(workers, len(layers)))
        barrier = ctx.Barrier(workers)
        results = ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(name, layers[i::workers], k_block, reps, barrier, results))
                 for i in range(workers)]
        for p in procs:
            p.start()
        per_rep = [[] for _ in range(reps)]
        for _ in range(workers * reps):
            r, t = results.get(timeout=1800)
            per_rep[r].append(t)
        for p in procs:
            p.join()
            if p.exitcode != 0:
                raise RuntimeError(f"oracle worker exited with {p.exitcode}")
        return [max(ts) for ts in per_rep]
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def cpu_baseline(w, k_block: int = 0) -> dict:
    """The oracle's decode step on the host: every layer spread over all
    cores (one process per core), and a sample of layers on one core scaled
    to the full step; median of 3 each."""
    cores = os.cpu_count() or 1
    t_all = statistics.median(oracle_decode_times(w.name, k_block, cores, list(range(w.layers)), 3))
    sample = list(range(min(w.layers, 4)))
    t_one = statistics.median(oracle_decode_times(w.name, k_block, 1, sample, 3)) * w.layers / len(sample)
    return {"value": round(w.agents / t_all, 4), "unit": UNIT, "cores": min(cores, w.layers), "kind": "oracle",
            "one_core": {"value": round(w.agents / t_one, 4), "cores": 1,
                         "sample": f"{len(sample)} of {w.layers} layers, scaled to the full step"},
            "host_cores": cores,
            "sample": f"the full decode step ({w.layers} layers: float64 dequantisation of the stored "
                      f"codes + float64 attention of all {w.agents} agents), layers spread over "
                      f"{min(cores, w.layers)} single-threaded processes; median of 3 steps"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from shared_quantized_kv_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    times = oracle_decode_times(w.name, args.k_block, cores, list(range(w.layers)), args.warmup + args.steps)
    step_s = statistics.mean(times[args.warmup:])
    value = w.agents / step_s
    used = min(cores, w.layers)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 2), "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f64 attention over the dequantised pool", "data": "synthetic (seeded)",
        "config": dict(workload_config(w, ws, args.k_block),
                       timing=f"full decode step on the host CPU, layers spread over {used} processes"),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"every step is the full {w.layers}-layer decode step; "
                                   f"{args.warmup} untimed + {args.steps} timed"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama3_8b_4k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--e2e-chunk", type=int, default=1,
                    help="end-to-end leg: layers per host<->device copy (default 1)")
    ap.add_argument("--per-layer-calls", action="store_true",
                    help="compress and decompress one layer per call (default: all layers in one call)")
    ap.add_argument("--k-block", type=int, default=0, choices=[0, 32],
                    help="K scales: 0 = one per layer (default), 32 = one per 32 elements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
