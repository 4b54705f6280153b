"""Benchmark of the shared quantized KV pool hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input on
the Llama-3-8B-shaped workload (32 layers, 8 KV heads, 32 query heads,
head_dim 128, 4096 shared-context tokens, 15 agents x 1 decode query, int8 K,
3-bit V): compress every layer (write-once encode of the shared context, all
layers in one call), attend every layer for all agents (one call per layer:
a layer's queries depend on the layer before), decompress every layer (the
per-agent materialisation path, all layers in one call). The three
phases are each captured once as a CUDA graph and replayed; CUDA events around
each replay give the per-phase device time, and L2 is flushed (a 512 MiB
write) before every phase, outside the events.

value = agents x ranks / (max over ranks of the mean step time): agent-decode
steps per second of the full path. The attend phase alone is reported under
"phases" with its fraction of the measured HBM copy bandwidth.

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
            "step": "compress+attend+decompress, all layers",
            "parallelism": f"replicas x{ws} (independent pools, no collective)"}


def launches_per_step(w, k_block, per_layer_calls, batch=32):
    """The library's kernel launches in one step, by phase. Compress: a max|K|
    kernel and an encode kernel per layer, or, for all layers in one call, one
    max|K| kernel and one encode kernel per V width per 32 layers. Attend: the
    tensor-core kernel per layer, or the split and combine kernels (block-
    scaled K). Decompress: one kernel per layer, or one per V width per 32
    layers."""
    bits = w.bits_list()
    chunks = [bits[i:i + batch] for i in range(0, len(bits), batch)]
    widths = sum(len(set(c)) for c in chunks)
    if per_layer_calls:
        comp, dec = 2 * len(bits), len(bits)
    else:
        comp, dec = len(chunks) + widths, widths
    return {"compress": comp, "attend": len(bits) * (2 if k_block else 1), "decompress": dec}


def max_over_ranks(step_ms, ph_ms, phases, device=None):
    """(step time, per-phase times) as the maximum over the ranks of the
    default process group (unchanged when no group is initialised). Ranks are
    replicas: the job takes as long as its slowest rank."""
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
    pool = kvpool.KVPool(L, w.kv_heads, w.head_dim, w.ctx, w.bits_list(), max_rows=max(w.rows, 1),
                         k_block=args.k_block)
    seed = rank  # each rank serves its own agents over its own pool
    K, V = [], []
    for l in range(L):
        k, v = wl.layer_kv_torch(w, l, dev, seed)
        K.append(k)
        V.append(v)
    Q = [torch.from_numpy(wl.layer_q(w, l, 0, seed).view(np.int16)).to(dev).view(torch.bfloat16)
         for l in range(L)]
    tail = None
    if w.tail_max:
        tail = []
        for l in range(L):
            kt, vt = wl.layer_tail(w, l, seed)
            lens = torch.full((A,), w.tail_len(w.decode_steps - 1), dtype=torch.int32, device=dev)
            tail.append((torch.from_numpy(kt.view(np.int16)).to(dev).view(torch.bfloat16),
                         torch.from_numpy(vt.view(np.int16)).to(dev).view(torch.bfloat16), lens))
    out = [torch.empty((A, w.q_heads, w.head_dim), dtype=torch.float32, device=dev) for _ in range(L)]
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

    def attend():  # per layer: layer l + 1's queries come from layer l's output
        for l in layers:
            pool.attend(l, Q[l], out[l], tail[l] if tail else None)

    def decompress():
        if args.per_layer_calls:
            for l in layers:
                pool.decompress(l, Kd[l], Vd[l])
        else:
            pool.decompress_layers(layers, Kd, Vd)

    # eager once (state + correctness of the calls), then capture each phase
    compress(); attend(); decompress()
    assert pool.status() == 0
    graphs = {}
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    for name, fn in (("compress", compress), ("attend", attend), ("decompress", decompress)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        graphs[name] = g
    torch.cuda.synchronize()

    phases = ("compress", "attend", "decompress")

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
    clocks = dict(sampler.stop(), window="0.6 s of the same step untimed, then the timed steps")
    assert pool.status() == 0

    ph_ms = {ph: 0.0 for ph in phases}
    for ev in rec:
        for ph, e0, e1 in ev:
            ph_ms[ph] += e0.elapsed_time(e1)
    ph_ms = {ph: v / args.steps for ph, v in ph_ms.items()}
    step_ms, ph_ms = max_over_ranks(sum(ph_ms.values()), ph_ms, phases, dev if ws > 1 else None)

    launches = launches_per_step(w, args.k_block, args.per_layer_calls)
    # algorithmic bytes per layer
    nvec = w.kv_heads * w.ctx
    kv_in = 2 * nvec * w.head_dim * 2
    pool_layer = pool.pool_bytes() / L
    tail_bytes = 2 * A * w.kv_heads * w.tail_len(w.decode_steps - 1) * w.head_dim * 2 if tail else 0
    algo = {"compress": kv_in + pool_layer, "attend": pool_layer + tail_bytes,
            "decompress": pool_layer + kv_in}
    peak, peak_kind = _peaks()
    ph_info = {}
    for ph in phases:
        per_call_s = ph_ms[ph] / 1e3 / L
        gbs = algo[ph] / per_call_s / 1e9
        ph_info[ph] = {"ms_per_step": round(ph_ms[ph], 4), "us_per_layer": round(per_call_s * 1e6, 3),
                       "algo_bytes_per_layer": int(algo[ph]), "GB_per_s": round(gbs, 1),
                       "hbm_frac": round(gbs / peak, 4), "launches_per_step": launches[ph]}
    ph_info["attend"]["agent_steps_per_s"] = round(A * ws / (ph_ms["attend"] / 1e3), 1)
    dom = max(phases, key=lambda p: ph_ms[p])
    dom_file = {"compress": "encode.cu", "attend": "attend_tc_impl.cuh", "decompress": "decompress.cu"}[dom]

    # end to end through the same calls with pinned host buffers
    e2e = run_e2e(args, pool, w, K, V, Q, tail, out, Kd, Vd, phases) if not args.no_e2e else None

    value = A * ws / (step_ms / 1e3)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8/u3+f32",
        "data": "synthetic (seeded; bf16 K/V with LogNormal(0,0.5) channel std and 1% x10 outlier "
                "channels, Q ~ N(0,1))",
        "config": dict(workload_config(w, ws, args.k_block),
                       calls="one call per layer" if args.per_layer_calls else
                       "compress and decompress: all layers per call; attend: one call per layer",
                       l2="flushed (512 MiB write) before every phase, outside the timed events"),
        "phases": ph_info,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ph_info[dom]["GB_per_s"],
                     "peak": peak, "unit": "GB/s", "frac": ph_info[dom]["hbm_frac"],
                     "traffic": _traffic(dom_file), "peak_source": peak_kind,
                     "algo_bytes_per_launch": int(algo[dom])},
        "gpu_launches": args.steps * sum(launches.values()),
        "clocks": clocks,
        "wall_s_timed": round(t_wall, 3),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, k_block=args.k_block)
    if rank == 0:
        print(json.dumps(line), flush=True)
    pool.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e(args, pool, w, K, V, Q, tail, out, Kd, Vd, phases):
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
                pool.attend(l, q, o, tail[l] if tail else None, stream=s_main)
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
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": round(w.agents * ws / (ms / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "how": "one CUDA graph per step: three streams pipelined over layers (upload, compute, download), "
                   f"one copy per {per} layer(s) each way"}


# ------------------------------------------------------------------ CPU legs

def _oracle_sample(name: str, layers: int, k_block: int = 0) -> dict:
    """Time the oracle (as it stands) on the first `layers` layers of the
    workload: encode, float64 attention for all agents, decompress. Runs in a
    fresh interpreter with one BLAS thread."""
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
from shared_quantized_kv_gb300 import workloads as wl
from oracle import attention, codec, lloyd_max
w = wl.WORKLOADS[{name!r}]
for b in set(w.bits_list()): lloyd_max.tables_f32(b)
t = 0.0
for l in range({layers}):
    K, V = wl.layer_kv(w, l)
    Q = wl.layer_q(w, l)
    tail = None
    if w.tail_max:
        Kt, Vt = wl.layer_tail(w, l)
        import numpy as np
        tail = (Kt, Vt, np.full(w.agents, w.tail_len(w.decode_steps - 1)))
    t0 = time.perf_counter()
    enc = codec.encode_layer(K, V, w.layer_bits(l), k_block={k_block})
    Kh, Vh = attention.dequantise_f64(enc)
    attention.attend_f64(Kh, Vh, Q, tail)
    codec.decompress_layer(enc)
    t += time.perf_counter() - t0
print(json.dumps({{"seconds": t, "layers": {layers}}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(w, layers: int = 1, k_block: int = 0) -> dict:
    res = _oracle_sample(w.name, layers, k_block)
    per_step = res["seconds"] / layers * w.layers
    return {"value": round(w.agents / per_step, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{layers} of {w.layers} layers (encode + float64 attention of all "
                      f"{w.agents} agents + decompress), scaled to a full step; "
                      f"{res['seconds']:.2f} s of CPU time; host has {os.cpu_count()} cores"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from shared_quantized_kv_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    _oracle_sample(w.name, 1, args.k_block)  # warm-up of the interpreter and tables
    times = []
    for _ in range(args.warmup):
        _oracle_sample(w.name, 1, args.k_block)
    for _ in range(args.steps):
        r = _oracle_sample(w.name, 1, args.k_block)
        times.append(r["seconds"] * w.layers)  # one layer per step, scaled to all layers
    step_s = statistics.mean(times)
    value = w.agents / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 encode / f64 attention", "data": "synthetic (seeded)",
        "config": dict(workload_config(w, ws, args.k_block),
                       timing="one layer per step on the host CPU, scaled to all layers"),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "1 layer per step scaled to all layers; one thread"},
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
