"""bench.py's reference arm (the oracle on the host CPU) prints one JSON line
with the contract's keys and the GPU arm's workload config."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "smollm2_2k"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    sys.path.insert(0, ROOT)
    import bench
    from shared_quantized_kv_gb300 import workloads as wl

    want = bench.workload_config(wl.WORKLOADS["smollm2_2k"], 1, 0)
    assert {k: d["config"][k] for k in want} == want


def test_launch_count_by_call_structure():
    sys.path.insert(0, ROOT)
    import bench
    from shared_quantized_kv_gb300 import workloads as wl

    llama = wl.WORKLOADS["llama3_8b_4k"]  # 32 layers, all 3-bit
    assert bench.launches_per_step(llama, 0, False) == {"compress": 2, "attend": 32, "attend_ws": 64,
                                                         "decompress": 1}
    assert bench.launches_per_step(llama, 0, True) == {"compress": 64, "attend": 32, "attend_ws": 64,
                                                        "decompress": 32}
    assert bench.launches_per_step(llama, 32, False)["attend"] == 32  # block-scaled K: the same kernel
    qwen = wl.WORKLOADS["qwen3_32b_32k"]  # 64 layers, 2/3/4 bits: two launch chunks of 32 layers
    widths = sum(len(set(qwen.bits_list()[c:c + 32])) for c in (0, 32))
    assert bench.launches_per_step(qwen, 0, False) == {"compress": 2 + widths, "attend": 64, "attend_ws": 128,
                                                        "decompress": widths}
