"""Seeded synthetic workloads for the shared quantized KV pool.

This module holds the shapes of the five workloads and the seeded generators of
their input tensors. It contains none of the method's arithmetic (no
quantisation, no rotation, no attention): it only draws numbers and rounds them
to bf16, so both the CUDA path and the CPU oracle can consume the same bytes.

Shapes follow the models the pages evaluate on (PolyKV summary, "4. Experimental
results": SmolLM2-1.7B and Llama-3-8B, contexts 600 to 7,194 tokens, up to 15
agents; CoMixKV article: Qwen3-32B with 2/3/4-bit mixed precision). No model
weights or text are involved: the tensors are random with the channel
statistics below.

Distributions
-------------
* ``tiny``: K, V, Q ~ N(0, 1); in each head, 2 channels (drawn per tensor) are
  scaled by 8.
* all others: K and V have a per-(kv-head, channel) standard deviation drawn
  from LogNormal(0, 0.5); round(1% of kv_heads*head_dim) (head, channel) pairs
  are outliers scaled by 10; Q ~ N(0, 1). The private recent-token tail of an
  agent uses the same per-channel statistics as the layer's K / V.

Every draw comes from ``numpy.random.default_rng`` seeded through
``SeedSequence(seed, spawn_key=(config index, layer, tensor id, step))`` and is
rounded to bf16 with round-to-nearest-even.
"""

from __future__ import annotations

import dataclasses

import numpy as np

# tensor ids for the seed sub-streams
_T_K, _T_V, _T_Q, _T_KTAIL, _T_VTAIL, _T_KSTAT, _T_VSTAT = range(7)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    layers: int
    kv_heads: int
    q_heads: int
    head_dim: int
    ctx: int
    agents: int
    dist: str  # "tiny" or "lognormal"
    tail_init: int = 0  # private bf16 tail tokens per agent before the first step
    decode_steps: int = 1  # decode steps; each appends one token to every tail
    bits: tuple = ()  # per-layer V bit width; empty means 3 for every layer

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def rows(self) -> int:
        """Query rows that share one KV head: agents x GQA group."""
        return self.agents * self.group

    @property
    def tail_max(self) -> int:
        return self.tail_init + self.decode_steps if self.tail_init else 0

    def layer_bits(self, layer: int) -> int:
        return self.bits[layer] if self.bits else 3

    def bits_list(self) -> list:
        return [self.layer_bits(l) for l in range(self.layers)]

    def tail_len(self, step: int) -> int:
        """Tail length seen by decode step ``step`` (0-based): the token of the
        step is appended before attention, so lengths run tail_init+1 ...
        tail_init+decode_steps."""
        return self.tail_init + step + 1 if self.tail_init else 0


def _qwen_bits() -> tuple:
    """21 layers at 2 bits, 22 at 3, 21 at 4 (mean exactly 3.0), in a seeded
    order."""
    base = np.array([2] * 21 + [3] * 22 + [4] * 21)
    perm = np.random.default_rng(0).permutation(64)
    return tuple(int(b) for b in base[perm])


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 0, 1, 2, 4, 64, 256, 3, "tiny"),
        Workload("smollm2_2k", 1, 24, 32, 32, 64, 2048, 10, "lognormal"),
        Workload("llama3_8b_4k", 2, 32, 8, 32, 128, 4096, 15, "lognormal"),
        Workload("llama3_8b_long", 3, 32, 8, 32, 128, 7194, 15, "lognormal",
                 tail_init=128, decode_steps=4),
        Workload("qwen3_32b_32k", 4, 64, 8, 64, 128, 32768, 32, "lognormal",
                 bits=_qwen_bits()),
    ]
}


# ---------------------------------------------------------------- bf16 bytes

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- generators

def _rng(w: Workload, layer: int, tensor: int, step: int = 0, seed: int = 0):
    ss = np.random.SeedSequence(seed, spawn_key=(w.index, layer, tensor, step))
    return np.random.default_rng(ss)


def _channel_std(w: Workload, layer: int, which: int, seed: int) -> np.ndarray:
    """Per-(kv-head, channel) standard deviation of K (which=_T_KSTAT) or V."""
    hk, d = w.kv_heads, w.head_dim
    rng = _rng(w, layer, which, 0, seed)
    if w.dist == "tiny":
        std = np.ones((hk, d), np.float32)
        for h in range(hk):
            std[h, rng.choice(d, 2, replace=False)] = 8.0
        return std
    std = rng.lognormal(0.0, 0.5, size=(hk, d)).astype(np.float32)
    n_out = int(round(0.01 * hk * d))
    flat = rng.choice(hk * d, n_out, replace=False)
    std.reshape(-1)[flat] *= 10.0
    return std


def layer_kv(w: Workload, layer: int, seed: int = 0):
    """Shared-context K and V of one layer: two uint16 (bf16 bits) arrays of
    shape [kv_heads, ctx, head_dim]."""
    out = []
    for tid, sid in ((_T_K, _T_KSTAT), (_T_V, _T_VSTAT)):
        std = _channel_std(w, layer, sid, seed)
        rng = _rng(w, layer, tid, 0, seed)
        x = rng.standard_normal((w.kv_heads, w.ctx, w.head_dim), dtype=np.float32)
        x *= std[:, None, :]
        out.append(f32_to_bf16_bits(x))
    return out[0], out[1]


def layer_q(w: Workload, layer: int, step: int = 0, seed: int = 0) -> np.ndarray:
    """Decode queries of all agents for one layer: uint16 [agents, q_heads, d]."""
    rng = _rng(w, layer, _T_Q, step, seed)
    x = rng.standard_normal((w.agents, w.q_heads, w.head_dim), dtype=np.float32)
    if w.dist == "tiny":
        for h in range(w.q_heads):
            x[:, h, rng.choice(w.head_dim, 2, replace=False)] *= 8.0
    return f32_to_bf16_bits(x)


def layer_tail(w: Workload, layer: int, seed: int = 0):
    """Private recent-token tails of all agents, full capacity ``tail_max``:
    uint16 K, V of shape [agents, kv_heads, tail_max, head_dim]. Decode step s
    uses the first ``tail_len(s)`` tokens of each agent."""
    if not w.tail_max:
        return None, None
    out = []
    for tid, sid in ((_T_KTAIL, _T_KSTAT), (_T_VTAIL, _T_VSTAT)):
        std = _channel_std(w, layer, sid, seed)
        rng = _rng(w, layer, tid, 0, seed)
        x = rng.standard_normal((w.agents, w.kv_heads, w.tail_max, w.head_dim),
                                dtype=np.float32)
        x *= std[None, :, None, :]
        out.append(f32_to_bf16_bits(x))
    return out[0], out[1]


def custom(name="custom", layers=1, kv_heads=2, q_heads=4, head_dim=64, ctx=256,
           agents=3, dist="lognormal", tail_init=0, decode_steps=1, bits=(),
           index=99) -> Workload:
    """A workload of arbitrary shape (tests of edge cases)."""
    return Workload(name, index, layers, kv_heads, q_heads, head_dim, ctx, agents,
                    dist, tail_init, decode_steps, tuple(bits))


# ------------------------------------------------- fast device-side generator

def layer_kv_torch(w: Workload, layer: int, device, seed: int = 0):
    """Same recipe as :func:`layer_kv`, drawn with torch on ``device`` (used by
    the benchmark, where numpy generation of gigabytes would dominate set-up).
    Returns two bf16 tensors [kv_heads, ctx, head_dim]."""
    import torch

    outs = []
    for tid, sid in ((_T_K, _T_KSTAT), (_T_V, _T_VSTAT)):
        std = torch.from_numpy(_channel_std(w, layer, sid, seed)).to(device)
        g = torch.Generator(device=device)
        g.manual_seed(int(np.random.SeedSequence(
            seed, spawn_key=(w.index, layer, tid, 0)).generate_state(1)[0]))
        x = torch.randn((w.kv_heads, w.ctx, w.head_dim), generator=g, device=device,
                        dtype=torch.float32)
        x *= std[:, None, :]
        outs.append(x.to(torch.bfloat16))
    return outs[0], outs[1]
