"""Decode attention over one shared pool whose context is split across ranks
(one process per GPU).

The PolyKV summary's pool is one object that every agent reads (section 2.A).
Across GPUs it can be split two ways without changing what any agent
computes:

* by KV head: rank r holds the pool of its share of the KV heads and serves
  the query heads that read them; attention needs no exchange (the outputs of
  all heads meet later, at the output projection, outside this path);
* by context: rank r holds a slice of the shared context's tokens. Every rank
  computes, for every (agent, query head) row, the softmax state of its slice
  (kvpool_attend_partial: a reference maximum m, the weight sum l and the
  rotated-domain accumulator), the states are all-gathered, and each rank
  merges them (kvpool_merge_partials: log-sum-exp combination, one inverse
  FWHT per row, the agents' private tails).

This module holds the host side of the context split: which tokens a rank
holds, the exchange, and the call sequence. The exchange is one all-gather of
rows x (head_dim + 2) floats per KV head and rank; nothing is copied through
host memory. Each rank's pool is compressed from its own slice, so with the
per-tensor K scale every slice has its own scale (block-scaled pools encode
each token on its own and are identical either way).
"""

from __future__ import annotations

TILE = 128  # slices start on a multiple of this (the attention kernel's tile)


def slice_bounds(ctx: int, rank: int, world: int, tile: int = TILE):
    """Token range [begin, end) of the shared context that rank `rank` of
    `world` holds: whole tiles, spread as evenly as possible, in rank order
    (a rank past the last tile holds an empty range)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    ntile = (ctx + tile - 1) // tile
    base, extra = divmod(ntile, world)
    first = rank * base + min(rank, extra)
    count = base + (1 if rank < extra else 0)
    begin = min(ctx, first * tile)
    end = min(ctx, (first + count) * tile)
    return begin, end


def gather(tensors, group=None):
    """All-gather each tensor of `tensors` (same shape on every rank) over the
    process group; returns, per tensor, a stacked tensor [world, ...] in rank
    order."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    out = []
    for t in tensors:
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t.contiguous(), group=group)
        out.append(torch.stack(parts))
    return out


def local_partial(pool, layer, Q, softmax_scale=0.0, stream=None):
    """This rank's softmax state over every token its pool holds (an empty
    pool slice contributes weight 0)."""
    import torch

    n = pool.layer_len(layer)
    if n > 0:
        return pool.attend_partial(layer, Q, 0, n, softmax_scale=softmax_scale, stream=stream)
    A, Hq, d = Q.shape
    R = A * (Hq // pool.kv_heads)
    ml = torch.zeros((pool.kv_heads, R, 2), dtype=torch.float32, device=Q.device)
    acc = torch.zeros((pool.kv_heads, R, d), dtype=torch.float32, device=Q.device)
    return ml, acc


def attend(pool, layer, Q, tail=None, group=None, softmax_scale=0.0, partial=None, merge=None):
    """Context-parallel decode attention of one layer: this rank's partial
    state, the all-gather, and the merge (with the agents' tails); every rank
    returns the full output float32 [agents, q_heads, head_dim].

    `partial(layer, Q)` and `merge(ml, acc, Q, tail)` default to the
    library's kvpool_attend_partial over this rank's pool and
    kvpool_merge_partials; they are parameters so that the exchange can be
    exercised on its own."""
    if partial is None:
        def partial(layer_, Q_):
            return local_partial(pool, layer_, Q_, softmax_scale)
    if merge is None:
        from . import kvpool

        def merge(ml_, acc_, Q_, tail_):
            return kvpool.merge_partials(ml_, acc_, Q_, pool.kv_heads, tail_, softmax_scale=softmax_scale)
    ml, acc = partial(layer, Q)
    ML, ACC = gather([ml, acc], group)
    return merge(ML, ACC, Q, tail)
