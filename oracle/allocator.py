"""Per-layer V bit widths under a byte budget from a local attention-error
estimate (test infrastructure: CPU only, float64, no part of the library).

Source: CoMixKV article (zicq.com), "online sensitivity estimation" and
"trade-offs": the controller builds a local attention-error bound from
recently observed queries, keys and values, and jointly chooses the layers'
bit widths (2, 3 or 4) within a total byte budget; sharp attention
distributions need more precision than flat ones. The article prints no
formula. The reading taken here (parity with the pages unpinned):

  * V error at b bits. A head-vector v is coded as y = H v / |v| with
    coordinates of unit variance, each quantised with Lloyd-Max distortion
    D_b = E (y - Q_b(y))^2 for N(0, 1); H is orthogonal up to sqrt(d), so
    E |v - v_hat|^2 = D_b |v|^2.
  * Attention output error. With independent zero-mean errors e_t,
    E |sum_t p_t e_t|^2 = D_b sum_t p_t^2 |v_t|^2. The relative error of a
    query row is sqrt(D_b) * r with r = sqrt(sum_t p_t^2 |v_t|^2) / |o|,
    o = sum_t p_t v_t, p = softmax(scale * q . k_t) over the recent tokens.
    r is 1 for a one-hot p and 1/sqrt(T) for T equal logits on one vector.
  * A layer's sensitivity s is the mean of r over its recent query rows
    (agents x query heads); its error at b bits is E(b) = sqrt(D_b) * s.
  * Allocation: bits b_l in {2, 3, 4} minimising sum_l E_l(b_l)^2 subject to
    sum_l c_l * b_l <= budget (c_l: the layer's V bytes per bit of width),
    solved exactly by dynamic programming over integer costs; among equal
    errors the cheaper allocation, then the lexicographically smaller one.
"""

from __future__ import annotations

import functools
import itertools
import math

import numpy as np

from oracle import codec, lloyd_max

BITS = (2, 3, 4)


@functools.lru_cache(maxsize=None)
def distortion(bits: int) -> float:
    """Lloyd-Max MSE for N(0, 1) at `bits` bits (float64, by quadrature)."""
    c, t = lloyd_max.lloyd_max_normal(1 << bits)
    return float(lloyd_max.mse_normal(c, t))


def row_ratio(q, K, V, scale) -> float:
    """r = sqrt(sum_t p_t^2 |v_t|^2) / |o| for one query row over tokens
    K, V [T, d] (float64); 0 when T = 0."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return 0.0
    lg = scale * (K @ q)
    p = np.exp(lg - lg.max())
    p /= p.sum()
    o = p @ V
    num = math.sqrt(float(np.sum(p * p * np.sum(V * V, axis=1))))
    den = float(np.linalg.norm(o))
    return num / den if den > 0 else 0.0


def layer_sensitivity(Q_bf16, K_bf16, V_bf16, lens, scale=None) -> float:
    """Mean of r over all (agent, query head) rows of one layer. Q: bf16
    [A, Hq, d]; K, V: bf16 recent tokens [A, Hk, T_max, d]; lens [A]. Rows of
    agents with no recent token count as 0."""
    Q = codec.bf16_to_f32(Q_bf16).astype(np.float64)
    K = codec.bf16_to_f32(K_bf16).astype(np.float64)
    V = codec.bf16_to_f32(V_bf16).astype(np.float64)
    A, Hq, d = Q.shape
    Hk = K.shape[1]
    G = Hq // Hk
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    tot = 0.0
    for a in range(A):
        n = int(lens[a])
        for h in range(Hq):
            tot += row_ratio(Q[a, h], K[a, h // G, :n], V[a, h // G, :n], sc)
    return tot / (A * Hq)


def layer_error(s: float, bits: int) -> float:
    return math.sqrt(distortion(bits)) * s


def allocate(sens, cost, budget):
    """Bits per layer (tuple) minimising sum_l (sqrt(D_b) s_l)^2 with
    sum_l cost_l * b_l <= budget (integers); None when even 2 bits
    everywhere exceed the budget."""
    L = len(sens)
    cost = [int(c) for c in cost]
    budget = int(budget)
    if sum(2 * c for c in cost) > budget:
        return None
    # best[l][u] = (error, bytes, bits of layers l..) for layers l.. with u units left
    D = {b: distortion(b) for b in BITS}
    memo = {}

    def best(l, left):
        if l == L:
            return (0.0, 0, ())
        key = (l, left)
        if key in memo:
            return memo[key]
        out = None
        for b in BITS:
            c = cost[l] * b
            rest_min = sum(2 * cc for cc in cost[l + 1:])
            if c + rest_min > left:
                continue
            e, by, bb = best(l + 1, left - c)
            cand = (D[b] * sens[l] ** 2 + e, by + c, (b,) + bb)
            if out is None or _better(cand, out):
                out = cand
        memo[key] = out
        return out

    return best(0, budget)[2]


def _better(a, b):
    """Lower error; then fewer bytes; then the lexicographically smaller bits."""
    if a[0] != b[0]:
        return a[0] < b[0]
    if a[1] != b[1]:
        return a[1] < b[1]
    return a[2] < b[2]


def allocate_brute_force(sens, cost, budget):
    """The same optimum by enumerating every allocation (tiny cases only)."""
    D = {b: distortion(b) for b in BITS}
    best = None
    for bits in itertools.product(BITS, repeat=len(sens)):
        by = sum(c * b for c, b in zip(cost, bits))
        if by > budget:
            continue
        e = sum(D[b] * s ** 2 for s, b in zip(sens, bits))
        cand = (e, by, bits)
        if best is None or _better(cand, best):
            best = cand
    return None if best is None else best[2]
