"""Float64 decode attention over the dequantised pool plus private bf16 tails.

Source: PolyKV summary, section 2.A: every PooledAgent reads the one shared,
compressed pool (it injects the decompressed K/V into its own cache and runs
ordinary attention); CoMixKV article, incremental quantisation: recent states
stay at native precision (the per-agent bf16 tail). The result every agent must
get is ordinary softmax attention over the dequantised shared context followed
by its own tail, which is what this module computes, by the plain definition:

  K_hat_t = q_t * s                             (float64)
  V_hat_t = n_t * H c[codes_t] / d              (float64, H the Sylvester
                                                 Hadamard matrix, c the float32
                                                 centroid table)
  for agent a, query head h, kv head g = floor(h / G)  (consecutive grouping):
    logit_t = scale * <q_{a,h}, K_t> over the pool tokens of head g, then the
              tail tokens of (a, g)
    p = softmax(logit) with the maximum subtracted
    o_{a,h} = sum_t p_t V_t

``scale`` defaults to 1/sqrt(d). K and Q arrive after positional encoding, as a
model's cache would hold them. Pinned by tests/test_oracle_attention.py (a pure
Python double loop on tiny inputs, equal-logit and dominant-logit closed forms,
tail-only cases).
"""

from __future__ import annotations

import numpy as np

from . import codec, lloyd_max


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (float64): H_ij = (-1)^popcount(i&j)."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def dequantise_f64(enc: dict):
    """(K_hat, V_hat) in float64, [kv_heads, ctx, d], from the stored codes."""
    codes = enc["codes"]
    d = codes.shape[-1]
    # centroid of every code (per-group widths: each token's own table)
    widths = codec.token_widths(enc, codes.shape[1])
    cval = np.zeros(codes.shape, dtype=np.float64)
    for b in np.unique(widths):
        cen, _ = lloyd_max.tables_f32(int(b))
        sel = widths == b
        cval[:, sel] = cen.astype(np.float64)[codes[:, sel]]
    if enc.get("k_block"):
        kb = enc["k_block"]
        q = enc["kq"].astype(np.float64)
        K = (q.reshape(q.shape[:-1] + (d // kb, kb)) * enc["kscales"].astype(np.float64)[..., None]).reshape(q.shape)
    else:
        K = enc["kq"].astype(np.float64) * float(enc["scale"])
    rot = cval * enc["norms"].astype(np.float64)[..., None]
    V = rot @ hadamard(d) / d
    return K, V


def attend_f64(K_hat, V_hat, Q_bf16, tail=None, scale=None) -> np.ndarray:
    """Decode attention of all agents.

    K_hat, V_hat: float64 [kv_heads, ctx, d]; Q_bf16: uint16 [agents, q_heads, d];
    tail: None or (K_tail_bf16, V_tail_bf16, lens) with the tails of shape
    [agents, kv_heads, T_max, d] and lens an int array [agents];
    returns float64 [agents, q_heads, d].
    """
    A, Hq, d = Q_bf16.shape
    Hk = K_hat.shape[0]
    G = Hq // Hk
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    Q = codec.bf16_to_f32(Q_bf16).astype(np.float64)
    if tail is not None:
        Kt = codec.bf16_to_f32(tail[0]).astype(np.float64)
        Vt = codec.bf16_to_f32(tail[1]).astype(np.float64)
        lens = np.asarray(tail[2])
    out = np.zeros((A, Hq, d))
    for a in range(A):
        for g in range(Hk):
            q = Q[a, g * G:(g + 1) * G]  # [G, d]
            keys, vals = K_hat[g], V_hat[g]
            if tail is not None and lens[a] > 0:
                keys = np.concatenate([keys, Kt[a, g, :lens[a]]])
                vals = np.concatenate([vals, Vt[a, g, :lens[a]]])
            logits = scale * (q @ keys.T)  # [G, T + tail]
            logits -= logits.max(axis=1, keepdims=True)
            p = np.exp(logits)
            p /= p.sum(axis=1, keepdims=True)
            out[a, g * G:(g + 1) * G] = p @ vals
    return out


def attend_rows_f64(K_hat, V_hat, Q_bf16, rows, tail=None, scale=None) -> np.ndarray:
    """The same as :func:`attend_f64` for a sample of (agent, q_head) pairs
    only: returns float64 [len(rows), d]."""
    A, Hq, d = Q_bf16.shape
    Hk = K_hat.shape[0]
    G = Hq // Hk
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((len(rows), d))
    for i, (a, h) in enumerate(rows):
        g = h // G
        q = codec.bf16_to_f32(Q_bf16[a, h]).astype(np.float64)
        keys, vals = K_hat[g], V_hat[g]
        if tail is not None and tail[2][a] > 0:
            n = int(tail[2][a])
            keys = np.concatenate([keys, codec.bf16_to_f32(tail[0][a, g, :n]).astype(np.float64)])
            vals = np.concatenate([vals, codec.bf16_to_f32(tail[1][a, g, :n]).astype(np.float64)])
        logits = scale * (keys @ q)
        logits -= logits.max()
        p = np.exp(logits)
        p /= p.sum()
        out[i] = p @ vals
    return out


def row_rel_error(out: np.ndarray, ref: np.ndarray) -> float:
    """Error metric of the attention parity bar: per output row (last axis),
    max_i |o_i - r_i| / max_i |r_i|; returns the maximum over rows."""
    o = np.asarray(out, dtype=np.float64).reshape(-1, out.shape[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    num = np.max(np.abs(o - r), axis=1)
    den = np.maximum(np.max(np.abs(r), axis=1), 1e-30)
    return float(np.max(num / den)) if len(num) else 0.0


# ------------------------------------------------------------ context split
# Softmax attention splits over the context: over each slice S of the tokens
# a row keeps lse2_S = log2 sum_{t in S} 2^(x_t) (x_t the logit in log2
# units) and the slice's own normalised output o_S; the output over the
# union is sum_S 2^(lse2_S - M) o_S / sum_S 2^(lse2_S - M), M = max_S lse2_S.
# This is the log-sum-exp combination of softmax partial sums; the functions
# below write it out in float64.

def attend_slice_f64(K_hat, V_hat, Q_bf16, t_begin, t_end, scale=None):
    """Attention state of every (agent, query head) row over pool tokens
    [t_begin, t_end): returns (lse2 float64 [agents, q_heads], o float64
    [agents, q_heads, d]), o the softmax-weighted mean of V_hat over the
    slice."""
    A, Hq, d = Q_bf16.shape
    Hk = K_hat.shape[0]
    G = Hq // Hk
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    Q = codec.bf16_to_f32(Q_bf16).astype(np.float64)
    lse2 = np.full((A, Hq), -np.inf)
    out = np.zeros((A, Hq, d))
    for a in range(A):
        for g in range(Hk):
            q = Q[a, g * G:(g + 1) * G]
            x = scale * (q @ K_hat[g, t_begin:t_end].T) / np.log(2.0)  # log2 units
            m = x.max(axis=1, keepdims=True)
            w = np.exp2(x - m)
            s = w.sum(axis=1, keepdims=True)
            lse2[a, g * G:(g + 1) * G] = (m + np.log2(s))[:, 0]
            out[a, g * G:(g + 1) * G] = (w / s) @ V_hat[g, t_begin:t_end]
    return lse2, out


def tail_slice_f64(Q_bf16, tail, kv_heads, scale=None):
    """The same state over each agent's private bf16 tail tokens (rows of an
    agent with no tail token: lse2 = -inf, o = 0)."""
    A, Hq, d = Q_bf16.shape
    G = Hq // kv_heads
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    Q = codec.bf16_to_f32(Q_bf16).astype(np.float64)
    Kt = codec.bf16_to_f32(tail[0]).astype(np.float64)
    Vt = codec.bf16_to_f32(tail[1]).astype(np.float64)
    lens = np.asarray(tail[2])
    lse2 = np.full((A, Hq), -np.inf)
    out = np.zeros((A, Hq, d))
    for a in range(A):
        n = int(lens[a])
        if n <= 0:
            continue
        for g in range(kv_heads):
            q = Q[a, g * G:(g + 1) * G]
            x = scale * (q @ Kt[a, g, :n].T) / np.log(2.0)
            m = x.max(axis=1, keepdims=True)
            w = np.exp2(x - m)
            s = w.sum(axis=1, keepdims=True)
            lse2[a, g * G:(g + 1) * G] = (m + np.log2(s))[:, 0]
            out[a, g * G:(g + 1) * G] = (w / s) @ Vt[a, g, :n]
    return lse2, out


def merge_slices_f64(parts):
    """Combine slice states [(lse2, o), ...] into the output over their
    union (parts with lse2 = -inf for a row carry no weight there)."""
    lse = np.stack([p[0] for p in parts])  # [P, A, Hq]
    outs = np.stack([p[1] for p in parts])  # [P, A, Hq, d]
    M = lse.max(axis=0)
    w = np.where(np.isfinite(lse), np.exp2(lse - M), 0.0)
    return (w[..., None] * outs).sum(axis=0) / w.sum(axis=0)[..., None]
