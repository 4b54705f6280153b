"""Write-once encode and decompress of one pool layer (float32, IEEE order).

Source: PolyKV summary, section 2.B "asymmetric compression scheme
(TurboQuant MSE)":
  * K: per-tensor linear quantisation to int8;
  * V: rotate each head-vector with the fast Walsh-Hadamard transform so the
    coordinates approach N(0, 1), map each coordinate to the pre-computed
    Lloyd-Max centroid for N(0, 1) (3 bits), dequantise by centroid lookup and
    the inverse FWHT.
CoMixKV article (2-4 bit per layer): the same V pipeline with 4 or 16 levels.

The codes are integers decided by float32 arithmetic, so the exact sequence of
float32 operations is part of the definition; the CUDA encoder must reproduce
it bit for bit. Readings where the pages are silent (all stated once more in
the design notes):

K (one layer, tensor [kv_heads, ctx, head_dim] of bf16):
  absmax = max |k| (exact); s = absmax / 127 (float32 division), s = 1 when
  absmax = 0; q = clamp(round_half_even(k / s), -127, 127) with a float32
  division. Symmetric: -128 is never produced.

V (each head-vector v of head_dim = d values, bf16 -> float32):
  1. norm: sq_i = v_i * v_i; pairwise tree sq_i += sq_{i+w} for i < w with
     w = d/2, d/4, ..., 1; n = sqrt(sq_0) (float32, correctly rounded).
  2. FWHT, Sylvester (natural) order, unnormalised, in place: stages
     h = 1, 2, 4, ..., d/2; in each, for every pair (i, i+h) with bit h of i
     clear: (x_i, x_{i+h}) <- (x_i + x_{i+h}, x_i - x_{i+h}).
  3. The rotated vector u = Hv has coordinates of RMS n, so y = u / n ~ N(0,1).
     The nearest-centroid decision "y > m_j" for the float32 midpoints m_j is
     taken as "u_i > fl(m_j * n)" (the same cell in exact arithmetic for n > 0,
     one float32 product per midpoint and vector instead of a division per
     coordinate): code_i = #{ j : u_i > fl(m_j * n) }. A tie goes to the lower
     code. A zero vector (n = 0) yields codes that decode to exactly 0 because
     the decoded vector is scaled by n.
  4. Packing of a code sequence, little-endian: 3 bits -> groups of 8 codes
     in 3 bytes, w = sum_k code_{8g+k} << 3k, bytes (w, w>>8, w>>16) & 255;
     2 bits -> 4 codes per byte, code_{4g+k} << 2k; 4 bits -> 2 codes per
     byte, low nibble first. The pages fix the packing (8 codes in 3 bytes)
     but not which codes form a sequence; the pool takes, per KV head, groups
     of 32 consecutive tokens and, inside a group, one sequence per rotated
     coordinate i holding the 32 tokens' codes in token order (4*bits bytes);
     the sequences of a group follow in coordinate order. Token slots past
     the context in the last group hold code 0.
  5. The norm n is stored as float32.

Decompress:
  K_hat = bf16(fl(q * s)); V_hat_i = bf16(fl(fl(z_i * n) * (1/d))) with
  z = FWHT(c[codes]) in float32 (same stage order). H H = d I, so the inverse
  transform is H / d; 1/d is a power of two and scaling by it is exact.
  bf16() rounds to nearest, ties to even.

Pinned by tests/test_oracle_codec.py (exact rational arithmetic on tiny inputs,
closed forms of the FWHT and of spike vectors, hand-derived packing bytes,
quantisation error bounds, pack/unpack round trips).
"""

from __future__ import annotations

import numpy as np

from . import lloyd_max

F32 = np.float32


# --------------------------------------------------------------- bf16 helpers

def bf16_to_f32(u16) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32)
    return (u << np.uint32(16)).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even."""
    a = np.asarray(x, dtype=np.float32)
    b = np.ascontiguousarray(a).reshape(a.shape).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


# ----------------------------------------------------------------- transforms

def fwht_f32(x: np.ndarray) -> np.ndarray:
    """Unnormalised FWHT over the last axis (length d, a power of two) in
    float32, stages h = 1, 2, ..., d/2, lower index first (x_i + x_{i+h},
    x_i - x_{i+h}). Returns a new array."""
    x = np.array(x, dtype=np.float32, copy=True)
    d = x.shape[-1]
    lead = x.shape[:-1]
    h = 1
    while h < d:
        y = x.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(lead + (d,))
        h *= 2
    return x


def norm_f32(v: np.ndarray) -> np.ndarray:
    """L2 norm over the last axis in float32: exact squares, pairwise tree sum
    sq_i += sq_{i+w} (w = d/2, ..., 1), correctly rounded square root."""
    sq = np.asarray(v, dtype=np.float32) * np.asarray(v, dtype=np.float32)
    w = sq.shape[-1] // 2
    while w >= 1:
        sq = sq[..., :w] + sq[..., w:2 * w]
        w //= 2
    return np.sqrt(sq[..., 0])


# ---------------------------------------------------------------------- K side

def k_scale(K_bf16) -> tuple:
    """(absmax, scale) of a layer's whole K tensor, both float32."""
    k = bf16_to_f32(K_bf16)
    if not np.all(np.isfinite(k)):
        raise ValueError("K holds a non-finite value")
    absmax = F32(np.max(np.abs(k))) if k.size else F32(0)
    scale = F32(absmax / F32(127)) if absmax > 0 else F32(1)
    return absmax, scale


def k_quantize(K_bf16, scale) -> np.ndarray:
    k = bf16_to_f32(K_bf16)
    r = np.rint(k / F32(scale))  # float32 division, ties to even
    return np.clip(r, -127, 127).astype(np.int8)


def k_dequantize_bf16(q: np.ndarray, scale) -> np.ndarray:
    return f32_to_bf16(q.astype(np.float32) * F32(scale))


# Block-scaled K (the "q8_0" reading of the PolyKV summary's section 2.B, a
# per-pool option): one scale per block of 32 consecutive elements of a
# head-vector, s_b = max|k| / 127 over the block (float32 division; 1 for an
# all-zero block), q = clamp(round_half_even(k / s_b), -127, 127) with a
# float32 division. Scales are kept as float32 (not q8_0's fp16: a bf16 K
# spans a range that fp16 cannot hold).
K_BLOCK = 32


def k_scales_block(K_bf16) -> np.ndarray:
    """Scales [..., d / 32] float32 of a K tensor [..., d]."""
    k = bf16_to_f32(K_bf16)
    if not np.all(np.isfinite(k)):
        raise ValueError("K holds a non-finite value")
    b = k.reshape(k.shape[:-1] + (k.shape[-1] // K_BLOCK, K_BLOCK))
    absmax = np.max(np.abs(b), axis=-1).astype(np.float32)
    return np.where(absmax > 0, absmax / F32(127), F32(1)).astype(np.float32)


def k_quantize_block(K_bf16, scales) -> np.ndarray:
    k = bf16_to_f32(K_bf16)
    b = k.reshape(k.shape[:-1] + (k.shape[-1] // K_BLOCK, K_BLOCK))
    r = np.rint(b / np.asarray(scales, dtype=np.float32)[..., None])  # float32 division, ties to even
    return np.clip(r, -127, 127).astype(np.int8).reshape(k.shape)


def k_dequantize_block_bf16(q: np.ndarray, scales) -> np.ndarray:
    b = q.astype(np.float32).reshape(q.shape[:-1] + (q.shape[-1] // K_BLOCK, K_BLOCK))
    return f32_to_bf16(b * np.asarray(scales, dtype=np.float32)[..., None]).reshape(q.shape)


# ---------------------------------------------------------------------- V side

def v_codes(V_bf16, bits: int):
    """Codes (uint8, same shape as V) and float32 norms (shape V.shape[:-1])."""
    _, mid = lloyd_max.tables_f32(bits)
    v = bf16_to_f32(V_bf16)
    if not np.all(np.isfinite(v)):
        raise ValueError("V holds a non-finite value")
    n = norm_f32(v)
    if not np.all(np.isfinite(n)):
        raise ValueError("a V norm is not finite")
    u = fwht_f32(v)
    codes = np.zeros(u.shape, dtype=np.uint8)
    for m in mid:
        tau = (F32(m) * n)[..., None]  # float32 product, one per vector
        codes += (u > tau)
    return codes, n


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes [..., d] into bytes [..., d*bits/8], little-endian."""
    c = np.asarray(codes, dtype=np.uint32)
    d = c.shape[-1]
    lead = c.shape[:-1]
    if bits == 3:
        g = c.reshape(lead + (d // 8, 8))
        w = np.zeros(lead + (d // 8,), dtype=np.uint32)
        for k in range(8):
            w |= g[..., k] << np.uint32(3 * k)
        out = np.stack([w & 255, (w >> 8) & 255, (w >> 16) & 255], axis=-1)
        return out.reshape(lead + (3 * d // 8,)).astype(np.uint8)
    if bits == 2:
        g = c.reshape(lead + (d // 4, 4))
        out = g[..., 0] | (g[..., 1] << 2) | (g[..., 2] << 4) | (g[..., 3] << 6)
        return out.astype(np.uint8)
    if bits == 4:
        g = c.reshape(lead + (d // 2, 2))
        return (g[..., 0] | (g[..., 1] << 4)).astype(np.uint8)
    raise ValueError("bits must be 2, 3 or 4")


def unpack_codes(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint32)
    lead = p.shape[:-1]
    if bits == 3:
        g = p.reshape(lead + (d // 8, 3))
        w = g[..., 0] | (g[..., 1] << 8) | (g[..., 2] << 16)
        out = np.stack([(w >> np.uint32(3 * k)) & 7 for k in range(8)], axis=-1)
    elif bits == 2:
        out = np.stack([(p >> np.uint32(2 * k)) & 3 for k in range(4)], axis=-1)
    elif bits == 4:
        out = np.stack([p & 15, p >> 4], axis=-1)
    else:
        raise ValueError("bits must be 2, 3 or 4")
    return out.reshape(lead + (d,)).astype(np.uint8)


GROUP = 32  # tokens per packed V group in the pool


def pack_pool_v(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pool layout of one layer's V codes: [kv_heads, ctx, d] -> uint8
    [kv_heads, ceil(ctx/32), d, 4*bits] (step 4 above)."""
    c = np.asarray(codes, dtype=np.uint8)
    H, T, d = c.shape
    ng = -(-T // GROUP)
    pad = np.zeros((H, ng * GROUP, d), dtype=np.uint8)
    pad[:, :T] = c
    seq = pad.reshape(H, ng, GROUP, d).transpose(0, 1, 3, 2)  # [H, group, coordinate, token]
    return pack_codes(seq, bits)


def unpack_pool_v(packed: np.ndarray, bits: int, ctx: int) -> np.ndarray:
    """Inverse of pack_pool_v: codes [kv_heads, ctx, d]."""
    p = np.asarray(packed, dtype=np.uint8)
    H, ng, d, _ = p.shape
    seq = unpack_codes(p, bits, GROUP)  # [H, group, coordinate, token]
    return seq.transpose(0, 1, 3, 2).reshape(H, ng * GROUP, d)[:, :ctx]


def v_decompress_bf16(codes: np.ndarray, norms: np.ndarray, bits: int) -> np.ndarray:
    cen, _ = lloyd_max.tables_f32(bits)
    d = codes.shape[-1]
    z = fwht_f32(cen[codes])
    return f32_to_bf16((z * norms[..., None].astype(np.float32)) * F32(1.0 / d))


# --------------------------------------------------------------------- a layer

def encode_layer(K_bf16, V_bf16, bits: int, k_block: int = 0) -> dict:
    """Everything the pool stores for one layer. k_block = 32: block-scaled K
    (per-tensor scale 1, the block scales in "kscales")."""
    codes, norms = v_codes(V_bf16, bits)
    enc = dict(bits=bits, codes=codes, packed=pack_pool_v(codes, bits), norms=norms, k_block=k_block)
    if k_block:
        if k_block != K_BLOCK:
            raise ValueError("k_block must be 0 or 32")
        sc = k_scales_block(K_bf16)
        enc.update(absmax=F32(0), scale=F32(1), kscales=sc, kq=k_quantize_block(K_bf16, sc))
    else:
        absmax, scale = k_scale(K_bf16)
        enc.update(absmax=absmax, scale=scale, kq=k_quantize(K_bf16, scale))
    return enc


def decompress_layer(enc: dict):
    if enc.get("k_block"):
        K = k_dequantize_block_bf16(enc["kq"], enc["kscales"])
    else:
        K = k_dequantize_bf16(enc["kq"], enc["scale"])
    if enc.get("widths") is None:
        return K, v_decompress_bf16(enc["codes"], enc["norms"], enc["bits"])
    # per-group widths: each group decodes with its own table
    V = np.zeros(enc["codes"].shape, dtype=np.uint16)
    for g, b in enumerate(enc["widths"]):
        sl = slice(g * GROUP, (g + 1) * GROUP)
        V[:, sl] = v_decompress_bf16(enc["codes"][:, sl], enc["norms"][:, sl], b)
    return K, V


def layer_bytes(kv_heads: int, ctx: int, head_dim: int, bits: int) -> int:
    """Stored bytes of one layer: int8 K, packed V, float32 norms, float32 K
    scale (no padding)."""
    n = kv_heads * ctx
    return n * head_dim + n * head_dim * bits // 8 + 4 * n + 4


# ------------------------------------------------- per-group V widths (appends)
#
# CoMixKV article, section "增量量化策略" (incremental quantisation strategy):
# a width newly chosen by the allocator applies only to cache blocks quantised
# afterwards; blocks already quantised keep their width and bytes. With the
# pool's 32-token groups as the blocks, a layer is then a sequence of groups,
# group g coded at its own width b_g with the same per-vector pipeline as
# above (norm, FWHT, midpoint count against b_g's table). Readings (the
# article fixes no layout):
#   * a group's bytes are the uniform layout's bytes for those 32 tokens at
#     b_g (d sequences of 4*b_g bytes, coordinate order);
#   * per KV head the groups follow each other in token order with no gap, so
#     group g starts at byte sum_{g' < g} d * 4 * b_{g'} of the head's codes.
# A layer whose groups all have width b is exactly pack_pool_v(codes, b).


def pack_pool_v_groups(codes: np.ndarray, widths) -> np.ndarray:
    """Per-group-width layout of one layer's V codes [kv_heads, ctx, d] with
    widths[g] the width of tokens [32 g, 32 g + 32): uint8 [kv_heads,
    sum_g d * 4 * widths[g]]."""
    c = np.asarray(codes, dtype=np.uint8)
    H, T, d = c.shape
    ng = -(-T // GROUP)
    if len(widths) != ng:
        raise ValueError("one width per 32-token group")
    parts = []
    for g in range(ng):
        tok = c[:, g * GROUP:(g + 1) * GROUP]
        parts.append(pack_pool_v(tok, int(widths[g])).reshape(H, -1))
    return np.concatenate(parts, axis=1)


def unpack_pool_v_groups(packed: np.ndarray, widths, ctx: int, d: int) -> np.ndarray:
    """Inverse of pack_pool_v_groups: codes [kv_heads, ctx, d]."""
    p = np.asarray(packed, dtype=np.uint8)
    H = p.shape[0]
    out, off = [], 0
    for b in widths:
        n = d * 4 * int(b)
        out.append(unpack_pool_v(p[:, off:off + n].reshape(H, 1, d, 4 * int(b)), int(b), GROUP))
        off += n
    if off != p.shape[1]:
        raise ValueError("byte count does not match the widths")
    return np.concatenate(out, axis=1)[:, :ctx]


def encode_layer_groups(K_bf16, V_bf16, widths, k_block: int = 32) -> dict:
    """Everything the pool stores for a layer built from 32-token groups of
    per-group V widths (widths[g] in {2, 3, 4} for tokens [32 g, 32 g + 32)).
    K as in encode_layer (block-scaled by default: the pools that take
    appends); every group's codes and norms are those of its own tokens."""
    V = np.asarray(V_bf16)
    H, T, d = V.shape
    widths = [int(b) for b in widths]
    if len(widths) != -(-T // GROUP):
        raise ValueError("one width per 32-token group")
    codes = np.zeros((H, T, d), dtype=np.uint8)
    norms = np.zeros((H, T), dtype=np.float32)
    for g, b in enumerate(widths):
        sl = slice(g * GROUP, min(T, (g + 1) * GROUP))
        codes[:, sl], norms[:, sl] = v_codes(V[:, sl], b)
    enc = dict(bits=None, widths=widths, codes=codes, norms=norms, packed=pack_pool_v_groups(codes, widths),
               k_block=k_block)
    if k_block:
        if k_block != K_BLOCK:
            raise ValueError("k_block must be 0 or 32")
        sc = k_scales_block(K_bf16)
        enc.update(absmax=F32(0), scale=F32(1), kscales=sc, kq=k_quantize_block(K_bf16, sc))
    else:
        absmax, scale = k_scale(K_bf16)
        enc.update(absmax=absmax, scale=scale, kq=k_quantize(K_bf16, scale))
    return enc


def token_widths(enc: dict, T: int) -> np.ndarray:
    """Width of every token of an encoded layer (int [T])."""
    if enc.get("widths") is None:
        return np.full(T, enc["bits"], dtype=np.int64)
    return np.repeat(np.asarray(enc["widths"], dtype=np.int64), GROUP)[:T]
