// Tensor-core decode attention over the shared pool, one thread per query row
// (sm_103a, tcgen05).
//
// What it computes is the PolyKV summary's per-agent attention over the
// dequantised pool (section 2.A: every agent reads the one pool; section 2.B:
// K = q * s, V = n * H c[codes] / d), plus each agent's private bf16 tail
// (CoMixKV article: recent states stay at native precision), in one softmax.
//
// Work split. One thread-block cluster per (KV head, group of up to 128 query
// rows); its S CTAs split the context. Every query row of every agent that
// shares the KV head is served by one pass over the packed pool bytes, so the
// pool is read once per step no matter how many agents there are.
//
// Per CTA (one per SM, 16 warps), per tile of 128 pool tokens:
//   warp 0 (loader)     TMA load of the tile's int8 K (128-byte swizzle) and
//                       bulk copies of its packed V code groups and norms into
//                       a ring of raw stages.
//   warps 12-15         expand the tile into fp16 MMA operands in shared
//   (expanders)         memory: K^ = int8 K (exact) as [token][channel] and
//                       V^ = lam * c[code] as [channel][token] (one thread per
//                       token for K, per rotated coordinate for V; both in the
//                       canonical 128-byte-swizzled K-major layout), and the
//                       token norms n_t / nref; a ring of operand stages whose
//                       K^ half is released as soon as the tile's S MMA is
//                       done, its V^ half and norms once its P'.V MMAs are.
//   warp 1 (issuer)     S = Q K^T into tensor memory (M = 128 query rows,
//                       N = 128 tokens, Q the A operand in tensor memory),
//                       two S buffers so that S of tile i+1 runs while the
//                       softmax of tile i does; then O += P' V^ with P' the A
//                       operand in tensor memory (M = rows, N = channels,
//                       K = tokens), accumulated in the rotated domain
//                       sum_t p_t n_t c[code_t]; the inverse FWHT runs once
//                       per output row in the epilogue.
//   warps 4-11          softmax, thread = query row (warp w owns tensor-memory
//   (softmax)           lanes 32 (w % 4) ...), two warps per row, one per half
//                       of the tile's columns: the tile's row maximum (the two
//                       halves meet in shared memory), a reference maximum
//                       that moves only when the row maximum passes it by
//                       more than 2^8 (then O and the row sum are rescaled
//                       once the previous P'.V is done), p = 2^(x - m), and
//                       P' = p * n_t / nref split into fp16 hi (top 11
//                       significant bits) and lo (the exact remainder), both
//                       written back over the tile's S columns; the P'.V MMAs
//                       take hi and lo, so P' carries ~22 bits.
//   epilogue            each CTA stages its rows (O row, m, l) in shared
//                       memory and sends the rows of each agent with one bulk
//                       copy into the shared memory of the CTA that owns the
//                       agent; owners merge (log-sum-exp), apply one inverse
//                       FWHT per row, join the agent's bf16 tail and write.
//   tails (instances with TAIL only): the owner CTA computes its agents' tail
//     attention on CUDA cores (all warps) before the main loop, while the first
//     tiles are in flight.
// Every mbarrier wait is bounded; on expiry the kernel records
// KVPOOL_ERR_TIMEOUT in the status word and carries on to its exit without
// waiting again, so a fault never hangs the device.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>

#include "kvpool_internal.cuh"
#include "tc_ptx.cuh"

namespace kvp {
namespace rows {

constexpr int kTile = 128;       // pool tokens per tile
constexpr int kM = 128;          // query rows per CTA (MMA M, tensor-memory lanes)
constexpr int kThreads = 512;    // 16 warps
constexpr int kWarpLoad = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpSm = 4;       // softmax warps 4..11
constexpr int kWarpExp = 12;     // expander warps 12..15
constexpr int kExpThreads = 128;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;
constexpr uint32_t kCols = 512;
constexpr int kMaxCluster = 16;
constexpr float kLazy = 8.0f;    // log2 units the reference maximum may trail the row maximum
constexpr uint32_t kBarTmem = 6; // named barrier: issuer warp + softmax warps (tensor memory address)

struct Params {
    const uint8_t* vcodes;
    const float* vnorm;
    const float* kscale;
    const uint32_t* vnmax;
    int ctx, ctx_pad, Hk;  // ctx: end of the context slice attended (tokens)
    int t0;                // start of the slice, a multiple of kTile
    const uint16_t* Q;
    int Hq, G, R, RW;  // RW: rows per row group (whole agents, <= 128)
    const uint16_t* tK;
    const uint16_t* tV;
    const int32_t* tlen;
    int tail_max;
    float* out;
    float scale_log2;
    int tps;     // tokens per CTA, a multiple of kTile
    int nraw;    // raw stages
    int early;   // 1: the layer's bytes may be read before the grid-dependency wait
    int own;     // merge slots per source CTA (the most rows one CTA owns)
    int* status;
    uint32_t tlo[4], thi[4];  // low / high bytes of fp16 lam * c[k], entry k in byte k % 4 of word k / 4
    float inv_lam;
    float* part_ml;   // partial mode ([nslice][Hk][R][2] and [nslice][Hk][R][D]), else null
    float* part_acc;
    float* ws_tail_ml;  // workspace mode with tails: the rows' tail (m, l), [Hk][R][2] (the
                        // unnormalised tail accumulators go to `out`, as in the cluster path)
    int rgn;          // row groups per KV head
    int nslice;       // context slices per (KV head, row group): blockIdx.z = row group + rgn * slice;
                      // slice s of a cluster of S CTAs covers tokens t0 + (s S + rank) tps ...
    const float* kscales;  // block-scaled K: [Hk][ctx_pad][D/32] (instances with KB), else unused
    // per-group V widths (instances with MIX): the width of each 32-token
    // group, its byte offset within a KV head's codes, the bytes per KV head,
    // and the operand tables of widths 2, 3, 4 under one lam (as tlo / thi)
    const uint8_t* gbits;
    const uint32_t* goff;
    long long vhead;
    uint32_t mlo[3][4], mhi[3][4];
};

// operand stages (block-scaled K^ takes twice the room, leaving one raw stage)
__host__ __device__ constexpr int num_op(bool kb) { return kb ? 2 : 2; }

struct Layout {
    uint32_t op, op_v, op_n;    // operand stage: K^ at 0 (block-scaled: hi, then lo), V^ at op_v, norms at op_n
    uint32_t raw, raw_v, raw_n; // raw stage: int8 K at 0, V codes at raw_v, norms at raw_n
    uint32_t raw0, misc, bars, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// bytes of the staging rows (W rows of D + 4 floats); the merge slots start there
__host__ __device__ inline uint32_t staging_bytes(int D, int W) { return align_up(W * (D + 4) * 4, 1024); }

// misc area: row factor [128], tile maxima [2][2][128], row-sum halves
// [2][128], |q| maxima [2][128], tail (m, l) [128][2], log2 nref (one word,
// padded)
// (block-scaled K: then the column factors sigma_t, [2][128])
constexpr uint32_t kMiscBytes = 128 * 4 * (1 + 4 + 2 + 2 + 2) + 16;
constexpr uint32_t kSigBytes = 2 * 128 * 4;
__host__ __device__ constexpr int kNumBars(int nraw, bool kb) { return 2 * nraw + 4 * num_op(kb) + 7 + (kb ? 4 : 0); }

__host__ __device__ inline Layout make_layout(int D, int bits, int nraw, bool kb) {
    Layout L;
    L.op_v = kTile * D * 2 * (kb ? 2 : 1);
    L.op_n = L.op_v + D * kTile * 2;
    L.op = align_up(L.op_n + kTile * 4, 1024);
    L.raw_v = kTile * D;
    L.raw_n = L.raw_v + kTile * D * bits / 8;
    L.raw = align_up(L.raw_n + kTile * 4, 1024);
    L.raw0 = num_op(kb) * L.op;
    L.misc = L.raw0 + nraw * L.raw;
    L.bars = align_up(L.misc + kMiscBytes + (kb ? kSigBytes : 0), 8);
    L.total = align_up(L.bars + 8 * kNumBars(nraw, kb) + 8, 1024);
    return L;
}

__device__ __forceinline__ float bf2f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// four int8 -> two fp16x2 holding the signed values exactly
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;  // biased by 128
    const uint32_t magic = 0x64646464u;  // fp16 0x64xx = 1024 + xx
    const uint32_t a = ptx::prmt(x, magic, 0x5140);
    const uint32_t b = ptx::prmt(x, magic, 0x7362);
    const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// an fp16x2 pair of int8 values q times r = rh + rl (rh = fp16(r), rl =
// fp16(r - rh)), as fp16x2 hi + lo: hi = fl(q rh); q rh - hi is exact in
// fp16 (a short remainder), so one fused step adds q rl to it; hi + lo
// carries ~21 significant bits of q r (ratios below 2^-14 lose bits to the
// fp16 range: blocks that much smaller than the token's largest)
__device__ __forceinline__ void split_scaled(uint32_t qh2, __half2 rh, __half2 rl, uint32_t& hi, uint32_t& lo) {
    const __half2 q = *reinterpret_cast<const __half2*>(&qh2);
    const __half2 h = __hmul2(q, rh);
    const __half2 e = __hfma2(q, rh, __hneg2(h));  // q rh - hi, exact
    const __half2 l = __hfma2(q, rl, e);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 8 codes of BITS bits (the low 8*BITS bits of x) -> 8 nibbles
template <int BITS>
__device__ __forceinline__ uint32_t spread8(uint32_t x) {
    if constexpr (BITS == 2) {
        uint32_t y = (x & 0xFFu) | ((x & 0xFF00u) << 8);
        y = (y & 0x000F000Fu) | ((y & 0x00F000F0u) << 4);
        return (y & 0x03030303u) | ((y & 0x0C0C0C0Cu) << 2);
    } else if constexpr (BITS == 3) {
        uint32_t y = (x & 0xFFFu) | ((x & 0xFFF000u) << 4);
        y = (y & 0x003F003Fu) | ((y & 0x0FC00FC0u) << 2);
        return (y & 0x07070707u) | ((y & 0x38383838u) << 1);
    } else {
        return x;
    }
}

// 4 codes (nibbles of the low 16 bits of sel) -> two fp16x2 of lam * c[code]
template <int BITS>
__device__ __forceinline__ void lookup4(uint32_t sel, const uint32_t (&tlo)[4], const uint32_t (&thi)[4],
                                        uint32_t& h01, uint32_t& h23) {
    uint32_t L, H;
    if constexpr (BITS <= 3) {
        L = ptx::prmt(tlo[0], tlo[1], sel);
        H = ptx::prmt(thi[0], thi[1], sel);
    } else {
        const uint32_t s3 = sel & 0x7777u;
        const uint32_t La = ptx::prmt(tlo[0], tlo[1], s3), Lb = ptx::prmt(tlo[2], tlo[3], s3);
        const uint32_t Ha = ptx::prmt(thi[0], thi[1], s3), Hb = ptx::prmt(thi[2], thi[3], s3);
        // byte mask of the codes >= 8: the sign-replicate mode of a selector
        // nibble with bit 3 set turns 0x80 into 0xFF
        uint32_t m = ptx::prmt(0x80808080u, 0x80808080u, sel) & 0x7F7F7F7Fu;
        m |= m << 1;
        L = (La & ~m) | (Lb & m);
        H = (Ha & ~m) | (Hb & m);
    }
    h01 = ptx::prmt(L, H, 0x5140);
    h23 = ptx::prmt(L, H, 0x7362);
}

// the 32 codes of one packed sequence (4*BITS bytes at `row`) -> 16 fp16x2,
// token order, the lower token in the low half
template <int BITS>
__device__ __forceinline__ void decode32(const unsigned char* row, const uint32_t (&tlo)[4],
                                         const uint32_t (&thi)[4], uint32_t* h) {
    uint32_t f[4];  // four fields of 8 codes
    if constexpr (BITS == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(row);
        f[0] = w.x; f[1] = w.x >> 16; f[2] = w.y; f[3] = w.y >> 16;
    } else if constexpr (BITS == 3) {
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(row);
        const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
        f[0] = w0; f[1] = __funnelshift_r(w0, w1, 24); f[2] = __funnelshift_r(w1, w2, 16); f[3] = w2 >> 8;
    } else {
        const uint4 w = *reinterpret_cast<const uint4*>(row);
        f[0] = w.x; f[1] = w.y; f[2] = w.z; f[3] = w.w;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t y = spread8<BITS>(f[k]);
        lookup4<BITS>(y, tlo, thi, h[4 * k], h[4 * k + 1]);
        lookup4<BITS>(y >> 16, tlo, thi, h[4 * k + 2], h[4 * k + 3]);
    }
}

// Offset of 16-byte chunk `chunk` (of 8 fp16 along K) of row `row` in a
// K-major operand of 128-byte swizzled K-blocks of 64 elements; `blk` is
// the byte stride between K-blocks (rows x 128).
__device__ __forceinline__ uint32_t kmajor_off(int row, int chunk, uint32_t blk) {
    return (uint32_t)(chunk >> 3) * blk + (uint32_t)(row >> 3) * 1024 + (uint32_t)(row & 7) * 128 +
           ((uint32_t)((chunk & 7) ^ (row & 7)) << 4);
}

// Attention of the owned agents' rows over their private bf16 tails (plain
// CUDA cores, online softmax in log2 units, 256 tokens per chunk). Writes the
// unnormalised accumulator to `out` and (m, l) per row to `tailml`; `stage`
// is 13 KB of shared memory that is free until the main loop. Every thread
// of the CTA calls it (it holds CTA barriers).
template <int D>
__device__ __noinline__ void tail_attention(const Params& p, unsigned char* stage, float* tailml,
                                            int S, int crank, int g, int row0, int nrows) {
    constexpr int TCH = 256;
    constexpr int RPT = kThreads / D;  // P.V phase: row sub-blocks
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    float* tq = reinterpret_cast<float*>(stage);                                // [8][D]
    float* tl = reinterpret_cast<float*>(stage + 8 * D * 4);                   // [8][TCH]
    float* tmx = reinterpret_cast<float*>(stage + 8 * D * 4 + 8 * TCH * 4);    // [8]
    // P.V: VR tail V rows at a time through shared memory (the next block's
    // loads in flight while this one is used), VCH 16-byte chunks per block
    constexpr int VR = 64;
    constexpr int VCH = VR * D / 8;
    constexpr int VPT = VCH / kThreads;  // chunks per thread
    static_assert(VCH % kThreads == 0, "V block chunks per thread");
    uint4* tv = reinterpret_cast<uint4*>(stage + 8 * D * 4 + 8 * TCH * 4 + 64);  // [VR][D] bf16
    const int c = tid % D, sub = tid / D;      // P.V phase: rows k with k % RPT == sub, channel c
    const int t = tid % TCH, k0 = tid / TCH;   // logit phase: token t, rows k0 + 2 * kk
    const int G = p.G;
    for (int ar = crank; ar * G < nrows; ar += S) {
        const int a = row0 / G + ar;
        const int tmax = min(max(p.tlen[a], 0), p.tail_max);
        const long long tbase = ((long long)a * p.Hk + g) * p.tail_max;
        for (int jb = 0; jb < G; jb += 8) {
            const int cnt = min(8, G - jb);
            for (int i = tid; i < 8 * D; i += kThreads) {
                const int k = i / D, cc = i % D;
                tq[k * D + cc] = k < cnt ? bf2f(p.Q[((long long)a * p.Hq + g * G + jb + k) * D + cc]) : 0.f;
            }
            float m_run[8], l_run[8], acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) { m_run[k] = -CUDART_INF_F; l_run[k] = 0.f; acc[k] = 0.f; }
            __syncthreads();
            for (int c0 = 0; c0 < tmax; c0 += TCH) {
                // logits of token t for this thread's rows: each 16-byte chunk of
                // the K row is loaded once and used for every row (per row, the
                // products are summed in channel order)
                float lg[4], dot[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) dot[kk] = 0.f;
                const bool tok_ok = c0 + t < tmax;
                if (tok_ok) {
                    const uint16_t* kr = p.tK + (tbase + c0 + t) * D;
#pragma unroll 2
                    for (int cc = 0; cc < D; cc += 8) {
                        const uint4 u = *reinterpret_cast<const uint4*>(kr + cc);
                        const float kv[8] = {bf2f(u.x & 0xFFFF), bf2f(u.x >> 16), bf2f(u.y & 0xFFFF), bf2f(u.y >> 16),
                                             bf2f(u.z & 0xFFFF), bf2f(u.z >> 16), bf2f(u.w & 0xFFFF), bf2f(u.w >> 16)};
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int k = k0 + 2 * kk;
                            if (k < cnt) {
                                const float* qq = tq + k * D + cc;
#pragma unroll
                                for (int e = 0; e < 8; ++e) dot[kk] = fmaf(qq[e], kv[e], dot[kk]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int k = k0 + 2 * kk;
                    lg[kk] = (tok_ok && k < cnt) ? __fmul_rn(dot[kk], p.scale_log2) : -CUDART_INF_F;
                    tl[k * TCH + t] = lg[kk];
                }
                __syncthreads();
                if (warp < 8) {  // row maximum of the chunk
                    float mx = -CUDART_INF_F;
#pragma unroll
                    for (int i = 0; i < TCH / 32; ++i) mx = fmaxf(mx, tl[warp * TCH + lane + 32 * i]);
#pragma unroll
                    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) tmx[warp] = mx;
                }
                __syncthreads();
                float alpha[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float mn = fmaxf(m_run[k], tmx[k]);
                    alpha[k] = (mn == -CUDART_INF_F) ? 1.f : ptx::ex2(m_run[k] - mn);
                    m_run[k] = mn;
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int k = k0 + 2 * kk;
                    float mk = m_run[0];
#pragma unroll
                    for (int q2 = 1; q2 < 8; ++q2) if (q2 == k) mk = m_run[q2];
                    tl[k * TCH + t] = (lg[kk] == -CUDART_INF_F) ? 0.f : ptx::ex2(lg[kk] - mk);
                }
                __syncthreads();
                {
                    const int n2 = min(TCH, tmax - c0);
                    auto vload = [&](int tb, uint4 (&u)[VPT]) {
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            const int ch = tid + i * kThreads, row = tb + ch / (D / 8);
                            u[i] = make_uint4(0, 0, 0, 0);
                            if (row < n2)
                                u[i] = *reinterpret_cast<const uint4*>(p.tV + (tbase + c0 + row) * D + (ch % (D / 8)) * 8);
                        }
                    };
                    constexpr int KPT = (8 + RPT - 1) / RPT;  // rows of this thread: k % RPT == sub
                    float sacc[KPT], ls[KPT];
#pragma unroll
                    for (int k = 0; k < KPT; ++k) { sacc[k] = 0.f; ls[k] = 0.f; }
                    uint4 nxt[VPT];
                    vload(0, nxt);
                    for (int tb = 0; tb < n2; tb += VR) {
#pragma unroll
                        for (int i = 0; i < VPT; ++i) tv[tid + i * kThreads] = nxt[i];
                        __syncthreads();
                        if (tb + VR < n2) vload(tb + VR, nxt);
                        const uint16_t* tv16 = reinterpret_cast<const uint16_t*>(tv) + c;
                        const int nb = min(VR, n2 - tb);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (k % RPT != sub || k >= cnt) continue;
                            for (int u = 0; u < nb; ++u) {  // token order, as one chain
                                const float pv = tl[k * TCH + tb + u];
                                sacc[k / RPT] = fmaf(pv, bf2f(tv16[u * D]), sacc[k / RPT]);
                                ls[k / RPT] += pv;
                            }
                        }
                        __syncthreads();
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (k % RPT != sub || k >= cnt) continue;
                        acc[k] = acc[k] * alpha[k] + sacc[k / RPT];
                        l_run[k] = l_run[k] * alpha[k] + ls[k / RPT];
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k % RPT != sub || k >= cnt) continue;
                const int rr = ar * G + jb + k;
                p.out[((long long)a * p.Hq + g * G + jb + k) * D + c] = acc[k];
                if (c == 0) {
                    tailml[2 * rr] = m_run[k];
                    tailml[2 * rr + 1] = l_run[k];
                }
            }
            __syncthreads();
        }
    }
}

// log2 of nref, the power of two >= the largest V norm of the layer (P' =
// p * n_t / nref keeps P' within the fp16 range whatever the V magnitude)
__device__ __forceinline__ int nref_log2(const uint32_t* vnmax) {
    const uint32_t nb = *vnmax;
    const int ex = (int)((nb >> 23) & 0xFF);
    if (nb != 0 && ex < 255 && ex > 0) return ex - 127 + ((nb & 0x7FFFFF) != 0 ? 1 : 0);
    return 0;
}

// Partial mode (kvpool_attend_partial), per merged row: the slice's (M, L)
// and its accumulator in the rotated domain, in the units where the output is
// H acc / (D L)
template <int D>
__device__ __forceinline__ void write_partial(const Params& p, int slice, int g, int row, int lane, float M,
                                              float L, const float (&acc)[D / 32], float scale) {
    constexpr int EPL = D / 32;
    const size_t base = ((size_t)slice * p.Hk + g) * p.R + row;
    float* dst = p.part_acc + base * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = acc[e] * scale;
    if (lane == 0) {
        p.part_ml[2 * base] = M;
        p.part_ml[2 * base + 1] = L;
    }
}

// Bounded wait shared by a warp: every lane waits, and the warp takes the
// timeout branch together if any lane gave up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, bool& bad) {
    bool ok = bad || ptx::mbar_wait(bar, parity, kWaitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) bad = true;
    return ok;
}

// SPREAD: row groups of at most 64 rows, each row on two lanes (four
// softmax threads per row, all four lane quarters busy).
// KB: block-scaled K (one scale s_b per 32 channels of a token). The
// expanders write K^ = q * s_b / sigma_t with sigma_t the power of two just
// above the token's largest s_b, as fp16 hi + lo (~21 significant bits), and
// sigma_t into a two-slot ring; S takes both halves (16 MMAs) and the softmax
// scales S column t by sigma_t (exact).
// the 32 codes of a group of width w (one coordinate's sequence at `seq`)
// with the tables of Params::mlo / mhi; w = 0 (a group not written): zeros
__device__ __forceinline__ void decode32_mixed(const unsigned char* seq, int w, const Params& p, uint32_t* h) {
    uint32_t tl[4], th[4];
    if (w == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) { tl[k] = p.mlo[0][k]; th[k] = p.mhi[0][k]; }
        decode32<2>(seq, tl, th, h);
    } else if (w == 3) {
#pragma unroll
        for (int k = 0; k < 4; ++k) { tl[k] = p.mlo[1][k]; th[k] = p.mhi[1][k]; }
        decode32<3>(seq, tl, th, h);
    } else if (w == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) { tl[k] = p.mlo[2][k]; th[k] = p.mhi[2][k]; }
        decode32<4>(seq, tl, th, h);
    } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) h[k] = 0u;
    }
}

// MIX: a block-scaled layer whose 32-token groups have their own V widths
// (at most BITS, which sizes the raw stages); a tile's code bytes are its four
// groups back to back
template <int D, int BITS, bool TAIL, bool SPREAD, bool KB, bool MIX = false>
__global__ void __launch_bounds__(kThreads, 1)
attend_rows_kernel(const __grid_constant__ CUtensorMap kmap, const Params p) {
    constexpr int HC = D / 2;                // O columns per softmax half
    constexpr int VB = D * BITS / 8;         // code bytes per token
    constexpr int GB = D * 4 * BITS;         // bytes per 32-token code group
    constexpr int EPL = D / 32;              // channels per lane in the merge
    constexpr int ROWF = D + 4;              // floats per merge row: O row, m, l, padding
    constexpr uint32_t KBLK = kTile * 128;   // K^: bytes per 64-channel K-block (128 tokens)
    constexpr uint32_t VBLK = D * 128;       // V^: bytes per 64-token K-block (D channels)
    constexpr uint32_t kColO = 0, kColS = 128, kColQ = 384;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = (int)ptx::cluster_size();
    const int crank = (int)ptx::cluster_rank();
    constexpr int kNumOp = num_op(KB);
    const Layout lay = make_layout(D, BITS, p.nraw, KB);
    const int NR = p.nraw;
    float* crow = reinterpret_cast<float*>(sm + lay.misc);       // [128] logit factor per row
    float* pmax = crow + 128;                                     // [2][2][128] tile maxima (parity, half)
    float* psum = pmax + 4 * 128;                                 // [2][128] row-sum halves
    uint32_t* pq = reinterpret_cast<uint32_t*>(psum + 2 * 128);   // [2][128] |q| maxima (bf16 bits)
    float* tailml = reinterpret_cast<float*>(pq + 2 * 128);       // [128][2]
    int* sNref = reinterpret_cast<int*>(tailml + 2 * 128);           // log2 nref, from the expanders
    float* sig = reinterpret_cast<float*>(sm + lay.misc + kMiscBytes);  // KB: [2][128] sigma_t per ring slot
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay.bars);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars(NR, KB));
    const uint32_t b_raw_full = ptx::smem_u32(bars);
    const uint32_t b_raw_empty = b_raw_full + 8 * NR;
    // operand stages: K^ is released once its S MMA is done, V^ and the norms
    // once the tile's P'.V MMAs are
    const uint32_t b_k_full = b_raw_empty + 8 * NR;
    const uint32_t b_k_empty = b_k_full + 8 * kNumOp;
    const uint32_t b_v_full = b_k_empty + 8 * kNumOp;
    const uint32_t b_v_empty = b_v_full + 8 * kNumOp;
    const uint32_t b_q = b_v_empty + 8 * kNumOp;  // Q rows are in tensor memory
    const uint32_t b_s = b_q + 8;                  // [2] S of a tile is in tensor memory
    const uint32_t b_p = b_s + 16;                 // [2] P' of a tile is in tensor memory
    const uint32_t b_o = b_p + 16;                 // a tile's P'.V MMAs are done
    const uint32_t b_fin = b_o + 8;                // every MMA is done
    const uint32_t b_m = b_fin + 8;                // every merge row sent here has landed
    const uint32_t b_sig_full = b_m + 8;           // KB: [2] sigma_t of a tile is written
    const uint32_t b_sig_empty = b_sig_full + 16;  // KB: [2] the softmax is done with the slot
    float* sO = reinterpret_cast<float*>(sm);      // epilogue: staging rows [128][ROWF]
    // one-CTA slices of at most 64 rows (SPREAD) write their partial states
    // straight from the softmax threads' registers, without staging rows
    const bool direct = SPREAD && S == 1 && p.part_acc != nullptr;

    const int g = blockIdx.y;
    const int slice = (int)blockIdx.z / p.rgn;
    const int row0 = ((int)blockIdx.z - slice * p.rgn) * p.RW;
    const int nrows = min(p.RW, p.R - row0);  // a multiple of G
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int t_begin = p.t0 + (slice * S + crank) * p.tps;
    const int t_end = min(p.ctx, t_begin + p.tps);
    const int ntile = (t_end - t_begin + kTile - 1) / kTile;  // >= 1
    const long long head_tok = (long long)g * p.ctx_pad;
    const uint32_t raw_bytes = kTile * D + kTile * VB + kTile * 4;
    const int nag = nrows / p.G;
    const int own_cnt = crank < nag ? ((nag - crank + S - 1) / S) * p.G : 0;

    // MIX: the widths of the four groups of tile i, one per byte (the tile
    // starts at a multiple of 128 tokens, so they are one aligned word)
    auto tile_widths = [&](int i) {
        return __ldg(reinterpret_cast<const uint32_t*>(p.gbits) + (t_begin + i * kTile) / 128);
    };
    auto issue_tile = [&](int i) {
        const int s = i % NR;
        const long long t0 = head_tok + t_begin + (long long)i * kTile;
        const uint32_t dst = ptx::smem_u32(sm + lay.raw0 + s * lay.raw);
        const uint32_t bar = b_raw_full + 8 * s;
        if constexpr (MIX) {
            const uint32_t wd = tile_widths(i);
            const uint32_t nb =
                (uint32_t)D * 4 * ((wd & 0xFFu) + ((wd >> 8) & 0xFFu) + ((wd >> 16) & 0xFFu) + (wd >> 24));
            ptx::mbar_expect_tx(bar, (uint32_t)(kTile * D + kTile * 4) + nb);
            ptx::tma_load_2d(dst, &kmap, 0, (int)t0, bar);
            if (nb)
                ptx::bulk_g2s(dst + lay.raw_v, p.vcodes + g * p.vhead + __ldg(p.goff + (t_begin + i * kTile) / 32),
                              nb, bar);
        } else {
            ptx::mbar_expect_tx(bar, raw_bytes);
            ptx::tma_load_2d(dst, &kmap, 0, (int)t0, bar);
            ptx::bulk_g2s(dst + lay.raw_v, p.vcodes + t0 * VB, kTile * VB, bar);
        }
        ptx::bulk_g2s(dst + lay.raw_n, p.vnorm + t0, kTile * 4, bar);
    };

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int s = 0; s < NR; ++s) {
            ptx::mbar_init(b_raw_full + 8 * s, 1);
            ptx::mbar_init(b_raw_empty + 8 * s, kExpThreads / 32);
        }
        for (int e = 0; e < kNumOp; ++e) {
            ptx::mbar_init(b_k_full + 8 * e, kExpThreads / 32);
            ptx::mbar_init(b_k_empty + 8 * e, 1);
            ptx::mbar_init(b_v_full + 8 * e, kExpThreads / 32);
            ptx::mbar_init(b_v_empty + 8 * e, 1);
        }
        ptx::mbar_init(b_q, 8);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(b_s + 8 * b, 1);
            ptx::mbar_init(b_p + 8 * b, 8);
        }
        ptx::mbar_init(b_o, 1);
        ptx::mbar_init(b_fin, 1);
        ptx::mbar_init(b_m, 1);
        if constexpr (KB) {
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(b_sig_full + 8 * b, kExpThreads / 32);
                ptx::mbar_init(b_sig_empty + 8 * b, 8);
            }
        }
        ptx::mbar_init_fence();
        if (own_cnt > 0) ptx::mbar_expect_tx(b_m, (uint32_t)(S * own_cnt * ROWF * 4));
        ptx::grid_dep_launch();
    }
    __syncthreads();
    // Tensor memory: allocated by the issuer warp and published to the
    // softmax warps only (named barrier kBarTmem), so that the loader and the
    // expanders start at once and the allocation overlaps the Q loads
    auto tmem_publish = [&]() {
        ptx::tc_fence_before();
        ptx::bar_sync(kBarTmem, 32 + 256);
        ptx::tc_fence_after();
        return *tslot;
    };

    // tails of the agents this CTA owns (CUDA cores, every warp), while the
    // first tiles are in flight; the (last) operand stage is free until then
    int first = 0;  // loader: tiles requested before the role loops
    if constexpr (TAIL) {
        // the layer's bytes may be requested before the grid-dependency wait
        // unless the launch before this one wrote them (the tails and Q after it)
        if (tid == 0 && p.early)
            for (; first < min(ntile, NR); ++first) issue_tile(first);
        ptx::grid_dep_wait();
        if (tid == 0)
            for (; first < min(ntile, NR); ++first) issue_tile(first);
        // the agents of this CTA: a mod S == rank in a cluster; a mod nslice
        // == slice for the one-CTA slices of workspace mode
        const bool ws = p.part_acc != nullptr;
        tail_attention<D>(p, sm + (kNumOp == 2 ? lay.op : 0), tailml, ws ? p.nslice : S, ws ? slice : crank, g,
                          row0, nrows);
    }

    bool bad = false;
    uint32_t tmem = 0;  // issuer and softmax warps: base of the 512 tensor-memory columns
    if (warp == kWarpLoad) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            // warm L2 with this CTA's query rows (the G rows of an agent are
            // consecutive): the softmax warps read them after the grid-
            // dependency wait, behind the tile traffic otherwise. A prefetch
            // reads nothing into the kernel; L2 stays coherent with a writer.
            for (int ar = 0; ar * p.G < nrows; ++ar)
                ptx::prefetch_l2(p.Q + ((long long)(row0 / p.G + ar) * p.Hq + g * p.G) * D, p.G * D * 2);
            // the layer's bytes may be read before the grid-dependency wait
            // unless the launch before this one wrote them
            if (!p.early) ptx::grid_dep_wait();
            for (int issued = first; issued < ntile; ++issued) {
                const int s = issued % NR;
                if (issued >= NR) {
                    if (!bad && !ptx::mbar_wait(b_raw_empty + 8 * s, ((issued / NR) - 1) & 1, kWaitNs)) bad = true;
                    ptx::fence_proxy_async();  // the expanders' reads of the stage come first
                }
                issue_tile(issued);
            }
            // every requested tile has landed before the CTA may exit
            for (int i = max(0, ntile - NR); i < ntile; ++i)
                ptx::mbar_wait(b_raw_full + 8 * (i % NR), (i / NR) & 1, kWaitNs);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ issuer
        ptx::tmem_alloc(ptx::smem_u32(tslot), kCols);
        tmem = tmem_publish();
        if (lane == 0) {
            const uint32_t idS = ptx::idesc_f16(kM, kTile, 0, 0);
            const uint32_t idO = ptx::idesc_f16(kM, D, 0, 0);
            const uint32_t op0 = ptx::smem_u32(sm);
            const uint32_t tQ = tmem + kColQ, tO = tmem + kColO;
            if (!bad && !ptx::mbar_wait(b_q, 0, kWaitNs)) bad = true;
            ptx::tc_fence_after();
            auto pv = [&](int j) {  // O += P'_j V^_j, hi then lo per 16 tokens
                const int e = j % kNumOp, b = j & 1;
                if (!bad && !ptx::mbar_wait(b_v_full + 8 * e, (j / kNumOp) & 1, kWaitNs)) bad = true;
                if (!bad && !ptx::mbar_wait(b_p + 8 * b, (j >> 1) & 1, kWaitNs)) bad = true;
                ptx::tc_fence_after();
                const uint32_t tP = tmem + kColS + 128 * b;
                const uint32_t aV = op0 + e * lay.op + lay.op_v;
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    // P' columns: per 32 tokens, 16 columns of hi, then 16 of lo
                    const uint32_t ch = (ks / 2) * 32 + (ks % 2) * 8;
                    const uint64_t bv = ptx::sdesc(aV + (ks / 4) * VBLK + (ks % 4) * 32, 16, 1024);
                    ptx::mma_f16_ta(tO, tP + ch, bv, idO, (j > 0 || ks > 0) ? 1u : 0u);
                    ptx::mma_f16_ta(tO, tP + ch + 16, bv, idO, 1u);
                }
                ptx::mma_commit(b_v_empty + 8 * e);
                ptx::mma_commit(b_o);
            };
            for (int i = 0; i < ntile; ++i) {
                const int e = i % kNumOp, b = i & 1;
                if (!bad && !ptx::mbar_wait(b_k_full + 8 * e, (i / kNumOp) & 1, kWaitNs)) bad = true;
                ptx::tc_fence_after();
                const uint32_t aK = op0 + e * lay.op;
                const uint32_t tS = tmem + kColS + 128 * b;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {  // S_i = Q K^_i^T
                    const uint64_t bk = ptx::sdesc(aK + (ks / 4) * KBLK + (ks % 4) * 32, 16, 1024);
                    ptx::mma_f16_ta(tS, tQ + ks * 8, bk, idS, ks > 0 ? 1u : 0u);
                }
                if constexpr (KB) {
                    // + Q (K^ lo)^T
                    const uint32_t aL = aK + kTile * D * 2;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t bk = ptx::sdesc(aL + (ks / 4) * KBLK + (ks % 4) * 32, 16, 1024);
                        ptx::mma_f16_ta(tS, tQ + ks * 8, bk, idS, 1u);
                    }
                }
                ptx::mma_commit(b_k_empty + 8 * e);
                ptx::mma_commit(b_s + 8 * b);
                if (i > 0) pv(i - 1);
            }
            pv(ntile - 1);
            ptx::mma_commit(b_fin);
            // the last commit covers every MMA issued; waited for even after a
            // timeout, so that no MMA is still running when the CTA moves on
            ptx::mbar_wait(b_fin, 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp >= kWarpExp) {
        // --------------------------------------------------------- expanders
        const int et = tid - kWarpExp * 32;  // 0..127: token for K^, coordinate for V^
        const int nl = nref_log2(p.vnmax);  // read once here, kept for the merge
        if (et == 0) *sNref = nl;
        const float vr = ldexpf(1.0f, -nl);
        uint32_t tlo[4], thi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) { tlo[k] = p.tlo[k]; thi[k] = p.thi[k]; }
        // KB: this token's block scales, one tile ahead (the padding's are 0)
        constexpr int NB = D / 32;
        float scn[NB] = {};
        auto load_scales = [&](int i) {
            const float* src = p.kscales + (head_tok + t_begin + (long long)i * kTile + et) * NB;
            if constexpr (NB == 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(src));
                scn[0] = v.x, scn[1] = v.y, scn[2] = v.z, scn[3] = v.w;
            } else {
                const float2 v = __ldg(reinterpret_cast<const float2*>(src));
                scn[0] = v.x, scn[1] = v.y;
            }
        };
        if constexpr (KB) load_scales(0);
        for (int i = 0; i < ntile; ++i) {
            const int s = i % NR, e = i % kNumOp;
            warp_wait(b_raw_full + 8 * s, (i / NR) & 1, bad);
            if (i >= kNumOp) warp_wait(b_k_empty + 8 * e, ((i / kNumOp) - 1) & 1, bad);
            const unsigned char* raw = sm + lay.raw0 + s * lay.raw;
            unsigned char* opk = sm + e * lay.op;
            unsigned char* opv = opk + lay.op_v;
            float* opn = reinterpret_cast<float*>(opk + lay.op_n);
            // KB: sigma_t = 2^(E + 1) for the largest scale m 2^E (1 if all are 0),
            // r_b = s_b / sigma_t (exact) into the ring slot of the tile
            float rb[NB];
            __half2 rbh[NB], rbl[NB];
            if constexpr (KB) {
                float sc[NB];
                float mx = 0.0f;
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    sc[k] = scn[k];
                    mx = fmaxf(mx, sc[k]);
                }
                if (i + 1 < ntile) load_scales(i + 1);
                int ex = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 126 : 0;  // E + 1
                ex = max(-125, min(127, ex));
                const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    rb[k] = __fmul_rn(sc[k], inv);
                    const __half h = __float2half_rn(rb[k]);
                    rbh[k] = __half2half2(h);
                    rbl[k] = __half2half2(__float2half_rn(rb[k] - __half2float(h)));
                }
                if (i >= 2) warp_wait(b_sig_empty + 8 * (i & 1), ((i >> 1) - 1) & 1, bad);
                sig[(i & 1) * 128 + et] = __uint_as_float((uint32_t)(127 + ex) << 23);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(b_sig_full + 8 * (i & 1));
            }
            // K^: token et, D int8 -> D fp16 (TMA swizzle of the raw row: 128 B
            // for D = 128, 64 B for D = 64); block-scaled: hi and lo of q r_b
            {
                const int t = et;
                const int sw = D == 128 ? (t & 7) : ((t >> 1) & 3);
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(raw + t * D + ((c ^ sw) << 4));
                    uint4 a, b;
                    i8x4_to_h2x2(u.x, a.x, a.y);
                    i8x4_to_h2x2(u.y, a.z, a.w);
                    i8x4_to_h2x2(u.z, b.x, b.y);
                    i8x4_to_h2x2(u.w, b.z, b.w);
                    if constexpr (KB) {
                        const __half2 rh = rbh[c / 2], rl = rbl[c / 2];  // block c / 2 of 32 channels
                        uint4 ah, al, bh, bl;
                        split_scaled(a.x, rh, rl, ah.x, al.x);
                        split_scaled(a.y, rh, rl, ah.y, al.y);
                        split_scaled(a.z, rh, rl, ah.z, al.z);
                        split_scaled(a.w, rh, rl, ah.w, al.w);
                        split_scaled(b.x, rh, rl, bh.x, bl.x);
                        split_scaled(b.y, rh, rl, bh.y, bl.y);
                        split_scaled(b.z, rh, rl, bh.z, bl.z);
                        split_scaled(b.w, rh, rl, bh.w, bl.w);
                        *reinterpret_cast<uint4*>(opk + kmajor_off(t, 2 * c, KBLK)) = ah;
                        *reinterpret_cast<uint4*>(opk + kmajor_off(t, 2 * c + 1, KBLK)) = bh;
                        *reinterpret_cast<uint4*>(opk + kTile * D * 2 + kmajor_off(t, 2 * c, KBLK)) = al;
                        *reinterpret_cast<uint4*>(opk + kTile * D * 2 + kmajor_off(t, 2 * c + 1, KBLK)) = bl;
                    } else {
                        *reinterpret_cast<uint4*>(opk + kmajor_off(t, 2 * c, KBLK)) = a;
                        *reinterpret_cast<uint4*>(opk + kmajor_off(t, 2 * c + 1, KBLK)) = b;
                    }
                }
            }
            ptx::fence_proxy_async();  // the MMAs read the operands through the async proxy
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_k_full + 8 * e);
            if (i >= kNumOp) warp_wait(b_v_empty + 8 * e, ((i / kNumOp) - 1) & 1, bad);
            // V^: coordinate c, the tile's 4 groups of 32 tokens (D = 64: two
            // threads per coordinate, two groups each)
            {
                constexpr int GPT = 4 * D / kExpThreads;  // groups per thread
                const int c = et % D, g0 = (et / D) * GPT;
                const uint32_t wd = MIX ? tile_widths(i) : 0u;
#pragma unroll
                for (int gg = 0; gg < GPT; ++gg) {
                    const int gi = g0 + gg;
                    uint32_t h[16];
                    if constexpr (MIX) {
                        // group gi's width (warp-uniform) and the bytes of the groups before it
                        const int w = (int)((wd >> (8 * gi)) & 0xFFu);
                        const uint32_t below = gi == 0 ? 0u : (wd & (0xFFFFFFFFu >> (32 - 8 * gi)));
                        const uint32_t nbelow = (below & 0xFFu) + ((below >> 8) & 0xFFu) + ((below >> 16) & 0xFFu);
                        decode32_mixed(raw + lay.raw_v + nbelow * (D * 4) + c * (4 * w), w, p, h);
                    } else {
                        decode32<BITS>(raw + lay.raw_v + gi * GB + c * (4 * BITS), tlo, thi, h);
                    }
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        *reinterpret_cast<uint4*>(opv + kmajor_off(c, gi * 4 + m, VBLK)) =
                            make_uint4(h[4 * m], h[4 * m + 1], h[4 * m + 2], h[4 * m + 3]);
                }
            }
            // norms n_t / nref, 0 past the split (their p is 0 too)
            {
                const int tok = t_begin + i * kTile + et;
                opn[et] = tok < t_end ? reinterpret_cast<const float*>(raw + lay.raw_n)[et] * vr : 0.f;
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(b_v_full + 8 * e);
                ptx::mbar_arrive(b_raw_empty + 8 * s);
            }
        }
    } else if (warp >= kWarpSm) {
        // ----------------------------------------------------------- softmax
        const int sg = (warp - kWarpSm) / 4;  // column half: tokens [64 sg, 64 sg + 64) of a tile
        const int q = warp & 3;               // tensor-memory lane quarter
        const int tl = q * 32 + lane;         // this thread's tensor-memory lane
        // the lane's query row: lane = row, or (SPREAD) row r at lane
        // 32 (r % 4) + r / 4 and again 16 lanes up, the two copies taking one
        // 32-token chunk each of the warp's 64 tokens (tensor-memory accesses
        // take one column address for the whole warp: both copies address
        // both chunks, and each uses or fills its own)
        const int dup = SPREAD ? (lane >> 4) : 0;
        const int r = SPREAD ? ((lane & 15) * 4 + q) : tl;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // a pair of warps whose 32 rows are all past the CTA's rows has no
        // work: it only keeps the barriers' counts (its lanes of S, P' and O
        // are never read; an MMA row depends on its own lane only)
        const bool act = SPREAD || q * 32 < nrows;
        if constexpr (!TAIL) ptx::grid_dep_wait();
        if (!act) {
            // keep the counts of the Q, S and P' barriers, tile by tile
            tmem = tmem_publish();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_q);
            for (int i = 0; i < ntile; ++i) {
                warp_wait(b_s + 8 * (i & 1), (i >> 1) & 1, bad);
                if (lane == 0) ptx::mbar_arrive(b_p + 8 * (i & 1));
                if constexpr (KB)
                    if (lane == 0) ptx::mbar_arrive(b_sig_empty + 8 * (i & 1));
            }
        } else {
            // Q row r -> fp16 in tensor memory (the A operand of S), scaled by the
            // power of two that puts its largest |q| in [2^14, 2^15) (exact); the
            // row's logit factor undoes it
            {
                constexpr int NQ = HC / 8;  // 16-byte chunks of the half row
                uint4 qv[NQ];
                uint32_t am = 0;
                const bool live = r < nrows;
                const int a = (row0 + r) / p.G, j = (row0 + r) % p.G;
                const uint16_t* qsrc = p.Q + ((long long)a * p.Hq + g * p.G + j) * D + sg * HC;
#pragma unroll
                for (int k = 0; k < NQ; ++k) {
                    qv[k] = live ? reinterpret_cast<const uint4*>(qsrc)[k] : make_uint4(0, 0, 0, 0);
                    const uint32_t m7 = 0x7FFF7FFFu;
                    am = __vmaxu2(am, __vmaxu2(__vmaxu2(qv[k].x & m7, qv[k].y & m7), __vmaxu2(qv[k].z & m7, qv[k].w & m7)));
                }
                pq[sg * 128 + tl] = max(am & 0xFFFFu, am >> 16);
                ptx::bar_sync(1 + q, 64);
                const uint32_t qmax = max(pq[tl], pq[128 + tl]);
                int qe = 0;
                if (qmax != 0 && qmax < 0x7F80u) qe = 14 - ((int)((qmax >> 7) & 0xFF) - 127);
                qe = max(-100, min(100, qe));
                const float qmul = ldexpf(1.0f, qe);
                tmem = tmem_publish();
                uint32_t w[HC / 2];
#pragma unroll
                for (int k = 0; k < NQ; ++k) {
                    const uint4 u = qv[k];
                    w[4 * k + 0] = pack_h2(bf2f(u.x & 0xFFFF) * qmul, bf2f(u.x >> 16) * qmul);
                    w[4 * k + 1] = pack_h2(bf2f(u.y & 0xFFFF) * qmul, bf2f(u.y >> 16) * qmul);
                    w[4 * k + 2] = pack_h2(bf2f(u.z & 0xFFFF) * qmul, bf2f(u.z >> 16) * qmul);
                    w[4 * k + 3] = pack_h2(bf2f(u.w & 0xFFFF) * qmul, bf2f(u.w >> 16) * qmul);
                }
                if constexpr (HC / 2 == 32) ptx::tmem_st32x(tmem + kColQ + lane_off + sg * 32, w);
                else ptx::tmem_st16(tmem + kColQ + lane_off + sg * 16, w);
                // rows past the CTA's rows (Q = 0, so S = 0) take factor 1: finite p
                if (sg == 0) crow[tl] = live ? p.scale_log2 * (*p.kscale) * ldexpf(1.0f, -qe) : 1.f;
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_q);
            ptx::bar_sync(1 + q, 64);  // crow published to the other half
            const float cr = crow[tl];
            // Row state: the reference s_ref in units of S and m_ref = fl(s_ref *
            // cr) in log2 units. p = 2^((s - s_ref) * cr): s - s_ref is exact for
            // the terms that matter and <= 0 once the reference has moved to the
            // maximum (a form that no fused multiply-add can push above it)
            float s_ref = -CUDART_INF_F, m_ref = -CUDART_INF_F, l = 0.f;
            for (int i = 0; i < ntile; ++i) {
                const int b = i & 1, e = i % kNumOp;
                warp_wait(b_s + 8 * b, (i >> 1) & 1, bad);
                ptx::tc_fence_after();
                const uint32_t tS = tmem + kColS + 128 * b + lane_off;
                const int nval = t_end - (t_begin + i * kTile);  // valid tokens of the tile
                if constexpr (KB) warp_wait(b_sig_full + 8 * (i & 1), (i >> 1) & 1, bad);
                // chunk ch (32 tokens) of S as loaded for this lane, finished in
                // place (block-scaled: column t times sigma_t; tokens past the
                // split at -inf)
                auto fix_s = [&](int ch, uint32_t (&u)[32]) {
                    if constexpr (KB) {
                        const float4* s4 = reinterpret_cast<const float4*>(sig + (i & 1) * 128 + 32 * ch);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            const float4 f = s4[k4];
                            u[4 * k4 + 0] = __float_as_uint(__uint_as_float(u[4 * k4 + 0]) * f.x);
                            u[4 * k4 + 1] = __float_as_uint(__uint_as_float(u[4 * k4 + 1]) * f.y);
                            u[4 * k4 + 2] = __float_as_uint(__uint_as_float(u[4 * k4 + 2]) * f.z);
                            u[4 * k4 + 3] = __float_as_uint(__uint_as_float(u[4 * k4 + 3]) * f.w);
                        }
                    }
                    if (nval < 32 * ch + 32) {  // the same in every thread
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (32 * ch + k >= nval) u[k] = __float_as_uint(-CUDART_INF_F);
                    }
                };
                auto load_s = [&](int ch, uint32_t (&u)[32]) {
                    ptx::tmem_ld32(tS + 32 * ch, u);
                    ptx::tmem_wait_ld();
                    fix_s(ch, u);
                };
                // SPREAD: this lane's own chunk, kept from the max pass for P'
                uint32_t uown[SPREAD ? 32 : 1];
                float smax = -CUDART_INF_F;
                // three-input maxima: 16 instructions for 32 values and smax
                auto chunk_max = [&](const uint32_t (&u)[32]) {
                    auto f = [&](int k) { return __uint_as_float(u[k]); };
                    float mm[11];
#pragma unroll
                    for (int k = 0; k < 10; ++k) mm[k] = ptx::max3(f(3 * k), f(3 * k + 1), f(3 * k + 2));
                    mm[10] = ptx::max3(f(30), f(31), smax);
                    const float a = ptx::max3(mm[0], mm[1], mm[2]), b = ptx::max3(mm[3], mm[4], mm[5]);
                    const float c = ptx::max3(mm[6], mm[7], mm[8]);
                    smax = ptx::max3(ptx::max3(a, b, c), mm[9], mm[10]);
                };
                if constexpr (SPREAD) {
                    // both chunks of the half under one wait; the lane keeps its own
                    uint32_t u0[32], u1[32];
                    ptx::tmem_ld32(tS + 32 * (2 * sg), u0);
                    ptx::tmem_ld32(tS + 32 * (2 * sg + 1), u1);
                    ptx::tmem_wait_ld();
                    fix_s(2 * sg, u0);
                    fix_s(2 * sg + 1, u1);
                    chunk_max(u0);
                    chunk_max(u1);
#pragma unroll
                    for (int k = 0; k < 32; ++k) uown[k] = dup ? u1[k] : u0[k];
                } else {
                    // both chunks of the half under one wait (read again for P')
                    uint32_t u0[32], u1[32];
                    ptx::tmem_ld32(tS + 32 * (2 * sg), u0);
                    ptx::tmem_ld32(tS + 32 * (2 * sg + 1), u1);
                    ptx::tmem_wait_ld();
                    fix_s(2 * sg, u0);
                    fix_s(2 * sg + 1, u1);
                    chunk_max(u0);
                    chunk_max(u1);
                }
                pmax[(b * 2 + sg) * 128 + tl] = smax;
                ptx::bar_sync(1 + q, 64);  // both halves read S; their maxima are published
                const float st = fmaxf(pmax[(b * 2) * 128 + tl], pmax[(b * 2 + 1) * 128 + tl]);
                const float mt = __fmul_rn(st, cr);
                // the reference moves when the tile's maximum passes it by more
                // than kLazy in log2 units (always on the first tile)
                const bool move = (i == 0) || (mt > m_ref + kLazy);
                if (__any_sync(0xffffffffu, move && i > 0)) {
                    // O and l in the old reference: wait for the previous P'.V
                    warp_wait(b_o, (i - 1) & 1, bad);
                    ptx::tc_fence_after();
                    const float alpha = move ? ptx::ex2(m_ref - mt) : 1.0f;
#pragma unroll
                    for (int c0 = 0; c0 < HC; c0 += 32) {
                        if constexpr (HC >= 32) {
                            uint32_t ov[32];
                            ptx::tmem_ld32(tmem + kColO + lane_off + sg * HC + c0, ov);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
                            ptx::tmem_st32x(tmem + kColO + lane_off + sg * HC + c0, ov);
                        }
                    }
                    ptx::tmem_wait_st();
                    l *= alpha;
                }
                if (move) {
                    s_ref = st;
                    m_ref = mt;
                }
                // the tile's norms come with V^
                warp_wait(b_v_full + 8 * e, (i / kNumOp) & 1, bad);
                // P' = p * n_t / nref as fp16 hi + lo over the chunk's own S
                // columns: hi in the first 16 columns, lo in the next 16
                const float4* nn4 = reinterpret_cast<const float4*>(sm + e * lay.op + lay.op_n);
                // While every row of the warp has |m_ref| <= 2^10 the exponent is
                // one fused s * cr - m_ref (the product exact, one rounding):
                // m_ref = fl(s_ref * cr) is then within 2^-14 of s_ref * cr, a
                // factor within 2^(+-2^-14) common to the row's weights under
                // that reference, and p stays below 2^(kLazy + 2^-13). Larger
                // logits take the difference s - s_ref first (in place, `shift`)
                // and then fl((s - s_ref) * cr + 0).
                const bool fused = __all_sync(0xffffffffu, fabsf(m_ref) <= 1024.f);
                const float2 c2 = make_float2(cr, cr);
                const float2 nm = fused ? make_float2(-m_ref, -m_ref) : make_float2(0.f, 0.f);
                auto shift = [&](uint32_t (&u)[32]) {
                    if (!fused) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__fsub_rn(__uint_as_float(u[k]), s_ref));
                    }
                };
                float2 l2 = make_float2(0.f, 0.f);
                // P' of one 32-token chunk of S (this lane's S row), packed hi / lo
                auto form = [&](int ch, const uint32_t (&u)[32], uint32_t (&hw)[16], uint32_t (&lw)[16]) {
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4) {
                        const float4 nn = nn4[ch * 8 + k4];
#pragma unroll
                        for (int w2 = 0; w2 < 2; ++w2) {
                            const int k = k4 * 2 + w2;  // token pair (2k, 2k + 1) of the chunk
                            const float2 sv = make_float2(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1]));
                            const float2 d = __ffma2_rn(sv, c2, nm);
                            const float2 pv = make_float2(ptx::ex2(d.x), ptx::ex2(d.y));  // -inf -> 0
                            l2 = __fadd2_rn(l2, pv);
                            const float2 pp = __fmul2_rn(pv, w2 ? make_float2(nn.z, nn.w) : make_float2(nn.x, nn.y));
                            // hi: 11 significant bits; lo: the exact remainder
                            const float2 hi = make_float2(__uint_as_float(__float_as_uint(pp.x) & 0xFFFFE000u),
                                                          __uint_as_float(__float_as_uint(pp.y) & 0xFFFFE000u));
                            const float2 lo = __fadd2_rn(pp, make_float2(-hi.x, -hi.y));
                            hw[k] = pack_h2(hi.x, hi.y);
                            lw[k] = pack_h2(lo.x, lo.y);
                        }
                    }
                };
                if constexpr (!SPREAD) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int ch = 2 * sg + c;
                        uint32_t u[32], hw[16], lw[16];
                        load_s(ch, u);  // this chunk's own columns: nothing of it was overwritten yet
                        shift(u);
                        form(ch, u, hw, lw);
                        ptx::tmem_st16(tS + 32 * ch, hw);
                        ptx::tmem_st16(tS + 32 * ch + 16, lw);
                    }
                } else {
                    // lanes 0-15 take chunk 2 sg, lanes 16-31 chunk 2 sg + 1; each
                    // lane writes zeros over the other chunk of its row copy
                    uint32_t hw[16], lw[16];
                    shift(uown);
                    form(2 * sg + dup, uown, hw, lw);
                    uint32_t a[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) a[k] = dup ? 0u : hw[k];
                    ptx::tmem_st16(tS + 64 * sg, a);
#pragma unroll
                    for (int k = 0; k < 16; ++k) a[k] = dup ? 0u : lw[k];
                    ptx::tmem_st16(tS + 64 * sg + 16, a);
#pragma unroll
                    for (int k = 0; k < 16; ++k) a[k] = dup ? hw[k] : 0u;
                    ptx::tmem_st16(tS + 64 * sg + 32, a);
#pragma unroll
                    for (int k = 0; k < 16; ++k) a[k] = dup ? lw[k] : 0u;
                    ptx::tmem_st16(tS + 64 * sg + 48, a);
                }
                l += l2.x + l2.y;
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(b_p + 8 * b);
                if constexpr (KB)
                    if (lane == 0) ptx::mbar_arrive(b_sig_empty + 8 * b);
            }
            // every MMA is done, so no stage is read any more: this half of the
            // row's O goes straight into the staging rows (SPREAD: the sum of
            // the row's two lanes), then (m, l) of the row
            warp_wait(b_fin, 0, bad);
            ptx::tc_fence_after();
            if constexpr (SPREAD) l += __shfl_xor_sync(0xffffffffu, l, 16);
            psum[sg * 128 + tl] = l;
            const bool stage = dup == 0 && r < nrows;
            // the half row's columns, every 32-column read under one wait
            constexpr int NO = HC >= 32 ? HC / 32 : 1;
            uint32_t uo[NO][32];
            if constexpr (HC >= 32) {
#pragma unroll
                for (int c = 0; c < NO; ++c) ptx::tmem_ld32(tmem + kColO + lane_off + sg * HC + 32 * c, uo[c]);
                ptx::tmem_wait_ld();
            }
#pragma unroll
            for (int c0 = 0; c0 < HC; c0 += 32) {
                if constexpr (HC >= 32) {
                    uint32_t (&u)[32] = uo[c0 / 32];
                    if constexpr (SPREAD) {
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            u[k] = __float_as_uint(__uint_as_float(u[k]) +
                                                   __uint_as_float(__shfl_xor_sync(0xffffffffu, u[k], 16)));
                    }
                    if (stage && direct) {
                        // the slice's accumulator row, in the units of
                        // write_partial (scale 2^nref / lam)
                        const float sc = ldexpf(1.0f, *sNref) * p.inv_lam;
                        float* dst = p.part_acc + (((size_t)slice * p.Hk + g) * p.R + row0 + r) * D + sg * HC + c0;
#pragma unroll
                        for (int c4 = 0; c4 < 32; c4 += 4)
                            *reinterpret_cast<float4*>(dst + c4) =
                                make_float4(__uint_as_float(u[c4]) * sc, __uint_as_float(u[c4 + 1]) * sc,
                                            __uint_as_float(u[c4 + 2]) * sc, __uint_as_float(u[c4 + 3]) * sc);
                    } else if (stage) {
                        float* dst = sO + r * ROWF + sg * HC + c0;
#pragma unroll
                        for (int c4 = 0; c4 < 32; c4 += 4)
                            *reinterpret_cast<uint4*>(dst + c4) = make_uint4(u[c4], u[c4 + 1], u[c4 + 2], u[c4 + 3]);
                    }
                }
            }
            ptx::bar_sync(1 + q, 64);  // both halves' row sums
            if (sg == 0 && stage && direct) {
                const float lt = psum[tl] + psum[128 + tl];
                const size_t base = ((size_t)slice * p.Hk + g) * p.R + row0 + r;
                p.part_ml[2 * base] = lt > 0.f ? m_ref : -CUDART_INF_F;
                p.part_ml[2 * base + 1] = lt;
            } else if (sg == 0 && stage) {
                sO[r * ROWF + D] = m_ref;
                sO[r * ROWF + D + 1] = psum[tl] + psum[128 + tl];
            }
        }
    }
    if (bad) atomicOr(p.status, kStTimeout);

    // one CTA per context slice (workspace mode): the staged rows are the
    // slice's partial states, written without a cluster merge (SPREAD: the
    // softmax threads have written them already)
    if (S == 1 && p.part_acc != nullptr) {
        ptx::tc_fence_before();  // the tensor-memory reads of O come before its release
        __syncthreads();
        const float oscale = ldexpf(1.0f, *sNref) / (float)D * p.inv_lam;
        for (int rr = warp; !direct && rr < nrows; rr += kThreads / 32) {
            const float* src = sO + rr * ROWF;
            const float m = src[D], l = src[D + 1];
            float acc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = l > 0.f ? src[lane * EPL + e] : 0.f;
            write_partial<D>(p, slice, g, row0 + rr, lane, l > 0.f ? m : -CUDART_INF_F, l, acc, oscale * (float)D);
        }
        if constexpr (TAIL) {  // the tails of this CTA's agents, for the merge kernel
            for (int rr = tid; rr < nrows; rr += kThreads)
                if ((rr / p.G) % p.nslice == slice)
                    *reinterpret_cast<float2*>(p.ws_tail_ml + 2 * ((size_t)g * p.R + row0 + rr)) =
                        make_float2(tailml[2 * rr], tailml[2 * rr + 1]);
        }
        if (warp == kWarpMma) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(tmem, kCols);
        }
        return;
    }

    // this CTA is done with its stages (and has read O out of tensor memory):
    // other CTAs may write merge slots here once every CTA of the cluster has
    // arrived
    ptx::fence_proxy_async();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_arrive();

    // send the G rows of each agent, consecutive here and at the owner of the
    // agent (agent ar -> CTA ar % S, slots from (ar / S) * G), with one copy
    float* slots = reinterpret_cast<float*>(sm + staging_bytes(D, kM));  // [S][own][ROWF]
    const int nsend = nrows / p.G;  // row groups hold whole agents
    ptx::cluster_wait();
    if (tid < nsend) {
        const uint32_t owner = (uint32_t)(tid % S);
        const float* dst = slots + (size_t)(crank * p.own + (tid / S) * p.G) * ROWF;
        ptx::bulk_s2cluster(ptx::dsmem_addr(dst, owner), ptx::smem_u32(sO + tid * p.G * ROWF),
                            (uint32_t)(p.G * ROWF * 4), ptx::dsmem_addr(bars + (b_m - b_raw_full) / 8, owner));
        ptx::bulk_commit();
    }

    // merge the owned rows once all S copies of each have landed, one warp per row
    if (own_cnt > 0) {
        const bool late = tid == 0 && !ptx::mbar_wait(b_m, 0, kWaitNs);
        const bool ok = !__syncthreads_or(late);
        if (late) atomicOr(p.status, kStTimeout);
        const int G = p.G;
        const float oscale = ldexpf(1.0f, *sNref) / (float)D * p.inv_lam;
        for (int loc = warp; ok && loc < own_cnt; loc += kThreads / 32) {
            const int ar = (loc / G) * S + crank, j = loc % G;
            const int rr = ar * G + j;
            const int a = row0 / G + ar;
            // lane s < S holds source s's (m, l); the row's maximum, the
            // weights and the row sum by shuffles; the partial rows are read
            // without branches (sources past S read source S - 1 at weight 0)
            float ms = -CUDART_INF_F, ls = 0.f;
            if (lane < S) {
                const float2 ml = *reinterpret_cast<const float2*>(slots + (size_t)(lane * p.own + loc) * ROWF + D);
                ms = ml.x;
                ls = ml.y;
            }
            float M = ls > 0.f ? ms : -CUDART_INF_F;
#pragma unroll
            for (int o2 = 16; o2; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
            const float w = ls > 0.f ? ptx::ex2(ms - M) : 0.f;
            float L = w * ls;
#pragma unroll
            for (int o2 = 16; o2; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
            float acc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxCluster; ++s) {
                const float ws = __shfl_sync(0xffffffffu, w, s);
                const float* src = slots + (size_t)(min(s, S - 1) * p.own + loc) * ROWF + lane * EPL;
                if constexpr (EPL == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(src);
                    acc[0] = fmaf(ws, v.x, acc[0]); acc[1] = fmaf(ws, v.y, acc[1]);
                    acc[2] = fmaf(ws, v.z, acc[2]); acc[3] = fmaf(ws, v.w, acc[3]);
                } else {
                    const float2 v = *reinterpret_cast<const float2*>(src);
                    acc[0] = fmaf(ws, v.x, acc[0]); acc[1] = fmaf(ws, v.y, acc[1]);
                }
            }
            if (p.part_acc != nullptr) {  // partial mode: the slice's state, no rotation, no tail
                write_partial<D>(p, slice, g, row0 + rr, lane, M, L, acc, oscale * (float)D);
                continue;
            }
            // inverse rotation H acc; lane holds EPL consecutive channels
#pragma unroll
            for (int h = 1; h < EPL; h <<= 1) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    if (!(e & h)) {
                        const float u = acc[e], v = acc[e + h];
                        acc[e] = u + v;
                        acc[e + h] = u - v;
                    }
                }
            }
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const bool upper = (lane & o2) != 0;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, acc[e], o2);
                    acc[e] = upper ? other - acc[e] : acc[e] + other;
                }
            }
            float mt = -CUDART_INF_F, lt = 0.f;
            float* orow = p.out + ((long long)a * p.Hq + g * G + j) * D + lane * EPL;
            float tacc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) tacc[e] = 0.f;
            if (TAIL) {
                mt = tailml[2 * rr];
                lt = tailml[2 * rr + 1];
                if (lt > 0.f) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) tacc[e] = orow[e];
                }
            }
            const float Mf = fmaxf(M, mt);
            const float wp = (L > 0.f) ? ptx::ex2(M - Mf) : 0.f;
            const float wt = (lt > 0.f) ? ptx::ex2(mt - Mf) : 0.f;
            const float inv = 1.0f / (L * wp + lt * wt);
#pragma unroll
            for (int e = 0; e < EPL; ++e) orow[e] = (acc[e] * oscale * wp + tacc[e] * wt) * inv;
        }
    }
    if (tid < nsend) ptx::bulk_wait_read();  // the staging rows may be released
    // tensor memory is released last, off the path to the sends and the merge
    if (warp == kWarpMma) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
}

// ------------------------------------------------------------------ launch

template <int D, int BITS, bool TAIL, bool SPREAD, bool KB, bool MIX>
void configure() {
    static bool done = false;
    if (done) return;
    auto kern = attend_rows_kernel<D, BITS, TAIL, SPREAD, KB, MIX>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    done = true;
}

// How many clusters of S CTAs with `smem` bytes each can be resident at once.
template <int D, int BITS, bool TAIL, bool SPREAD, bool KB, bool MIX>
int max_clusters(int S, size_t smem) {
    static int cache[kMaxCluster + 1][2] = {};  // [S] -> (smem key / 1024 + 1, count)
    const int key = (int)(smem / 1024) + 1;
    if (cache[S][0] == key) return cache[S][1];
    configure<D, BITS, TAIL, SPREAD, KB, MIX>();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attend_rows_kernel<D, BITS, TAIL, SPREAD, KB, MIX>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[S][0] = key;
    cache[S][1] = n;
    return n;
}

// ws_ctas > 0: workspace mode (partial results of many context slices, one
// CTA each, at most ws_ctas CTAs in all); *nslice gets the slices per
// (KV head, row group). ws_ctas = 0: clusters merge the whole slice
// [t0, ctx) in distributed shared memory.
template <int D, int BITS, bool TAIL, bool SPREAD, bool KB, bool MIX>
cudaError_t launch_cfg(const CUtensorMap& kmap, Params prm, int ntiles, int Hk, int RGN, int ws_ctas,
                       int nslice_max, int* nslice, cudaStream_t st) {
    configure<D, BITS, TAIL, SPREAD, KB, MIX>();
    constexpr uint32_t kMaxSmem = 227 * 1024;
    const int rows_cta = std::min(prm.RW, prm.R);
    const int agents_cta = rows_cta / prm.G;
    const int clusters = Hk * RGN;
    // raw stages: as many as fit (up to 3)
    int max_nr = 3;
    while (max_nr > 1 && make_layout(D, BITS, max_nr, KB).total + 1024 > kMaxSmem) --max_nr;
    if (make_layout(D, BITS, max_nr, KB).total + 1024 > kMaxSmem) return cudaErrorInvalidConfiguration;
    prm.rgn = RGN;
    prm.nslice = 1;
    if (ws_ctas > 0) {
        // tiles per CTA: the fewest for which every slice fits in one wave
        const long long jobs = (long long)Hk * RGN;
        if (jobs > ws_ctas) return cudaErrorInvalidValue;
        if (nslice_max < 1) return cudaErrorInvalidValue;
        int per = (int)std::max(1LL, (jobs * ntiles + ws_ctas - 1) / ws_ctas);
        while (jobs * ((ntiles + per - 1) / per) > ws_ctas || (ntiles + per - 1) / per > nslice_max) ++per;
        prm.nslice = (ntiles + per - 1) / per;
        prm.tps = per * kTile;
        prm.own = agents_cta * prm.G;
        prm.nraw = std::min(max_nr, per);
        const Layout lay = make_layout(D, BITS, prm.nraw, KB);
        if (staging_bytes(D, kM) + (size_t)prm.own * (D + 4) * 4 > lay.misc) return cudaErrorInvalidConfiguration;
        if (max_clusters<D, BITS, TAIL, SPREAD, KB, MIX>(1, lay.total + 1024) < 1)
            return cudaErrorInvalidConfiguration;
        *nslice = prm.nslice;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, Hk, RGN * prm.nslice);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = lay.total + 1024;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, attend_rows_kernel<D, BITS, TAIL, SPREAD, KB, MIX>, kmap, prm);
    }
    // cluster size: fewest (waves x tiles per CTA), then the larger cluster;
    // the staging rows and the merge slots must fit in the stage area
    int bestS = 0;
    long long best = -1;
    for (int S = 1; S <= kMaxCluster && S <= ntiles; ++S) {
        const int per = (ntiles + S - 1) / S;
        const int own = (agents_cta + S - 1) / S * prm.G;
        const Layout lay = make_layout(D, BITS, std::min(max_nr, per), KB);
        if (staging_bytes(D, kM) + (size_t)S * own * (D + 4) * 4 > lay.misc) continue;
        const size_t smem = lay.total + 1024;
        const int n = max_clusters<D, BITS, TAIL, SPREAD, KB, MIX>(S, smem);
        if (n < 1) continue;
        const long long waves = (clusters + n - 1) / n;
        const long long cost = waves * per;
        if (best < 0 || cost <= best) {
            best = cost;
            bestS = S;
        }
    }
    if (bestS == 0) return cudaErrorInvalidConfiguration;
    const int per = (ntiles + bestS - 1) / bestS;
    const int S = (ntiles + per - 1) / per;  // never more CTAs than needed for `per` tiles each
    prm.tps = per * kTile;
    prm.own = (agents_cta + S - 1) / S * prm.G;
    prm.nraw = std::min(max_nr, per);
    const Layout lay = make_layout(D, BITS, prm.nraw, KB);
    if (staging_bytes(D, kM) + (size_t)S * prm.own * (D + 4) * 4 > lay.misc) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, Hk, RGN);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = lay.total + 1024;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, attend_rows_kernel<D, BITS, TAIL, SPREAD, KB, MIX>, kmap, prm);
}

}  // namespace rows

// Launch for layers whose V codes have BITS bits (MIX: block-scaled layers
// whose groups have their own widths, BITS the largest).
template <int BITS, bool MIX>
cudaError_t launch_attend_rows_bits(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                                    cudaStream_t st) {
    using namespace rows;
    const int D = s.head_dim;
    // row groups of up to 128 rows hold whole agents; at most 64 rows in all
    // take the spread layout
    const bool spread = a.rows <= 64;
    const int RW = ((spread ? 64 : kM) / a.group) * a.group;
    if (RW < 1) return cudaErrorInvalidValue;
    const int RGN = (a.rows + RW - 1) / RW;
    const int ntiles = (a.t1 - a.t0 + kTile - 1) / kTile;
    Params prm = {};
    prm.vcodes = L.vcodes;
    prm.vnorm = L.vnorm;
    prm.kscale = L.kscale;
    prm.vnmax = L.vnmax;
    prm.ctx = a.t1;
    prm.t0 = a.t0;
    prm.part_ml = a.part_ml;
    prm.part_acc = a.part_acc;
    prm.ws_tail_ml = a.ws_tail_ml;
    prm.ctx_pad = s.ctx_pad;
    prm.Hk = s.kv_heads;
    prm.Q = (const uint16_t*)a.Q;
    prm.Hq = a.q_heads;
    prm.G = a.group;
    prm.R = a.rows;
    prm.RW = RW;
    prm.tK = (const uint16_t*)a.tailK;
    prm.tV = (const uint16_t*)a.tailV;
    prm.tlen = a.tail_len;
    prm.tail_max = a.tail_max;
    prm.out = a.out;
    prm.scale_log2 = a.scale_log2;
    prm.early = a.early;
    prm.status = status;
    if constexpr (MIX) {
        if (!L.kscales || !L.gbits || !L.goff) return cudaErrorInvalidValue;
        const MixBook& mb = mixbook();
        for (int w = 0; w < 3; ++w)
            for (int k = 0; k < 16; ++k) {
                prm.mlo[w][k / 4] |= (uint32_t)(mb.c16[w][k] & 0xFF) << (8 * (k % 4));
                prm.mhi[w][k / 4] |= (uint32_t)(mb.c16[w][k] >> 8) << (8 * (k % 4));
            }
        prm.inv_lam = 1.0f / mb.lam;
        prm.gbits = L.gbits;
        prm.goff = L.goff;
        prm.vhead = L.vhead;
    } else {
        const Codebook& cb = codebook(BITS);
        for (int k = 0; k < 16; ++k) {
            prm.tlo[k / 4] |= (uint32_t)(cb.c16[k] & 0xFF) << (8 * (k % 4));
            prm.thi[k / 4] |= (uint32_t)(cb.c16[k] >> 8) << (8 * (k % 4));
        }
        prm.inv_lam = 1.0f / cb.lam;
    }
    prm.kscales = L.kscales;
    const CUtensorMap& km = *L.kmap;
    const bool tail = prm.tK != nullptr;
    const bool kb = L.kscales != nullptr;
#define KVP_ROWS_LAUNCH(DD, TT, SS, KK) \
    launch_cfg<DD, BITS, TT, SS, KK, MIX>(km, prm, ntiles, s.kv_heads, RGN, a.ws_ctas, a.ws_nslice_max, \
                                          a.ws_nslice, st)
// (MIX instances are block-scaled only: their second branch is the first)
#define KVP_ROWS_KB(DD, TT, SS) (kb ? KVP_ROWS_LAUNCH(DD, TT, SS, true) : KVP_ROWS_LAUNCH(DD, TT, SS, MIX))
    if (D == 64) {
        if (spread) return tail ? KVP_ROWS_KB(64, true, true) : KVP_ROWS_KB(64, false, true);
        return tail ? KVP_ROWS_KB(64, true, false) : KVP_ROWS_KB(64, false, false);
    }
    if (spread) return tail ? KVP_ROWS_KB(128, true, true) : KVP_ROWS_KB(128, false, true);
    return tail ? KVP_ROWS_KB(128, true, false) : KVP_ROWS_KB(128, false, false);
#undef KVP_ROWS_KB
#undef KVP_ROWS_LAUNCH
}

}  // namespace kvp
