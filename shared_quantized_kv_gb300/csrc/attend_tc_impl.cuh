// Tensor-core decode attention over the shared pool (sm_103a, tcgen05).
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
// Per CTA (one per SM): 16 worker warps and one issuer warp. Worker warp w
// owns TMEM lane quarter w % 4 and column group w / 4. The issuer warp
// allocates tensor memory and its lane 0 issues every bulk copy and MMA, so
// that the time the tensor pipe takes to accept a batch of MMAs never stalls
// a worker; workers tell it that operands are ready through counted
// mbarriers, and wait for its copies and MMAs on mbarriers (one worker thread
// polls, the others sleep in a named barrier).
//   * copies: per tile of 128 tokens a TMA load of int8 K (128-byte swizzle,
//     so that one thread per token reads its row without bank conflicts) and
//     bulk copies of the tile's packed V code groups and norms into a ring of
//     stages, one mbarrier per stage. When no kernel before it in the stream
//     can still be writing the layer, the first tiles are requested before
//     the grid-dependency wait, overlapping the previous kernel's tail.
//   * the context split of a CTA is processed in chunks of up to three tiles
//     (two for 128 query rows), sized by tensor memory:
//     - K^ of every tile of the chunk: int8 -> fp16 (exact, byte permutes)
//       straight into TMEM as the A operand of S^T = K^ Q^T (tokens on
//       M = 128, query rows on N); Q is fp16 in shared memory, each row scaled
//       by its own power of two. One batch of MMAs for the chunk.
//     - V^T: thread = (rotated coordinate, 32 tokens): codes of the pool
//       layout (one packed sequence per coordinate and 32-token group) ->
//       fp16 lam * c[code] by byte-permute table lookups, into the K^
//       columns once the S^T MMAs are done, as the A operand of
//       O^T += V^T P'^T. The accumulator stays in the rotated domain,
//       sum_t p_t n_t c[code_t]; the inverse FWHT runs once per output row.
//     - one exact maximum per row over the chunk (thread = token, then
//       redux across lanes and shared memory across lane quarters); O^T and
//       the row sums are rescaled at most once per chunk.
//     - per tile, P' = p * n_t / 2^k split into fp16 hi (top 11 significant
//       bits) and fp16 lo (the exact remainder), two MN-major operands, so P'
//       carries ~22 bits into the MMA; the tile's P'.V MMAs run while the
//       next tile's P' is formed.
//   epilogue: each CTA stages its partial rows (O^T column, m, l) in shared
//     memory and sends the rows of each agent (consecutive at both ends)
//     with one bulk copy into the shared memory of the CTA that owns the
//     agent, completing on the owner's mbarrier; each owner merges its rows
//     (log-sum-exp), applies one inverse FWHT per row (warp shuffles), joins
//     the agent's tail and writes the row.
//   tails (instances with TAIL only): the owner CTA computes its agents' tail
//     attention on CUDA cores in the prologue, while the first tiles are in
//     flight; tail V rows pass through shared memory in blocks, the next
//     block's loads in flight while one is used.
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
namespace {

constexpr int kTile = 128;
constexpr int kWorkers = 512;               // 16 worker warps: (TMEM lane quarter) x (column group)
constexpr int kWorkerWarps = kWorkers / 32;
constexpr int kThreads = kWorkers + 32;     // + the issuer warp
constexpr int kIssuer = kWorkerWarps;       // warp index of the issuer
constexpr int kGroups = 4;                  // column groups of worker warps
constexpr uint32_t kBarWork = 1;            // named barrier of the worker warps
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;
constexpr uint32_t kCols = 512;             // TMEM: O^T, S^T per chunk tile, K^/V^T per chunk tile
constexpr int kMaxChunk = 3;
constexpr int kMaxCluster = 16;             // CTAs per cluster (context splits of one KV head)

struct TcParams {
    const uint8_t* vcodes;
    const float* vnorm;
    const float* kscale;
    const uint32_t* vnmax;
    int ctx, ctx_pad, Hk;
    const uint16_t* Q;
    int Hq, G, R;
    const uint16_t* tK;
    const uint16_t* tV;
    const int32_t* tlen;
    int tail_max;
    float* out;
    float scale_log2;
    int tps;     // tokens per CTA, a multiple of kTile
    int nstage;  // shared-memory stages of raw tiles
    int nc;      // tiles per chunk, at most the stages
    int early;   // 1: the layer's bytes may be read before the grid-dependency wait
    int own;     // merge slots per source CTA (the most rows one CTA owns)
    int* status;
    uint32_t tlo[4], thi[4];  // low / high bytes of fp16 lam * c[k], entry k in byte k % 4 of word k / 4
    float inv_lam;
};

struct Layout {
    uint32_t stage, rv, rn;  // bytes per raw stage; V codes and norms inside one
    uint32_t q, p, plo, misc, bars, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// most tiles per chunk for W query rows (TMEM: O^T, then S^T and K^/V^T per tile)
__host__ __device__ constexpr int chunk_tiles(int W) { return W <= 64 ? 3 : 2; }

// W = query rows per CTA (MMA N). After the main loop everything below misc
// (raw stages, Q, P') is reused: this CTA's staging rows at 0, the merge
// slots that other CTAs fill right after them.
__host__ __device__ inline Layout make_layout(int D, int bits, int W, int nstage) {
    Layout L;
    L.rv = kTile * D;
    L.rn = L.rv + kTile * D * bits / 8;
    L.stage = align_up(L.rn + kTile * 4, 1024);
    uint32_t o = nstage * L.stage;  // raw stages start at 0
    L.q = o;
    o = align_up(o + W * D * 2, 1024);
    L.p = o;
    L.plo = W <= 64 ? 16384 : 32768;  // per chunk tile: P' hi, then P' lo
    o += chunk_tiles(W) * 2 * L.plo;
    L.misc = o;
    o += 15 * W * 4;
    L.bars = align_up(o, 8);
    o = L.bars + 8 * (nstage + 4 + kMaxChunk) + 8;
    L.total = align_up(o, 1024);
    return L;
}

// bytes of the staging rows (W rows of D + 4 floats); the merge slots start there
__host__ __device__ inline uint32_t staging_bytes(int D, int W) { return align_up(W * (D + 4) * 4, 1024); }

__device__ __forceinline__ float bf2f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ int f2ord(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

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

// the 32 codes of one packed sequence (4*BITS bytes at `row`) -> 16 fp16x2
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

// sum over the 32 lanes for each of N values; afterwards lane l holds the
// sums of columns [l*N/32, l*N/32 + N/32) when N >= 32, or column l*N/32
// (replicated over 32/N lanes) when N < 32.
template <int N>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N], int lane) {
    int len = N;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (len > 1) {
            const int half = len / 2;
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                if (k < half) {
                    const float send = up ? v[k] : v[k + half];
                    const float keep = up ? v[k + half] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            len = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}


template <int N>
__device__ __forceinline__ void tmem_ld_f(uint32_t taddr, float (&v)[N]) {
    uint32_t r[N];
    ptx::tmem_ldn<N>(taddr, r);
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = __uint_as_float(r[e]);
}

// 16 codes (half h of one packed 32-token sequence at `row`) -> 8 fp16x2
template <int BITS>
__device__ __forceinline__ void decode16(const unsigned char* row, int h, const uint32_t (&tlo)[4],
                                         const uint32_t (&thi)[4], uint32_t (&r)[8]) {
    uint32_t f0, f1;  // two fields of 8 codes
    if constexpr (BITS == 2) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(row)[h];
        f0 = w; f1 = w >> 16;
    } else if constexpr (BITS == 3) {
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(row) + h;
        const uint32_t a = wp[0], b = wp[1];
        if (h == 0) { f0 = a; f1 = __funnelshift_r(a, b, 24); }
        else { f0 = __funnelshift_r(a, b, 16); f1 = b >> 8; }
    } else {
        const uint2 w = reinterpret_cast<const uint2*>(row)[h];
        f0 = w.x; f1 = w.y;
    }
    const uint32_t y0 = spread8<BITS>(f0), y1 = spread8<BITS>(f1);
    lookup4<BITS>(y0, tlo, thi, r[0], r[1]);
    lookup4<BITS>(y0 >> 16, tlo, thi, r[2], r[3]);
    lookup4<BITS>(y1, tlo, thi, r[4], r[5]);
    lookup4<BITS>(y1 >> 16, tlo, thi, r[6], r[7]);
}

// Attention of the owned agents' rows over their private bf16 tails (plain
// CUDA cores on the worker threads, online softmax in log2 units, 256 tokens
// per chunk). Writes the unnormalised accumulator to `out` and (m, l) per row
// to `tailml`; `stage` is 13 KB of shared memory that is free until the main
// loop. Every thread of the CTA calls it (it holds CTA barriers).
template <int D>
__device__ __noinline__ void tail_attention(const TcParams& p, unsigned char* stage, float* tailml,
                                            int S, int crank, int g, int row0, int nrows) {
    constexpr int TCH = 256;
    constexpr int RPT = kWorkers / D;  // P.V phase: row sub-blocks
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const bool worker = tid < kWorkers;
    float* tq = reinterpret_cast<float*>(stage);                                // [8][D]
    float* tl = reinterpret_cast<float*>(stage + 8 * D * 4);                   // [8][TCH]
    float* tmx = reinterpret_cast<float*>(stage + 8 * D * 4 + 8 * TCH * 4);    // [8]
    // P.V: VR tail V rows at a time through shared memory (the next block's
    // loads in flight while this one is used), VCH 16-byte chunks per block
    constexpr int VR = 64;
    constexpr int VCH = VR * D / 8;
    constexpr int VPT = VCH / kWorkers;  // chunks per worker thread
    static_assert(VCH % kWorkers == 0, "V block chunks per worker");
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
            for (int i = tid; worker && i < 8 * D; i += kWorkers) {
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
                const bool tok_ok = worker && c0 + t < tmax;
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
                    if (worker) tl[k * TCH + t] = lg[kk];
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
                if (worker) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int k = k0 + 2 * kk;
                        float mk = m_run[0];
#pragma unroll
                        for (int q2 = 1; q2 < 8; ++q2) if (q2 == k) mk = m_run[q2];
                        tl[k * TCH + t] = (lg[kk] == -CUDART_INF_F) ? 0.f : ptx::ex2(lg[kk] - mk);
                    }
                }
                __syncthreads();
                {
                    const int n2 = min(TCH, tmax - c0);
                    auto vload = [&](int tb, uint4 (&u)[VPT]) {
#pragma unroll
                        for (int i = 0; i < VPT; ++i) {
                            const int ch = tid + i * kWorkers, row = tb + ch / (D / 8);
                            u[i] = make_uint4(0, 0, 0, 0);
                            if (worker && row < n2)
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
                        if (worker) {
#pragma unroll
                            for (int i = 0; i < VPT; ++i) tv[tid + i * kWorkers] = nxt[i];
                        }
                        __syncthreads();
                        if (tb + VR < n2) vload(tb + VR, nxt);
                        if (worker) {
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
                        }
                        __syncthreads();
                    }
                    if (worker) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (k % RPT != sub || k >= cnt) continue;
                            acc[k] = acc[k] * alpha[k] + sacc[k / RPT];
                            l_run[k] = l_run[k] * alpha[k] + ls[k / RPT];
                        }
                    }
                }
            }
            if (worker) {
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
            }
            __syncthreads();
        }
    }
}

// TAIL: the call has private bf16 tails (instances without them hold no tail code)
template <int D, int W, int BITS, bool TAIL>
__global__ void __launch_bounds__(kThreads, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap kmap, const TcParams p) {
    constexpr int CPT = W / kGroups;         // query rows (TMEM columns) per worker thread: 4..32
    constexpr int CH = CPT < 16 ? CPT : 16;  // columns per TMEM load
    constexpr int EPL = D / 32;              // channels per lane in the merge
    constexpr int VB = D * BITS / 8;         // code bytes per token
    constexpr int GB = D * 4 * BITS;         // bytes per 32-token code group
    constexpr int KC = D / 64;               // 16-byte K chunks per worker thread (of D / 16 per row)
    constexpr int ROWF = D + 4;              // floats per merge row: O^T column, m, l, padding
    constexpr int NC = chunk_tiles(W);
    constexpr uint32_t kColS = 128, kColKV = 128 + NC * W;  // O^T at column 0

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = (int)ptx::cluster_size();
    const int crank = (int)ptx::cluster_rank();
    const Layout lay = make_layout(D, BITS, W, p.nstage);
    unsigned char* sQ = sm + lay.q;
    unsigned char* sP = sm + lay.p;
    float* sO = reinterpret_cast<float*>(sm);                             // epilogue: [W][ROWF]
    float* slots = reinterpret_cast<float*>(sm + staging_bytes(D, W));    // epilogue: [S][own][ROWF]
    // [2][W] (logit factor, running maximum in log2 units) per row, one copy
    // per chunk parity: chunk k reads copy k & 1 and writes copy (k + 1) & 1
    float2* sFM = reinterpret_cast<float2*>(sm + lay.misc);
    float* lsum = reinterpret_cast<float*>(sFM + 2 * W);   // [4][W] row-sum partials
    float* colmax = lsum + 4 * W;                          // [4][W] chunk maxima; then alpha per row
    float* tailml = colmax + 4 * W;                        // [W][2]
    uint32_t* sOwn = reinterpret_cast<uint32_t*>(tailml + 2 * W);  // [W] owner << 16 | slot
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay.bars);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + p.nstage + 4 + kMaxChunk);
    const uint32_t bar_full = ptx::smem_u32(bars);
    const uint32_t bar_s = bar_full + 8 * p.nstage;  // S^T of the chunk is in TMEM
    const uint32_t bar_o = bar_s + 8;                // the chunk's P'.V MMAs are done
    const uint32_t bar_m = bar_o + 8;                // every merge row sent to this CTA has landed
    const uint32_t bar_k = bar_m + 8;                // workers: K^ of the chunk is in TMEM
    const uint32_t bar_p = bar_k + 8;                // workers: P'_j (and V^T) ready, one per chunk tile

    const int g = blockIdx.y;
    const int row0 = blockIdx.z * W;
    const int nrows = min(W, p.R - row0);  // a multiple of G
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const bool worker = warp < kWorkerWarps;
    const int q = warp & 3, cgp = (warp >> 2) & 3;
    const int tok = q * 32 + lane;      // token of a worker in S^T / K^; channel in O^T / V^T
    const bool has_ch = worker && q * 32 < D;  // warp-uniform
    const int t_begin = crank * p.tps;
    const int t_end = min(p.ctx, t_begin + p.tps);
    const int ntile = (t_end - t_begin + kTile - 1) / kTile;  // >= 1
    const int nchunk = (ntile + p.nc - 1) / p.nc;
    const long long head_tok = (long long)g * p.ctx_pad;
    const uint32_t stage_bytes = kTile * D + kTile * VB + kTile * 4;
    // rows owned here: the G rows of every agent ar (relative) with ar % S == crank
    const int nag = nrows / p.G;
    const int own_cnt = crank < nag ? ((nag - crank + S - 1) / S) * p.G : 0;
    const bool leader = warp == kIssuer && lane == 0;  // issues copies and MMAs

    auto issue_tile = [&](int i) {
        const int s = i % p.nstage;
        const long long t0 = head_tok + t_begin + (long long)i * kTile;
        const uint32_t dst = ptx::smem_u32(sm + s * lay.stage);
        const uint32_t bar = bar_full + 8 * s;
        ptx::mbar_expect_tx(bar, stage_bytes);
        ptx::tma_load_2d(dst, &kmap, 0, (int)t0, bar);
        ptx::bulk_g2s(dst + lay.rv, p.vcodes + t0 * VB, kTile * VB, bar);
        ptx::bulk_g2s(dst + lay.rn, p.vnorm + t0, kTile * 4, bar);
    };
    auto issue_first = [&]() {
        for (int i = 0; i < min(ntile, p.nstage); ++i) issue_tile(i);
        for (int i = p.nstage; i < ntile; ++i) {  // later tiles: warm L2
            const long long t0 = head_tok + t_begin + (long long)i * kTile;
            ptx::tma_prefetch_2d(&kmap, 0, (int)t0);
            ptx::prefetch_l2(p.vcodes + t0 * VB, kTile * VB);
            ptx::prefetch_l2(p.vnorm + t0, kTile * 4);
        }
    };

    // ---------------------------------------------------------------- setup
    if (leader) {
        for (int s = 0; s < p.nstage + 3; ++s) ptx::mbar_init(bar_full + 8 * s, 1);  // stages, S^T, P'.V, merge
        ptx::mbar_init(bar_k, kWorkerWarps);
        for (int j = 0; j < kMaxChunk; ++j) ptx::mbar_init(bar_p + 8 * j, kWorkerWarps);
        ptx::mbar_init_fence();
        if (own_cnt > 0) ptx::mbar_expect_tx(bar_m, (uint32_t)(S * own_cnt * ROWF * 4));
        if (p.early) issue_first();
    }
    if (warp == kIssuer) ptx::tmem_alloc(ptx::smem_u32(tslot), kCols);  // overlaps the Q load
    if (tid < W) {
        sFM[tid].y = -CUDART_INF_F;
        const int ar = tid / p.G;  // agent of row tid, relative to the CTA's first agent
        sOwn[tid] = ((uint32_t)(ar % S) << 16) | (uint32_t)((ar / S) * p.G + tid % p.G);
    }

    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    if (leader && !p.early) issue_first();
    bool timed_out = false;
    // P' = p * n_t / nref with nref the power of two >= the largest norm of the layer
    const uint32_t nb = *p.vnmax;
    const float kscale = *p.kscale;

    // 1. Q rows -> fp16 in a 128-byte-swizzled K-major operand; each row is
    //    scaled by the power of two that puts its largest |q| in [2^14, 2^15)
    //    (exact), and the logit factor of the row undoes it.
    if (worker) {
        constexpr int CPR = D / 8;            // 16-byte chunks per row
        constexpr int RPP = kWorkers / CPR;   // rows per pass
        constexpr int NP = (W + RPP - 1) / RPP;
        uint4 qv[NP];
        const int c = tid % CPR;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const int r = k * RPP + tid / CPR;
            qv[k] = make_uint4(0, 0, 0, 0);
            if (r < nrows) {
                const int a = (row0 + r) / p.G, j = (row0 + r) % p.G;
                qv[k] = *reinterpret_cast<const uint4*>(p.Q + ((long long)a * p.Hq + g * p.G + j) * D + c * 8);
            }
        }
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const int r = k * RPP + tid / CPR;
            const uint32_t m7 = 0x7FFF7FFFu;
            const uint4 u = qv[k];
            const uint32_t am = __vmaxu2(__vmaxu2(u.x & m7, u.y & m7), __vmaxu2(u.z & m7, u.w & m7));
            uint32_t qmax = max(am & 0xFFFFu, am >> 16);
#pragma unroll
            for (int o = CPR / 2; o >= 1; o >>= 1) qmax = max(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
            int qe = 0;
            if (qmax != 0 && qmax < 0x7F80u) qe = 14 - ((int)((qmax >> 7) & 0xFF) - 127);
            qe = max(-100, min(100, qe));
            const float qmul = ldexpf(1.0f, qe);
            if (r < W) {
                uint4 v;
                v.x = pack_h2(bf2f(u.x & 0xFFFF) * qmul, bf2f(u.x >> 16) * qmul);
                v.y = pack_h2(bf2f(u.y & 0xFFFF) * qmul, bf2f(u.y >> 16) * qmul);
                v.z = pack_h2(bf2f(u.z & 0xFFFF) * qmul, bf2f(u.z >> 16) * qmul);
                v.w = pack_h2(bf2f(u.w & 0xFFFF) * qmul, bf2f(u.w >> 16) * qmul);
                *reinterpret_cast<uint4*>(sQ + (c / 8) * (W * 128) + (r / 8) * 1024 + (r % 8) * 128 +
                                          (((c % 8) ^ (r % 8)) * 16)) = v;
                if (c == 0) {
                    const float cf = r < nrows ? p.scale_log2 * kscale * ldexpf(1.0f, -qe) : 0.f;
                    sFM[r].x = cf;
                    sFM[W + r].x = cf;
                }
            }
        }
    }
    float vr = 1.0f, nref = 1.0f;
    {
        const int ex = (int)((nb >> 23) & 0xFF);
        if (nb != 0 && ex < 255 && ex > 0) {
            const int k = ex - 127 + ((nb & 0x7FFFFF) != 0 ? 1 : 0);
            nref = ldexpf(1.0f, k);
            vr = ldexpf(1.0f, -k);
        }
    }

    // 2. tails of the agents this CTA owns (CUDA cores), overlapping the first
    //    copies; the P' area is free until the first softmax
    if constexpr (TAIL) tail_attention<D>(p, sP, tailml, S, crank, g, row0, nrows);
    ptx::fence_proxy_async();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t tO = tmem;                  // O^T: W columns
    const uint32_t tS = tmem + kColS;          // S^T of chunk tile j: W columns at tS + j*W
    const uint32_t tKV = tmem + kColKV;        // K^, then V^T, of chunk tile j: 64 columns at tKV + 64*j
    float lp[CPT];     // worker: row-sum partials of its token
#pragma unroll
    for (int j = 0; j < CPT; ++j) lp[j] = 0.f;
    const int colb = cgp * CPT;

    if (warp == kIssuer) {
        // 3a. issuer: S^T MMAs once the chunk's K^ is in TMEM, P'.V MMAs per
        //     tile once its P' is in shared memory; refills the chunk's stages
        //     once the first P' shows that the workers are done with them
        if (lane == 0) {
            const uint32_t idesc1 = ptx::idesc_f16(128, W, 0, 0);
            const uint32_t idesc2 = ptx::idesc_f16(128, W, 0, 1);
            const uint32_t aQ = ptx::smem_u32(sQ), aP = ptx::smem_u32(sP);
            for (int c0 = 0, k = 0; c0 < ntile; c0 += p.nc, ++k) {
                const int n = min(p.nc, ntile - c0);
                if (!timed_out && !ptx::mbar_wait(bar_k, k & 1, kWaitNs)) timed_out = true;
                ptx::tc_fence_after();
                for (int j = 0; j < n; ++j) {  // S^T_j = K^_j Q^T
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t bd = ptx::sdesc(aQ + (ks / 4) * (W * 128) + (ks % 4) * 32, 16, 1024);
                        ptx::mma_f16_ta(tS + j * W, tKV + 64 * j + ks * 8, bd, idesc1, ks > 0 ? 1u : 0u);
                    }
                }
                ptx::mma_commit(bar_s);
                for (int j = 0; j < n; ++j) {  // O^T += V^T_j (P'_hi + P'_lo)_j^T
                    if (!timed_out && !ptx::mbar_wait(bar_p + 8 * j, k & 1, kWaitNs)) timed_out = true;
                    ptx::tc_fence_after();
                    const uint32_t aPj = aP + j * 2 * lay.plo;
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks) {
                        const uint64_t bh = ptx::sdesc(aPj + ks * 2048, 16384, 1024);
                        const uint64_t bl = ptx::sdesc(aPj + lay.plo + ks * 2048, 16384, 1024);
                        ptx::mma_f16_ta(tO, tKV + 64 * j + ks * 8, bh, idesc2, (c0 + j > 0 || ks > 0) ? 1u : 0u);
                        ptx::mma_f16_ta(tO, tKV + 64 * j + ks * 8, bl, idesc2, 1u);
                    }
                    if (j == 0)
                        for (int jj = 0; jj < n; ++jj)
                            if (c0 + jj + p.nstage < ntile) issue_tile(c0 + jj + p.nstage);
                }
                ptx::mma_commit(bar_o);
            }
            // the last commit covers every MMA issued; waited for even after
            // a timeout, so that no MMA is still running when TMEM is released
            if (!ptx::mbar_wait(bar_o, (nchunk - 1) & 1, kWaitNs)) timed_out = true;
            if (timed_out) {
                // give the copies still in flight a bounded chance to land
                for (int i = max(0, ntile - p.nstage); i < ntile; ++i)
                    ptx::mbar_wait(bar_full + 8 * (i % p.nstage), (i / p.nstage) & 1, kWaitNs);
            }
        }
        __syncwarp();
    } else {
        // 3b. workers
        uint32_t tlo[4], thi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) { tlo[k] = p.tlo[k]; thi[k] = p.thi[k]; }
        // one worker polls, the others sleep in the workers' named barrier
        auto wwait = [&](uint32_t bar, uint32_t parity) {
            if (tid == 0 && !timed_out && !ptx::mbar_wait(bar, parity, kWaitNs)) timed_out = true;
        };
        // after a warp's own TMEM stores / shared-memory writes, one arrive for the warp
        auto warp_arrive = [&](uint32_t bar) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar);
            __syncwarp();
        };
        for (int c0 = 0, k = 0; c0 < ntile; c0 += p.nc, ++k) {
            const int n = min(p.nc, ntile - c0);
            int sj[NC];  // raw stage of chunk tile j
#pragma unroll
            for (int j = 0; j < NC; ++j) sj[j] = (c0 + j) % p.nstage;
            // (a) the previous chunk's P'.V MMAs are done (K^/V^T columns, P'
            //     free, O^T final for this chunk's rescale); the tiles landed
            if (k > 0) wwait(bar_o, (k - 1) & 1);
            for (int j = 0; j < n; ++j) wwait(bar_full + 8 * sj[j], ((c0 + j) / p.nstage) & 1);
            ptx::bar_sync(kBarWork, kWorkers);
            ptx::tc_fence_after();

            // (b) K^ of the chunk: token tok, channels 16*KC*cgp .. +16*KC
            if (cgp * KC < D / 16) {
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    if (j >= n) break;
                    const unsigned char* st = sm + sj[j] * lay.stage;
                    const int sw = D == 128 ? (tok & 7) : ((tok >> 1) & 3);  // TMA 128 B / 64 B swizzle
                    uint32_t r[8 * KC];
#pragma unroll
                    for (int kc = 0; kc < KC; ++kc) {
                        const uint4 u = *reinterpret_cast<const uint4*>(st + tok * D + (((cgp * KC + kc) ^ sw) << 4));
                        i8x4_to_h2x2(u.x, r[8 * kc + 0], r[8 * kc + 1]);
                        i8x4_to_h2x2(u.y, r[8 * kc + 2], r[8 * kc + 3]);
                        i8x4_to_h2x2(u.z, r[8 * kc + 4], r[8 * kc + 5]);
                        i8x4_to_h2x2(u.w, r[8 * kc + 6], r[8 * kc + 7]);
                    }
                    if constexpr (KC == 2) ptx::tmem_st16(tKV + 64 * j + lane_off + cgp * 16, r);
                    else ptx::tmem_stn<8>(tKV + 64 * j + lane_off + cgp * 8, r);
                }
                ptx::tmem_wait_st();
            }
            warp_arrive(bar_k);

            // (c) token norms of the chunk while the S^T MMAs run
            float nsj[NC];
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                nsj[j] = 0.f;
                if (j < n) {
                    const bool valid = (t_begin + (c0 + j) * kTile + tok) < t_end;
                    nsj[j] = valid ? reinterpret_cast<const float*>(sm + sj[j] * lay.stage + lay.rn)[tok] * vr : 0.f;
                }
            }

            // (d) S^T is in TMEM and K^ is consumed: V^T (channel tok, tokens
            //     32*cgp .. 32*cgp+31) into the same columns
            wwait(bar_s, k & 1);
            ptx::bar_sync(kBarWork, kWorkers);
            ptx::tc_fence_after();
            if (has_ch) {
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    if (j >= n) break;
                    uint32_t r[16];
                    decode32<BITS>(sm + sj[j] * lay.stage + lay.rv + cgp * GB + tok * (4 * BITS), tlo, thi, r);
                    ptx::tmem_st16(tKV + 64 * j + lane_off + cgp * 16, r);
                }
            }

            // (e) exact maxima of the chunk's rows: this thread's token over its
            //     tiles, then across lanes (redux) and lane quarters (shared
            //     memory); thread r < W then raises the running maximum of row r
            const float2* fmo = sFM + (k & 1) * W;  // before the chunk
            float2* fmn = sFM + ((k + 1) & 1) * W;  // after it
#pragma unroll
            for (int e0 = 0; e0 < CPT; e0 += CH) {
                float cmax[CH];
#pragma unroll
                for (int e = 0; e < CH; ++e) cmax[e] = -CUDART_INF_F;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    if (j >= n) break;
                    const bool valid = (t_begin + (c0 + j) * kTile + tok) < t_end;
                    float y[CH];
                    tmem_ld_f<CH>(tS + j * W + lane_off + colb + e0, y);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < CH; ++e)
                        if (valid) cmax[e] = fmaxf(cmax[e], __fmul_rn(y[e], fmo[colb + e0 + e].x));
                }
#pragma unroll
                for (int e = 0; e < CH; ++e) {
                    const float mx = ord2f(__reduce_max_sync(0xffffffffu, f2ord(cmax[e])));
                    if (lane == (e & 31)) colmax[q * W + colb + e0 + e] = mx;
                }
            }
            ptx::bar_sync(kBarWork, kWorkers);  // colmax complete
            if (tid < W) {
                const float2 fo = fmo[tid];
                const float mn = fmaxf(fo.y, fmaxf(fmaxf(colmax[tid], colmax[W + tid]),
                                                   fmaxf(colmax[2 * W + tid], colmax[3 * W + tid])));
                fmn[tid] = make_float2(fo.x, mn);
                colmax[tid] = (fo.y == -CUDART_INF_F) ? 0.f : ptx::ex2(fo.y - mn);  // alpha of row tid
            }
            ptx::bar_sync(kBarWork, kWorkers);  // new maxima and alphas published
            constexpr int RS = CPT < 8 ? CPT : 8;  // columns per O^T rescale access
#pragma unroll
            for (int e0 = 0; e0 < CPT; e0 += RS) {
                float alpha[RS];
                bool any = false;  // the same in every lane (the warp's columns)
#pragma unroll
                for (int e = 0; e < RS; ++e) {
                    alpha[e] = colmax[colb + e0 + e];
                    any |= alpha[e] != 1.f;
                    lp[e0 + e] *= alpha[e];
                }
                if (k > 0 && has_ch && any) {  // O^T of earlier chunks (their MMAs are done)
                    uint32_t r[RS];
                    ptx::tmem_ldn<RS>(tO + lane_off + colb + e0, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < RS; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha[e]);
                    ptx::tmem_stn<RS>(tO + lane_off + colb + e0, r);
                }
            }

            // (f) per tile: P'^T = p * n_t / nref as fp16 hi + lo (MN-major, one
            //     128-byte swizzled row of 64 query rows per token) and the
            //     row-sum partials of p; then the issuer's P'.V MMAs
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                if (j >= n) break;
                const bool valid = (t_begin + (c0 + j) * kTile + tok) < t_end;
                unsigned char* pj = sP + j * 2 * lay.plo;
#pragma unroll
                for (int e0 = 0; e0 < CPT; e0 += CH) {
                    float y[CH];
                    tmem_ld_f<CH>(tS + j * W + lane_off + colb + e0, y);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e8 = 0; e8 < CH; e8 += 8) {
                        constexpr int NW = CH < 8 ? CH / 2 : 4;  // fp16x2 words per store
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 2 * NW; e += 2) {
                            float hi[2], lo[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int ee = e8 + e + u;
                                const int col = colb + e0 + ee;
                                const float2 fm = fmn[col];
                                // the logit rounded exactly as for the row maximum, so that
                                // it never exceeds the maximum (a fused product would, by up
                                // to half an ulp of the logit, which is large for huge logits)
                                const float pv = valid ? ptx::ex2(__fmul_rn(y[ee], fm.x) - fm.y) : 0.f;
                                lp[e0 + ee] += pv;
                                const float pp = pv * nsj[j];
                                hi[u] = __uint_as_float(__float_as_uint(pp) & 0xFFFFE000u);  // 11 significant bits
                                lo[u] = pp - hi[u];                                          // exact
                            }
                            hw[e / 2] = pack_h2(hi[0], hi[1]);
                            lw[e / 2] = pack_h2(lo[0], lo[1]);
                        }
                        const int col0 = colb + e0 + e8;
                        const int off = (col0 >> 6) * 16384 + (tok >> 3) * 1024 + (tok & 7) * 128 +
                                        ((((col0 & 63) >> 3) ^ (tok & 7)) << 4) + (col0 & 7) * 2;
                        if constexpr (NW == 4) {
                            *reinterpret_cast<uint4*>(pj + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            *reinterpret_cast<uint4*>(pj + lay.plo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        } else {
                            *reinterpret_cast<uint2*>(pj + off) = make_uint2(hw[0], hw[1]);
                            *reinterpret_cast<uint2*>(pj + lay.plo + off) = make_uint2(lw[0], lw[1]);
                        }
                    }
                }
                if (j == 0) ptx::tmem_wait_st();  // V^T and any O^T rescale
                ptx::fence_proxy_async();
                warp_arrive(bar_p + 8 * j);
            }
        }
        wwait(bar_o, (nchunk - 1) & 1);
        ptx::bar_sync(kBarWork, kWorkers);
        ptx::tc_fence_after();
    }

    // this CTA is done with its stages, Q and P': other CTAs may write merge
    // slots there once every CTA of the cluster has arrived (the wait comes
    // right before the sends; the barrier inits are older still)
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_arrive();

    // 4. epilogue: row sums and O^T columns into the staging rows, TMEM released
    float o[CPT];
    if (worker) {
        warp_reduce_scatter<CPT>(lp, lane);
        constexpr int REP = CPT >= 32 ? 1 : 32 / CPT;  // lanes holding the same sum
        if (lane % REP == 0) lsum[q * W + colb + lane / REP] = lp[0];
        __syncwarp();
        if (has_ch) {
#pragma unroll
            for (int e0 = 0; e0 < CPT; e0 += CH) {
                float y[CH];
                tmem_ld_f<CH>(tO + lane_off + colb + e0, y);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < CH; ++e) o[e0 + e] = y[e];
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();  // every MMA is done: the stage area becomes staging rows
    if (has_ch) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int r = colb + j;
            if (r < nrows) sO[r * ROWF + tok] = o[j];
        }
    }
    if (tid < nrows) {
        sO[tid * ROWF + D] = sFM[(nchunk & 1) * W + tid].y;  // final row maximum
        sO[tid * ROWF + D + 1] = lsum[tid] + lsum[W + tid] + lsum[2 * W + tid] + lsum[3 * W + tid];
    }
    if (timed_out) atomicOr(p.status, kStTimeout);
    ptx::fence_proxy_async();
    __syncthreads();

    // 5. send the G rows of each agent, consecutive here and at the owner of
    //    the agent, with one copy: slots (this rank, owner's row index)
    const int nsend = nrows / p.G;  // row groups hold whole agents
    ptx::cluster_wait();
    if (tid < nsend) {
        const uint32_t ow = sOwn[tid * p.G], owner = ow >> 16;
        const float* dst = slots + (size_t)(crank * p.own + (int)(ow & 0xFFFF)) * ROWF;
        ptx::bulk_s2cluster(ptx::dsmem_addr(dst, owner), ptx::smem_u32(sO + tid * p.G * ROWF),
                            (uint32_t)(p.G * ROWF * 4), ptx::dsmem_addr(bars + p.nstage + 2, owner));
        ptx::bulk_commit();
    }

    // 6. merge the owned rows once all S copies of each have landed, one warp per row
    if (own_cnt > 0) {
        const bool bad = tid == 0 && !ptx::mbar_wait(bar_m, 0, kWaitNs);
        const bool ok = !__syncthreads_or(bad);
        if (bad) atomicOr(p.status, kStTimeout);
        const int G = p.G;
        for (int loc = warp; ok && loc < own_cnt; loc += kThreads / 32) {
            const int ar = (loc / G) * S + crank, j = loc % G;
            const int rr = ar * G + j;
            const int a = row0 / G + ar;
            // every lane reads the S (m, l) pairs itself (broadcast loads)
            // and all S partial rows at once: no shuffle chains
            float ms[kMaxCluster], ls[kMaxCluster];
#pragma unroll
            for (int s = 0; s < kMaxCluster; ++s) {
                ms[s] = -CUDART_INF_F;
                ls[s] = 0.f;
                if (s < S) {
                    const float2 ml = *reinterpret_cast<const float2*>(slots + (size_t)(s * p.own + loc) * ROWF + D);
                    ms[s] = ml.x;
                    ls[s] = ml.y;
                }
            }
            float M = -CUDART_INF_F;
#pragma unroll
            for (int s = 0; s < kMaxCluster; ++s)
                if (ls[s] > 0.f) M = fmaxf(M, ms[s]);
            float L = 0.f;
            float acc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxCluster; ++s) {
                if (s < S) {
                    const float w = (ls[s] > 0.f) ? ptx::ex2(ms[s] - M) : 0.f;
                    L = fmaf(w, ls[s], L);
                    const float* src = slots + (size_t)(s * p.own + loc) * ROWF + lane * EPL;
                    if constexpr (EPL == 4) {
                        const float4 v = *reinterpret_cast<const float4*>(src);
                        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
                        acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
                    } else {
                        const float2 v = *reinterpret_cast<const float2*>(src);
                        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
                    }
                }
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
            const float oscale = nref / (float)D * p.inv_lam;
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
    // tensor memory is released last (nothing after the O^T loads uses it), so
    // that its release is off the path to the sends and the merge
    if (warp == kIssuer) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
}


template <int D, int W, int BITS, bool TAIL>
void configure() {
    static bool done = false;
    if (done) return;
    auto kern = attend_tc_kernel<D, W, BITS, TAIL>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    done = true;
}

// How many clusters of S CTAs with `smem` bytes each can be resident at once.
template <int D, int W, int BITS, bool TAIL>
int max_clusters(int S, size_t smem) {
    static int cache[17][2] = {};  // [S] -> (smem key / 1024 + 1, count)
    const int key = (int)(smem / 1024) + 1;
    if (cache[S][0] == key) return cache[S][1];
    configure<D, W, BITS, TAIL>();
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
    if (cudaOccupancyMaxActiveClusters(&n, attend_tc_kernel<D, W, BITS, TAIL>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[S][0] = key;
    cache[S][1] = n;
    return n;
}

template <int D, int W, int BITS, bool TAIL>
cudaError_t launch_cfg(const CUtensorMap& kmap, TcParams prm, int ntiles, int Hk, int RGN, cudaStream_t st) {
    configure<D, W, BITS, TAIL>();
    constexpr uint32_t kMaxSmem = 227 * 1024;
    // one CTA per SM (it uses all 512 TMEM columns): the floor on shared
    // memory keeps a second CTA off the SM, where it would wait in
    // tcgen05.alloc
    constexpr size_t kFloor = 116 * 1024;
    const int rows_cta = std::min(W, prm.R);
    const int agents_cta = (rows_cta + prm.G - 1) / prm.G;
    const int clusters = Hk * RGN;
    // raw stages: as many as fit (up to 4), never fewer than two when a CTA
    // has more than one tile (tile i+1 is expanded while tile i is in use)
    int max_ns = 4;
    while (max_ns > 2 && make_layout(D, BITS, W, max_ns).total + 1024 > kMaxSmem) --max_ns;
    if (make_layout(D, BITS, W, max_ns).total + 1024 > kMaxSmem) return cudaErrorInvalidConfiguration;
    // cluster size: fewest (waves x tiles per CTA), then the larger cluster;
    // the staging rows and the merge slots must fit in the stage area
    int bestS = 0;
    long long best = -1;
    for (int S = 1; S <= kMaxCluster && S <= ntiles; ++S) {
        const int per = (ntiles + S - 1) / S;
        const int own = (agents_cta + S - 1) / S * prm.G;
        const Layout lay = make_layout(D, BITS, W, std::min(max_ns, per));
        if (staging_bytes(D, W) + (size_t)S * own * (D + 4) * 4 > lay.misc) continue;
        const size_t smem = std::max<size_t>(lay.total + 1024, kFloor);
        const int n = max_clusters<D, W, BITS, TAIL>(S, smem);
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
    prm.nstage = std::min(max_ns, per);
    // tiles per chunk: as many as TMEM holds, all resident in their stages
    prm.nc = std::min(W <= 64 ? 3 : 2, prm.nstage);
    const Layout lay = make_layout(D, BITS, W, prm.nstage);
    if (staging_bytes(D, W) + (size_t)S * prm.own * (D + 4) * 4 > lay.misc) return cudaErrorInvalidConfiguration;
    const size_t smem = std::max<size_t>(lay.total + 1024, kFloor);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, Hk, RGN);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
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
    return cudaLaunchKernelEx(&cfg, attend_tc_kernel<D, W, BITS, TAIL>, kmap, prm);
}

template <bool TAIL, int BITS>
cudaError_t launch_w(const CUtensorMap& km, const TcParams& prm, int D, int W, int ntiles, int Hk, int RGN,
                     cudaStream_t st) {
    if (D == 64) {
        if (W == 16) return launch_cfg<64, 16, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
        if (W == 32) return launch_cfg<64, 32, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
        if (W == 64) return launch_cfg<64, 64, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
        return launch_cfg<64, 128, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
    }
    if (W == 16) return launch_cfg<128, 16, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
    if (W == 32) return launch_cfg<128, 32, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
    if (W == 64) return launch_cfg<128, 64, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
    return launch_cfg<128, 128, BITS, TAIL>(km, prm, ntiles, Hk, RGN, st);
}

}  // namespace

// Launch for layers whose V codes have BITS bits.
template <int BITS>
cudaError_t launch_attend_tc_bits(const Shape& s, const LayerBufs& L, const AttendArgs& a,
                                  int* status, cudaStream_t st) {
    const int D = s.head_dim;
    int W;
    if (a.rows <= 16) W = 16;
    else if (a.rows <= 32) W = 32;
    else if (a.rows <= 64) W = 64;
    else W = 128;
    // row groups of W rows must hold whole agents
    if (a.rows > W && W % a.group != 0) return cudaErrorInvalidValue;
    const int RGN = (a.rows + W - 1) / W;
    const int ntiles = (s.ctx + kTile - 1) / kTile;
    TcParams prm = {};
    prm.vcodes = L.vcodes;
    prm.vnorm = L.vnorm;
    prm.kscale = L.kscale;
    prm.vnmax = L.vnmax;
    prm.ctx = s.ctx;
    prm.ctx_pad = s.ctx_pad;
    prm.Hk = s.kv_heads;
    prm.Q = (const uint16_t*)a.Q;
    prm.Hq = a.q_heads;
    prm.G = a.group;
    prm.R = a.rows;
    prm.tK = (const uint16_t*)a.tailK;
    prm.tV = (const uint16_t*)a.tailV;
    prm.tlen = a.tail_len;
    prm.tail_max = a.tail_max;
    prm.out = a.out;
    prm.scale_log2 = a.scale_log2;
    prm.early = a.early;
    prm.status = status;
    const Codebook& cb = codebook(BITS);
    for (int k = 0; k < 16; ++k) {
        prm.tlo[k / 4] |= (uint32_t)(cb.c16[k] & 0xFF) << (8 * (k % 4));
        prm.thi[k / 4] |= (uint32_t)(cb.c16[k] >> 8) << (8 * (k % 4));
    }
    prm.inv_lam = 1.0f / cb.lam;
    const CUtensorMap& km = *L.kmap;
    if (prm.tK != nullptr) return launch_w<true, BITS>(km, prm, D, W, ntiles, s.kv_heads, RGN, st);
    return launch_w<false, BITS>(km, prm, D, W, ntiles, s.kv_heads, RGN, st);
}

}  // namespace kvp
