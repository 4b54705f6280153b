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
// Per CTA (512 threads, 16 warps; warp w reads TMEM lane quarter w % 4 and
// column group w / 4; lane 0 of warp 15 issues the bulk copies and MMAs and
// warp 15 takes no share of the operand conversion):
//   lane 0 of warp 15 keeps a ring of shared-memory stages filled with bulk copies
//     (cp.async.bulk) of the raw tiles -- 128 tokens of int8 K, packed V codes
//     and float norms -- refilling a stage right after the barrier that ends
//     its conversion; one mbarrier per stage tracks the bytes.
//   all warps, per tile of 128 tokens:
//     * int8 K -> fp16 K^ (exact) into a 128-byte-swizzled K-major operand;
//       V codes -> fp16 lam * c[code] into a swizzled MN-major operand (d on
//       the M axis, padded to 128 when d = 64);
//     * one thread issues S^T = K^ Q^T (tokens on M = 128, rows on N) into TMEM;
//     * softmax with the thread = token layout of TMEM: logits in log2 units,
//       a running per-row maximum that is only raised (with a rescale of the
//       TMEM accumulator) when a logit exceeds it by more than 2^8;
//       P' = p * n_t / 2^k is split into fp16 hi (the top 11 significant
//       bits) and fp16 lo (the exact remainder), two swizzled MN-major
//       operands, so P' carries ~22 bits into the MMA;
//     * one thread issues O^T += V^T (P'_hi + P'_lo)^T as two MMAs. V^T is a
//       pure table lookup, fp16(lam * c[code]), with lam chosen so that all
//       lam * c[k] sit within 2^-13..2^-22 of an fp16 value. The accumulator
//       lives in the rotated domain, sum_t p_t n_t c[code_t], and never needs
//       the inverse FWHT per token.
//   epilogue: row sums and O^T are staged in shared memory; the cluster's CTAs
//     merge their splits through distributed shared memory (log-sum-exp), each
//     CTA for the rows of the agents it owns; one inverse FWHT per row (warp
//     shuffles), the agent's tail (computed in the prologue while the first
//     tiles are in flight) joins, and the row is written.
// Every mbarrier wait is bounded; on expiry the kernel records
// KVPOOL_ERR_TIMEOUT in the status word and carries on to its exit without
// waiting again, so a fault never hangs the device.
#pragma once

#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "kvpool_internal.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace kvp {
namespace {

constexpr int kTile = 128;
constexpr int kWork = 512;       // 16 warps: (TMEM lane quarter) x (column group)
constexpr int kThreads = kWork;
constexpr int kMmaWarp = 15;     // its lane 0 issues bulk copies and MMAs; it converts nothing
constexpr int kConv = 480;       // threads of warps 0..14, which convert the operands
constexpr float kTau = 8.0f;                  // P <= 2^kTau between rescales
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;

struct TcParams {
    const int8_t* kq;
    const uint8_t* vcodes;
    const float* vnorm;
    const float* kscale;
    const uint32_t* vnmax;
    int ctx, ctx_pad, Hk;
    const uint16_t* Q;
    int Hq, G, R, agents;
    const uint16_t* tK;
    const uint16_t* tV;
    const int32_t* tlen;
    int tail_max;
    float* out;
    float scale_log2;
    int tps;  // tokens per split, multiple of kTile
    int bits, nstage;
    uint32_t tmem_cols;
    int* status;
    uint32_t c16[8];  // fp16 pairs: lam * centroid[2k], lam * centroid[2k+1]
    float inv_lam;
};

struct Layout {
    uint32_t q, khat, vhat, p, raw, lut, bars, misc, total;
    uint32_t stage, rk, rv, rn;  // bytes per stage and offsets inside one
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// W = rows per row block (MMA N), NB = row blocks per CTA.
__host__ __device__ inline Layout make_layout(int D, int bits, int W, int NB, int nstage) {
    Layout L;
    uint32_t o = 0;
    L.q = o;
    o += NB * W * D * 2;
    o = align_up(o, 1024);
    L.khat = o;
    o += kTile * D * 2;
    L.vhat = o;  // two buffers of 128 (M) x 128 (tokens) fp16
    o += 2 * 32768;
    L.p = o;  // per row block: P hi and P lo, each 16 token-groups x 1024 B
    o += NB * 2 * 16384;
    L.raw = o;
    L.rk = 0;
    L.rv = kTile * D;
    L.rn = L.rv + kTile * D * bits / 8;
    L.stage = align_up(L.rn + kTile * 4, 128);
    o += nstage * L.stage;
    o = align_up(o, 16);
    L.lut = o;  // pair table: 2^(2*bits) fp16x2 entries
    o += 1024;
    L.bars = o;  // full[nstage], mma
    o += 8 * 8;
    L.misc = o;
    // misc: tmem slot, flags, qexp, lsum[4][128], colmax[4][128], M[128], l[128], tail m/l[128][2]
    o += 128 + 4 * 128 * 4 * 2 + 128 * 4 * 2 + 128 * 8;
    L.total = align_up(o, 1024);
    return L;
}

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

// four int8 (biased by 128) -> two fp16x2 holding the signed values exactly
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t magic = 0x64646464u;  // fp16 0x64xx = 1024 + xx
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(x), "r"(magic));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(x), "r"(magic));
    const __half2 bias = __floats2half2_rn(1152.0f, 1152.0f);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// sum over the 32 lanes for each of N values; afterwards lane l holds the
// sums of columns [l*N/32, l*N/32 + N/32) when N >= 32, or column l*N/32
// (replicated over 32/N lanes) when N < 32. Returns the number of values kept.
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

// 32 V codes of token t (channels 32*qd .. 32*qd+31) -> fp16 lam * c[code]
// via a table of code pairs, into four 16-byte chunks of the token's
// MN-major swizzled row of the V^T operand.
template <int BITS>
__device__ __forceinline__ void convert_v_quarter(const unsigned char* src, const uint32_t* pairs,
                                                  unsigned char* vrow, int t, int dc0) {
    constexpr uint32_t PMASK = (1u << (2 * BITS)) - 1;
    uint32_t w[BITS + 1];  // 32 codes = 4*BITS bytes = BITS words
#pragma unroll
    for (int k = 0; k < BITS; ++k) w[k] = *reinterpret_cast<const uint32_t*>(src + 4 * k);
    w[BITS] = 0;
#pragma unroll
    for (int dc = 0; dc < 4; ++dc) {
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int bit = (dc * 8 + 2 * e) * BITS, wi = bit >> 5, off = bit & 31;
            h[e] = pairs[__funnelshift_r(w[wi], w[wi + 1], off) & PMASK];
        }
        *reinterpret_cast<uint4*>(vrow + (((dc0 + dc) ^ (t % 8)) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// Attention of the owned agents' rows over their private bf16 tails (plain
// CUDA cores, online softmax in log2 units). Writes the unnormalised
// accumulator to `out` and (m, l) per row to `tailml`; uses the K^ operand
// area as staging (free before the main loop).
template <int D>
__device__ __noinline__ void tail_attention(const TcParams& p, unsigned char* sK, float* tailml, int S,
                                            int crank, int g, int row0, int nrows) {
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // staging in the K^ operand area, unused until the main loop
    float* tq = reinterpret_cast<float*>(sK);                                // [8][D]
    float* tl = reinterpret_cast<float*>(sK + 8 * D * 4);                   // [8][256]
    float* tred = reinterpret_cast<float*>(sK + 8 * D * 4 + 8 * 256 * 4);   // [8 warps][8]
    constexpr int TCH = 256;                                                 // tokens per chunk
    constexpr int RPT = kWork / D;  // row sub-blocks in the P.V phase
    const int c = tid % D, sub = tid / D;
    const int G = p.G;
    const int a_first = row0 / G, a_last = (row0 + nrows - 1) / G;
    for (int a = a_first + ((crank - a_first % S) % S + S) % S; a <= a_last; a += S)
    for (int jb = max(0, row0 - a * G); jb < min(G, row0 + nrows - a * G); jb += 8) {
        // rows k = 0..7 of the batch are (agent a, head jb + k)
        const int cnt = min(8, min(G, row0 + nrows - a * G) - jb);
        const int ownmask = (1 << cnt) - 1;
        const int rr0 = a * G + jb - row0;
        const int tmax = min(max(p.tlen[a], 0), p.tail_max);
        for (int i = tid; i < 8 * D; i += kThreads) {
            const int k = i / D, cc = i % D;
            float v = 0.f;
            if ((ownmask >> k) & 1)
                v = bf2f(p.Q[((long long)a * p.Hq + g * G + jb + k) * D + cc]);
            tq[k * D + cc] = v;
        }
        float m_run[8], l_run[8], acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) { m_run[k] = -CUDART_INF_F; l_run[k] = 0.f; acc[k] = 0.f; }
        __syncthreads();
        for (int c0 = 0; c0 < tmax; c0 += TCH) {
            const int t = c0 + tid;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float lg = -CUDART_INF_F;
                if (tid < TCH && ((ownmask >> k) & 1)) {
                    if (t < tmax) {
                        const uint16_t* kr = p.tK + (((long long)a * p.Hk + g) * p.tail_max + t) * D;
                        const float* qq = tq + k * D;
                        float dot = 0.f;
                        for (int cc = 0; cc < D; cc += 8) {
                            const uint4 u = *reinterpret_cast<const uint4*>(kr + cc);
                            dot = fmaf(qq[cc + 0], bf2f(u.x & 0xFFFF), dot);
                            dot = fmaf(qq[cc + 1], bf2f(u.x >> 16), dot);
                            dot = fmaf(qq[cc + 2], bf2f(u.y & 0xFFFF), dot);
                            dot = fmaf(qq[cc + 3], bf2f(u.y >> 16), dot);
                            dot = fmaf(qq[cc + 4], bf2f(u.z & 0xFFFF), dot);
                            dot = fmaf(qq[cc + 5], bf2f(u.z >> 16), dot);
                            dot = fmaf(qq[cc + 6], bf2f(u.w & 0xFFFF), dot);
                            dot = fmaf(qq[cc + 7], bf2f(u.w >> 16), dot);
                        }
                        lg = dot * p.scale_log2;
                    }
                }
                if (tid < TCH) {
                    tl[k * TCH + tid] = lg;
                    const float mx = ord2f(__reduce_max_sync(0xffffffffu, f2ord(lg)));
                    if (lane == 0) tred[warp * 8 + k] = mx;
                }
            }
            __syncthreads();
            float mnew[8], alpha[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int w = 0; w < TCH / 32; ++w) mx = fmaxf(mx, tred[w * 8 + k]);
                mnew[k] = fmaxf(m_run[k], mx);
                alpha[k] = (mnew[k] == -CUDART_INF_F) ? 1.f : ptx::ex2(m_run[k] - mnew[k]);
                if (tid < TCH) {
                    const float lg = tl[k * TCH + tid];
                    tl[k * TCH + tid] = (lg == -CUDART_INF_F) ? 0.f : ptx::ex2(lg - mnew[k]);
                }
            }
            __syncthreads();
            const int cend = min(TCH, tmax - c0);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                l_run[k] *= alpha[k];
                acc[k] *= alpha[k];
                m_run[k] = mnew[k];
                if ((k % RPT) != sub || !((ownmask >> k) & 1)) continue;
                const int n = tmax;
                const uint16_t* vr0 = p.tV + (((long long)a * p.Hk + g) * p.tail_max + c0) * D + c;
                const int cnt = min(cend, n - c0);
                float sacc = 0.f, ls = 0.f;
                for (int t2 = 0; t2 < cnt; ++t2) {
                    const float pv = tl[k * TCH + t2];
                    sacc = fmaf(pv, bf2f(vr0[(long long)t2 * D]), sacc);
                    ls += pv;
                }
                acc[k] += sacc;
                l_run[k] += ls;
            }
            __syncthreads();
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if ((k % RPT) != sub || !((ownmask >> k) & 1)) continue;
            const int rr = rr0 + k, j = jb + k;
            p.out[((long long)a * p.Hq + g * G + j) * D + c] = acc[k];
            if (c == 0) {
                tailml[2 * rr] = m_run[k];
                tailml[2 * rr + 1] = l_run[k];
            }
        }
        __syncthreads();
    }
}

template <int D, int W, int NB, int BITS>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const TcParams p) {
    constexpr int RG = NB * W;                   // rows per CTA (W = MMA N per row block)
    constexpr int NCG = (W / 8) < 4 ? (W / 8) : 4;  // column groups of warps
    constexpr int HC = W / NCG;                  // columns per thread per row block (8 or 16)
    constexpr int CPT = NB * HC;                 // columns per thread
    constexpr int EPL = D / 32;                  // elements per lane in the epilogue

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Layout lay = make_layout(D, BITS, W, NB, p.nstage);
    unsigned char* sQ = sm + lay.q;
    unsigned char* sK = sm + lay.khat;
    unsigned char* sV = sm + lay.vhat;
    unsigned char* sP = sm + lay.p;
    unsigned char* sRaw = sm + lay.raw;
    uint32_t* pairs = reinterpret_cast<uint32_t*>(sm + lay.lut);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay.bars);
    unsigned char* misc = sm + lay.misc;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(misc);
    float* sred = reinterpret_cast<float*>(misc + 16);      // [16] block reduction scratch
    float* lsum = reinterpret_cast<float*>(misc + 128);     // [4][128]
    float* colmax = lsum + 4 * 128;                          // [4][128]
    float* sM = colmax + 4 * 128;                            // [128] running row maxima
    float* sL = sM + 128;                                    // [128] row sums
    float* tailml = sL + 128;                                // [128][2]
    float* sO = reinterpret_cast<float*>(sK);                // epilogue: [RG][D], aliases K^, V^

    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    const int g = blockIdx.y;
    const int row0 = blockIdx.z * RG;
    const int nrows = min(RG, p.R - row0);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int t_begin = crank * p.tps;
    const int t_end = min(p.ctx, t_begin + p.tps);
    const int ntile = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
    constexpr int VB = D * BITS / 8;
    const uint32_t stage_bytes = kTile * D + kTile * VB + kTile * 4;
    const uint32_t bar_full = ptx::smem_u32(bars);
    const uint32_t bar_mma = bar_full + 8 * p.nstage;

    // ---------------------------------------------------------------- setup
    if (warp == 0) ptx::tmem_alloc(ptx::smem_u32(tslot), p.tmem_cols);
    if (tid == 32) {
        for (int s = 0; s < p.nstage; ++s) ptx::mbar_init(bar_full + 8 * s, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::mbar_init_fence();
    }
    {
        for (int i = tid; i < (1 << (2 * BITS)); i += kThreads) {
            const int c0 = i & ((1 << BITS) - 1), c1 = i >> BITS;
            const uint32_t h0 = (p.c16[c0 >> 1] >> (16 * (c0 & 1))) & 0xFFFFu;
            const uint32_t h1 = (p.c16[c1 >> 1] >> (16 * (c1 & 1))) & 0xFFFFu;
            pairs[i] = h0 | (h1 << 16);
        }
    }
    if (tid < 128) sM[tid] = -CUDART_INF_F;
    if (D == 64) {  // rows 64..127 of both V^T operand buffers stay zero
        for (int i = tid; i < 2 * 1024; i += kThreads)
            reinterpret_cast<uint4*>(sV + (i / 1024) * 32768 + 16384)[i % 1024] = make_uint4(0, 0, 0, 0);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem;            // S^T: NB*W columns
    const uint32_t tO = tmem + NB * W;   // O^T: NB*W columns

    const long long head_tok = (long long)g * p.ctx_pad;
    if (tid == 0) {  // warm L2 while the previous kernel in the stream drains
        for (int i = 0; i < ntile; ++i) {
            const long long t0 = head_tok + t_begin + (long long)i * kTile;
            ptx::prefetch_l2(p.kq + t0 * D, kTile * D);
            ptx::prefetch_l2(p.vcodes + t0 * VB, kTile * VB);
        }
    }
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    bool timed_out = false;
    // P' = p * n_t / nref with nref the power of two >= the largest norm of the layer
    float vr = 1.0f, nref = 1.0f;
    {
        const uint32_t nb = *p.vnmax;
        const int ex = (int)((nb >> 23) & 0xFF);
        if (nb != 0 && ex < 255 && ex > 0) {
            const int k = ex - 127 + ((nb & 0x7FFFFF) != 0 ? 1 : 0);
            nref = ldexpf(1.0f, k);
            vr = ldexpf(1.0f, -k);
        }
    }
    auto issue_tile = [&](int i) {
        const int s = i % p.nstage;
        const long long t0 = head_tok + t_begin + (long long)i * kTile;
        const uint32_t dst = ptx::smem_u32(sRaw + s * lay.stage);
        ptx::mbar_expect_tx(bar_full + 8 * s, stage_bytes);
        ptx::bulk_g2s(dst + lay.rk, p.kq + t0 * D, kTile * D, bar_full + 8 * s);
        ptx::bulk_g2s(dst + lay.rv, p.vcodes + t0 * VB, kTile * VB, bar_full + 8 * s);
        ptx::bulk_g2s(dst + lay.rn, p.vnorm + t0, kTile * 4, bar_full + 8 * s);
    };
    if (warp == kMmaWarp && lane == 0)
        for (int i = 0; i < min(ntile, p.nstage); ++i) issue_tile(i);

    // 1. Q rows of this CTA -> fp16, scaled by a power of two, swizzled K-major.
    //    All loads of a thread are issued before any is used.
    constexpr int QCH = RG * (D / 8);                     // 16-byte chunks
    constexpr int QPT = (QCH + kWork - 1) / kWork;  // chunks per compute thread
    uint4 qv[QPT];
    uint32_t qmax = 0;
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
        const int idx = k * kWork + tid, rr = idx / (D / 8), c = idx % (D / 8);
        qv[k] = make_uint4(0, 0, 0, 0);
        if (idx < QCH && rr < nrows) {
            const int r = row0 + rr, a = r / p.G, j = r % p.G;
            qv[k] = *reinterpret_cast<const uint4*>(p.Q + ((long long)a * p.Hq + g * p.G + j) * D + c * 8);
        }
    }
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
        const uint32_t m = 0x7FFF7FFFu;
        const uint32_t a = __vmaxu2(__vmaxu2(qv[k].x & m, qv[k].y & m), __vmaxu2(qv[k].z & m, qv[k].w & m));
        qmax = max(qmax, max(a & 0xFFFFu, a >> 16));
    }
    qmax = __reduce_max_sync(0xffffffffu, qmax);
    if (lane == 0) reinterpret_cast<uint32_t*>(sred)[warp] = qmax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) qmax = max(qmax, reinterpret_cast<uint32_t*>(sred)[w]);
    const float amax = __uint_as_float(qmax << 16);
    int qe = 0;  // scale Q by 2^qe so that max |q| lands in [2^14, 2^15)
    if (qmax != 0 && qmax < 0x7F80u) qe = 14 - ((int)((qmax >> 7) & 0xFF) - 127);
    (void)amax;
    qe = max(-100, min(100, qe));
    const float qmul = ldexpf(1.0f, qe);
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
        const int idx = k * kWork + tid, rr = idx / (D / 8), c = idx % (D / 8);
        if (idx >= QCH) continue;
        const uint4 u = qv[k];
        uint4 v;
        v.x = pack_h2(bf2f(u.x & 0xFFFF) * qmul, bf2f(u.x >> 16) * qmul);
        v.y = pack_h2(bf2f(u.y & 0xFFFF) * qmul, bf2f(u.y >> 16) * qmul);
        v.z = pack_h2(bf2f(u.z & 0xFFFF) * qmul, bf2f(u.z >> 16) * qmul);
        v.w = pack_h2(bf2f(u.w & 0xFFFF) * qmul, bf2f(u.w >> 16) * qmul);
        const int rb = rr / W, rl = rr % W;
        *reinterpret_cast<uint4*>(sQ + rb * W * D * 2 + (c / 8) * (W * 128) + (rl / 8) * 1024 +
                                  (rl % 8) * 128 + (((c % 8) ^ (rl % 8)) * 16)) = v;
    }
    const float cf = p.scale_log2 * (*p.kscale) * ldexpf(1.0f, -qe);

    // 2. tails of the agents this CTA owns (CUDA cores), overlapping the first
    //    bulk copies; acc (unnormalised) goes to `out`, m and l to shared memory
    if (p.tK != nullptr) tail_attention<D>(p, sK, tailml, S, crank, g, row0, nrows);
    __syncthreads();

    // 3. main loop over this CTA's tiles
    const int wq = warp & 3;           // TMEM lane quarter
    const int cgr = warp >> 2;         // column group
    const bool has_cols = cgr < NCG;   // warp-uniform
    const int tok = wq * 32 + lane;    // token (S^T lanes) / channel (O^T lanes)
    float lp[CPT];                     // per-thread row-sum partials
#pragma unroll
    for (int j = 0; j < CPT; ++j) lp[j] = 0.f;
    const uint32_t idesc1 = ptx::idesc_f16(128, W, 0, 0);
    const uint32_t idesc2 = ptx::idesc_f16(128, W, 1, 1);
    const uint32_t aK = ptx::smem_u32(sK), aQ = ptx::smem_u32(sQ), aV = ptx::smem_u32(sV),
                   aP = ptx::smem_u32(sP);

    for (int i = 0; i < ntile; ++i) {
        const int s = i % p.nstage;
        const int buf = i & 1;
        if (!timed_out && !ptx::mbar_wait(bar_full + 8 * s, (i / p.nstage) & 1, kWaitNs))
            timed_out = true;
        const unsigned char* rk = sRaw + s * lay.stage + lay.rk;
        const unsigned char* rv = sRaw + s * lay.stage + lay.rv;
        const float* rn = reinterpret_cast<const float*>(sRaw + s * lay.stage + lay.rn);
        // K: 16 int8 per step -> two 16-byte fp16 chunks of the swizzled operand
#pragma unroll
        for (int it = 0; it < (kTile * D / 16 + kConv - 1) / kConv; ++it) {
            const int q = it * kConv + tid;
            if (tid >= kConv || q >= kTile * D / 16) break;
            const int t = q / (D / 16), c16 = q % (D / 16);
            const uint4 u = *reinterpret_cast<const uint4*>(rk + t * D + c16 * 16);
            uint4 o0, o1;
            i8x4_to_h2x2(u.x, o0.x, o0.y);
            i8x4_to_h2x2(u.y, o0.z, o0.w);
            i8x4_to_h2x2(u.z, o1.x, o1.y);
            i8x4_to_h2x2(u.w, o1.z, o1.w);
            const int dc0 = 2 * c16, dc1 = dc0 + 1;
            unsigned char* base = sK + (t / 8) * 1024 + (t % 8) * 128;
            unsigned char* d0 = base + (dc0 / 8) * 16384 + (((dc0 % 8) ^ (t % 8)) * 16);
            unsigned char* d1 = base + (dc1 / 8) * 16384 + (((dc1 % 8) ^ (t % 8)) * 16);
            if (c16 < 4) {
                *reinterpret_cast<uint4*>(d0) = o0;
                *reinterpret_cast<uint4*>(d1) = o1;
            } else {
                *reinterpret_cast<uint4*>(d1) = o1;
                *reinterpret_cast<uint4*>(d0) = o0;
            }
        }
        // V: task = (token, quarter of 32 channels)
        for (int task = tid; tid < kConv && task < kTile * D / 32; task += kConv) {
            const int t = task % kTile, qd = task / kTile;
            const unsigned char* src = rv + t * VB + qd * 4 * BITS;
            unsigned char* vrow = sV + buf * 32768 + (qd / 2) * 16384 + (t / 8) * 1024 + (t % 8) * 128;
            convert_v_quarter<BITS>(src, pairs, vrow, t, (qd % 2) * 4);
        }
        const float ns = rn[tok] * vr;  // this thread's token norm, read before the stage is refilled
        ptx::fence_proxy_async();
        __syncthreads();  // (A) operands of tile i ready
        if (warp == kMmaWarp && lane == 0) {
            if (i + p.nstage < ntile) issue_tile(i + p.nstage);  // stage s is free again
            ptx::tc_fence_after();
#pragma unroll
            for (int rb = 0; rb < NB; ++rb) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ad = ptx::sdesc(aK + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024);
                    const uint64_t bd = ptx::sdesc(aQ + rb * W * D * 2 + (ks / 4) * (W * 128) + (ks % 4) * 32, 16, 1024);
                    ptx::mma_f16(tS + rb * W, ad, bd, idesc1, ks > 0 ? 1u : 0u);
                }
            }
            ptx::mma_commit(bar_mma);
        }
        if (!timed_out && !ptx::mbar_wait(bar_mma, i & 1, kWaitNs)) timed_out = true;
        ptx::tc_fence_after();

        // softmax, one row block at a time (rows are independent)
        const bool valid = (t_begin + i * kTile + tok) < t_end;
        float sv[CPT];
        if (has_cols) {  // all of this thread's scores, one TMEM wait
#pragma unroll
            for (int rb = 0; rb < NB; ++rb) {
                const uint32_t ta = tS + ((uint32_t)(wq * 32) << 16) + rb * W + cgr * HC;
                if constexpr (HC == 16) {
                    uint32_t r[16];
                    ptx::tmem_ld16(ta, r);
#pragma unroll
                    for (int e = 0; e < 16; ++e) sv[rb * HC + e] = __uint_as_float(r[e]);
                } else {
                    uint32_t r[8];
                    ptx::tmem_ld8(ta, r);
#pragma unroll
                    for (int e = 0; e < 8; ++e) sv[rb * HC + e] = __uint_as_float(r[e]);
                }
            }
            ptx::tmem_wait_ld();
        }
#pragma unroll
        for (int rb = 0; rb < NB; ++rb) {
            const int colb = rb * W + cgr * HC;  // this thread's first column
            float x[HC], m[HC];
            float over = -CUDART_INF_F;
#pragma unroll
            for (int e = 0; e < HC; ++e) {
                x[e] = (valid && has_cols) ? sv[rb * HC + e] * cf : -CUDART_INF_F;
                m[e] = has_cols ? sM[colb + e] : 0.f;
                over = fmaxf(over, x[e] - m[e]);
            }
            if (ptx::bar_or(1, kWork, over > kTau)) {
                // exact maxima of this tile's rows, then raise the running maxima
                if (has_cols) {
#pragma unroll
                    for (int j = 0; j < HC; ++j) {
                        const float mx = ord2f(__reduce_max_sync(0xffffffffu, f2ord(x[j])));
                        if (lane == j) colmax[wq * 128 + colb + j] = mx;
                    }
                }
                ptx::bar_sync(1, kWork);
                float alpha[HC];
#pragma unroll
                for (int j = 0; j < HC; ++j) {
                    const int col = colb + j;
                    float mn = m[j];
                    if (has_cols)
                        mn = fmaxf(m[j], fmaxf(fmaxf(colmax[col], colmax[128 + col]),
                                              fmaxf(colmax[256 + col], colmax[384 + col])));
                    alpha[j] = (m[j] == -CUDART_INF_F) ? 0.f : ptx::ex2(m[j] - mn);
                    lp[rb * HC + j] *= alpha[j];
                    m[j] = mn;
                }
                if (i > 0 && has_cols) {  // the MMAs into O^T finished before this tile's S^T
                    const uint32_t ta = tO + ((uint32_t)(wq * 32) << 16) + colb;
#pragma unroll
                    for (int c0 = 0; c0 < HC; c0 += 8) {
                        uint32_t r8[8];
                        ptx::tmem_ld8(ta + c0, r8);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            r8[e] = __float_as_uint(__uint_as_float(r8[e]) * alpha[c0 + e]);
                        ptx::tmem_st8(ta + c0, r8);
                    }
                    ptx::tmem_wait_st();
                }
                ptx::bar_sync(1, kWork);  // every compute thread has read sM and colmax
                if (has_cols && wq == 0 && lane == 0) {
#pragma unroll
                    for (int j = 0; j < HC; ++j) sM[colb + j] = m[j];
                }
            }
            // P'^T = p * n_t / nref as fp16 hi + lo (MN-major: one 128-byte row per
            // token) and the row-sum partials of p
            if (has_cols) {
#pragma unroll
                for (int c0 = 0; c0 < HC; c0 += 8) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float pv = valid ? ptx::ex2(x[c0 + e] - m[c0 + e]) : 0.f;
                        lp[rb * HC + c0 + e] += pv;
                        const float pp = pv * ns;
                        hi[e] = __uint_as_float(__float_as_uint(pp) & 0xFFFFE000u);  // 11 significant bits
                        lo[e] = pp - hi[e];                                          // exact
                    }
                    const int chunk = (cgr * HC + c0) / 8;
                    const int off = (tok / 8) * 1024 + (tok % 8) * 128 + ((chunk ^ (tok % 8)) * 16);
                    *reinterpret_cast<uint4*>(sP + rb * 32768 + off) =
                        make_uint4(pack_h2(hi[0], hi[1]), pack_h2(hi[2], hi[3]), pack_h2(hi[4], hi[5]),
                                   pack_h2(hi[6], hi[7]));
                    *reinterpret_cast<uint4*>(sP + rb * 32768 + 16384 + off) =
                        make_uint4(pack_h2(lo[0], lo[1]), pack_h2(lo[2], lo[3]), pack_h2(lo[4], lo[5]),
                                   pack_h2(lo[6], lo[7]));
                }
            }
        }
        ptx::fence_proxy_async();
        ptx::tc_fence_before();
        __syncthreads();  // (B) P of tile i ready
        if (warp == kMmaWarp && lane == 0) {  // overlaps the other warps' next conversion
            ptx::tc_fence_after();
#pragma unroll
            for (int rb = 0; rb < NB; ++rb) {
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks) {
                    const uint64_t ad = ptx::sdesc(aV + buf * 32768 + ks * 2048, 16384, 1024);
                    const uint64_t bh = ptx::sdesc(aP + rb * 32768 + ks * 2048, 16384, 1024);
                    const uint64_t bl = ptx::sdesc(aP + rb * 32768 + 16384 + ks * 2048, 16384, 1024);
                    ptx::mma_f16(tO + rb * W, ad, bh, idesc2, (i > 0 || ks > 0) ? 1u : 0u);
                    ptx::mma_f16(tO + rb * W, ad, bl, idesc2, 1u);
                }
            }
        }
    }
    if (ntile > 0) {
        if (warp == kMmaWarp && lane == 0) ptx::mma_commit(bar_mma);
        if (!timed_out && !ptx::mbar_wait(bar_mma, ntile & 1, kWaitNs)) timed_out = true;
        ptx::tc_fence_after();
    }
    if (warp == kMmaWarp && lane == 0 && timed_out) {
        // give the copies still in flight a bounded chance to land before exit
        for (int i = max(0, ntile - p.nstage); i < ntile; ++i)
            ptx::mbar_wait(bar_full + 8 * (i % p.nstage), (i / p.nstage) & 1, kWaitNs);
    }

    // 4. epilogue: row sums and O^T to shared memory (sM already holds the maxima)
    warp_reduce_scatter<CPT>(lp, lane);
    {
        constexpr int KEEP = CPT >= 32 ? CPT / 32 : 1;  // sums kept per lane
        constexpr int REP = CPT >= 32 ? 1 : 32 / CPT;    // lanes holding the same sum
#pragma unroll
        for (int k = 0; k < KEEP; ++k) {
            const int j = lane / REP * KEEP + k;
            const int col = (j / HC) * W + cgr * HC + (j % HC);
            if (has_cols && lane % REP == 0) lsum[wq * 128 + col] = lp[k];
        }
    }
    __syncthreads();  // all MMAs have completed; sO may now alias the operands
    if (tid < RG) sL[tid] = ntile > 0 ? lsum[tid] + lsum[128 + tid] + lsum[256 + tid] + lsum[384 + tid] : 0.f;
    if (ntile > 0 && has_cols && wq * 32 < D) {  // warp-uniform
#pragma unroll
        for (int rb = 0; rb < NB; ++rb) {
#pragma unroll
            for (int c0 = 0; c0 < HC; c0 += 8) {
                uint32_t r8[8];
                ptx::tmem_ld8(tO + ((uint32_t)(wq * 32) << 16) + rb * W + cgr * HC + c0, r8);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    sO[(rb * W + cgr * HC + c0 + e) * D + tok] = __uint_as_float(r8[e]);
            }
        }
    }
    if (timed_out) atomicOr(p.status, kStTimeout);
    ptx::tc_fence_before();
    cluster.sync();  // every CTA's partial is in its shared memory

    // 5. merge the splits for the rows of owned agents (agent % S == rank),
    //    one warp per row; the walk steps over owned agents only, so the
    //    integer divisions happen once per CTA
    {
        const int G = p.G;
        const int a_first = row0 / G, a_last = (row0 + nrows - 1) / G;
        int item = 0;
        for (int a = a_first + ((crank - a_first % S) % S + S) % S; a <= a_last; a += S)
        for (int j = max(0, row0 - a * G); j < min(G, row0 + nrows - a * G); ++j) {
            if ((item++ % (kWork / 32)) != warp) continue;
            const int rr = a * G + j - row0;
            // lane s fetches CTA s's running maximum and row sum
            float Ms = -CUDART_INF_F, Ls = 0.f;
            if (lane < S) {
                Ms = ptx::ld_dsmem(ptx::dsmem_addr(sM + rr, lane));
                Ls = ptx::ld_dsmem(ptx::dsmem_addr(sL + rr, lane));
            }
            float M = (Ls > 0.f) ? Ms : -CUDART_INF_F;
#pragma unroll
            for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float wl = (Ls > 0.f) ? ptx::ex2(Ms - M) : 0.f;
            float L = wl * Ls;
#pragma unroll
            for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            // partial rows are fetched 8 CTAs at a time, all loads before any use
            float acc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
#pragma unroll
            for (int s0 = 0; s0 < 16; s0 += 8) {
                if (s0 >= S) break;
                // unconditional loads (ranks past S re-read the last CTA and get
                // weight 0) so that all eight are in flight before any is used
                float part[8][EPL];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ra = ptx::dsmem_addr(sO + rr * D + lane * EPL, min(s0 + k, S - 1));
                    if constexpr (EPL == 4) {
                        const float4 v = ptx::ld_dsmem4(ra);
                        part[k][0] = v.x; part[k][1] = v.y; part[k][2] = v.z; part[k][3] = v.w;
                    } else {
                        const float2 v = ptx::ld_dsmem2(ra);
                        part[k][0] = v.x; part[k][1] = v.y;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float w = __shfl_sync(0xffffffffu, wl, s0 + k);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w, part[k][e], acc[e]);
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
            for (int o = 1; o < 32; o <<= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float other = __shfl_xor_sync(0xffffffffu, acc[e], o);
                    acc[e] = upper ? other - acc[e] : acc[e] + other;
                }
            }
            const float oscale = nref / (float)D * p.inv_lam;
            float mt = -CUDART_INF_F, lt = 0.f;
            float* orow = p.out + ((long long)a * p.Hq + g * p.G + j) * D + lane * EPL;
            float tacc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) tacc[e] = 0.f;
            if (p.tK != nullptr) {
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
    cluster.sync();  // remote shared memory stays valid until every CTA has read it
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, p.tmem_cols);
}

template <int D, int W, int NB, int BITS>
void configure() {
    static bool done = false;
    if (done) return;
    auto kern = attend_tc_kernel<D, W, NB, BITS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    done = true;
}

// How many clusters of S CTAs with `smem` bytes each can be resident at once.
template <int D, int W, int NB, int BITS>
int max_clusters(int S, size_t smem) {
    static int cache[17][2] = {};  // [S] -> (smem key / 1024 + 1, count)
    const int key = (int)(smem / 1024) + 1;
    if (cache[S][0] == key) return cache[S][1];
    configure<D, W, NB, BITS>();
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
    if (cudaOccupancyMaxActiveClusters(&n, attend_tc_kernel<D, W, NB, BITS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[S][0] = key;
    cache[S][1] = n;
    return n;
}

template <int D, int W, int NB, int BITS>
cudaError_t launch_cfg(TcParams prm, int ntiles, int Hk, int RGN, size_t smem, cudaStream_t st) {
    configure<D, W, NB, BITS>();
    // cluster size: fewest (waves x tiles per CTA), then the larger cluster
    const int clusters = Hk * RGN;
    int bestS = 1;
    long long best = -1;
    for (int S = 1; S <= 16 && S <= ntiles; ++S) {
        const int n = max_clusters<D, W, NB, BITS>(S, smem);
        if (n < 1) continue;
        const int per = (ntiles + S - 1) / S;
        const long long waves = (clusters + n - 1) / n;
        const long long cost = waves * per;
        if (best < 0 || cost <= best) {
            best = cost;
            bestS = S;
        }
    }
    const int per = (ntiles + bestS - 1) / bestS;
    const int S = (ntiles + per - 1) / per;
    prm.tps = per * kTile;
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
    return cudaLaunchKernelEx(&cfg, attend_tc_kernel<D, W, NB, BITS>, prm);
}

}  // namespace

// Launch for layers whose V codes have BITS bits.
template <int BITS>
cudaError_t launch_attend_tc_bits(const Shape& s, const LayerBufs& L, const AttendArgs& a,
                                  int* status, cudaStream_t st) {
    const int D = s.head_dim;
    int CPT;
    if (a.rows <= 16) CPT = 8;
    else if (a.rows <= 32) CPT = 16;
    else if (a.rows <= 64) CPT = 32;
    else CPT = 64;
    const int W = CPT >= 32 ? 64 : 2 * CPT, NB = 2 * CPT / W, RG = NB * W;
    const int RGN = (a.rows + RG - 1) / RG;
    const int ntiles = (s.ctx + kTile - 1) / kTile;
    TcParams prm = {};
    prm.kq = L.kq;
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
    prm.agents = a.agents;
    prm.tK = (const uint16_t*)a.tailK;
    prm.tV = (const uint16_t*)a.tailV;
    prm.tlen = a.tail_len;
    prm.tail_max = a.tail_max;
    prm.out = a.out;
    prm.scale_log2 = a.scale_log2;
    prm.bits = BITS;
    prm.status = status;
    const Codebook& cb = codebook(BITS);
    for (int k = 0; k < 8; ++k) prm.c16[k] = (uint32_t)cb.c16[2 * k] | ((uint32_t)cb.c16[2 * k + 1] << 16);
    prm.inv_lam = 1.0f / cb.lam;
    uint32_t cols = 2 * NB * W;
    uint32_t tc = 32;
    while (tc < cols) tc <<= 1;
    prm.tmem_cols = tc;
    int nstage = 3;
    Layout lay = make_layout(D, BITS, W, NB, nstage);
    while (lay.total + 1024 > 227 * 1024 && nstage > 1) lay = make_layout(D, BITS, W, NB, --nstage);
    prm.nstage = nstage;
    const size_t smem = lay.total + 1024;
    if (D == 64) {
        if (CPT == 8) return launch_cfg<64, 16, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
        if (CPT == 16) return launch_cfg<64, 32, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
        if (CPT == 32) return launch_cfg<64, 64, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
        return launch_cfg<64, 64, 2, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
    }
    if (CPT == 8) return launch_cfg<128, 16, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
    if (CPT == 16) return launch_cfg<128, 32, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
    if (CPT == 32) return launch_cfg<128, 64, 1, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
    return launch_cfg<128, 64, 2, BITS>(prm, ntiles, s.kv_heads, RGN, smem, st);
}

}  // namespace kvp
