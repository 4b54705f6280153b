// Decode attention of many agents directly over the shared pool.
//
// PolyKV summary, section 2.A: every agent reads the same compressed pool;
// section 2.B: K = q * s, V = n * H c[codes] / d. Instead of materialising V
// per agent, the pool is streamed once per step for all agents that share a
// KV head, and P.V is accumulated in the rotated domain:
//   sum_t p_t V_t = H (sum_t p_t n_t c[codes_t]) / d,
// so the inverse FWHT runs once per output row instead of once per token.
// The private bf16 tail of each agent (CoMixKV article: recent states stay at
// native precision) joins the same softmax.
//
// CUDA-core path (split context):
//   attend_split: grid (context split, kv head, row block). A CTA walks its
//     token range in tiles of 32 tokens (one V code group of the pool
//     layout): K int8 and the V codes are expanded
//     to float32 in shared memory (V already scaled by its norm), then each
//     warp runs an online softmax for its rows (lane = token for the logits,
//     lane = channel for the rotated accumulator). It writes (m, l, acc) per
//     row for its split.
//   attend_combine: one CTA per (row, kv head): log-sum-exp merge of the
//     splits, inverse FWHT / d, the agent's tail tokens, final normalisation.
//   merge_rows: the same merge with one warp per (row, kv head), for the
//     context slices of kvpool_attend_partial (kvpool_merge_partials) and of
//     kvpool_attend_ws, the partials laid out by slice.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

constexpr int kTileTok = 32;
constexpr int kRowsPerWarp = 2;
constexpr int kWarps = 8;
constexpr int kRowsPerBlock = kRowsPerWarp * kWarps;

__device__ __forceinline__ float bf2f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D, int BITS>
__global__ void __launch_bounds__(kWarps * 32)
attend_split_kernel(const int8_t* __restrict__ kq, const uint8_t* __restrict__ vcodes,
                    const float* __restrict__ vnorm, const float* __restrict__ kscale,
                    const float* __restrict__ kscales, int ctx,
                    int ctx_pad, const uint16_t* __restrict__ Q, int Hq, int G, int R,
                    float scale_log2, int tok_per_split, float* __restrict__ part_acc,
                    float* __restrict__ part_ml, int nsplit, int max_rows, Codebook cb) {
    constexpr int VB = D * BITS / 8;
    constexpr uint32_t MASK = (1u << BITS) - 1;
    constexpr int DPL = D / 32;  // channels per lane
    __shared__ float Ks[kTileTok][D + 1];
    __shared__ float Vs[kTileTok][D];
    __shared__ float Qs[kRowsPerBlock][D];
    __shared__ float cen[16];

    const int split = blockIdx.x, g = blockIdx.y, rb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < kRowsPerBlock * D; i += blockDim.x) {
        const int rr = i / D, c = i % D, r = rb * kRowsPerBlock + rr;
        float val = 0.f;
        if (r < R) {
            const int a = r / G, j = r % G;
            val = bf2f(Q[((long long)a * Hq + g * G + j) * D + c]);
        }
        Qs[rr][c] = val;
    }
    if (tid < 16) cen[tid] = cb.c[tid];

    const float lscale = *kscale * scale_log2;
    const int t_begin = split * tok_per_split;
    const int t_end = min(ctx, t_begin + tok_per_split);
    const int8_t* kbase = kq + (long long)g * ctx_pad * D;
    const uint8_t* vbase = vcodes + (long long)g * ctx_pad * VB;
    const float* nbase = vnorm + (long long)g * ctx_pad;

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -CUDART_INF_F;
        l[r] = 0.f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[r][k] = 0.f;
    }
    __syncthreads();

    for (int t0 = t_begin; t0 < t_end; t0 += kTileTok) {
        // K tile: int8 -> float (the layer's scale s joins the logit scale; a
        // block-scaled pool's 32-element scales multiply here, s being 1)
        for (int i = tid; i < kTileTok * D / 16; i += blockDim.x) {
            const int tt = i / (D / 16), c = i % (D / 16);
            const uint4 w = *reinterpret_cast<const uint4*>(kbase + (long long)(t0 + tt) * D + c * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            const float sb = kscales ? kscales[((long long)g * ctx_pad + t0 + tt) * (D / 32) + c / 2] : 1.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                Ks[tt][c * 16 + e] = (float)(int8_t)((ws[e / 4] >> (8 * (e % 4))) & 0xFF) * sb;
        }
        // V tile (one 32-token code group, t0 % 32 == 0): a task is 8 tokens of
        // one coordinate, BITS bytes of that coordinate's code sequence -> n_t * c[code]
        const uint8_t* grp = vbase + (long long)t0 * VB;
        for (int i = tid; i < 4 * D; i += blockDim.x) {
            const int ch = i / D, c = i % D;
            const uint8_t* p = grp + c * (4 * BITS) + ch * BITS;
            uint32_t word = 0;
#pragma unroll
            for (int b = 0; b < BITS; ++b) word |= (uint32_t)p[b] << (8 * b);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int t = t0 + ch * 8 + k;  // slots past the range hold 0 (their p is 0)
                Vs[ch * 8 + k][c] = t < t_end ? cen[(word >> (BITS * k)) & MASK] * nbase[t] : 0.f;
            }
        }
        __syncthreads();

        const bool valid = (t0 + lane) < t_end;
#pragma unroll
        for (int r4 = 0; r4 < kRowsPerWarp; ++r4) {
            const int rr = warp * kRowsPerWarp + r4;
            float dot = 0.f;
#pragma unroll 16
            for (int i = 0; i < D; ++i) dot = fmaf(Qs[rr][i], Ks[lane][i], dot);
            const float lg = valid ? __fmul_rn(dot, lscale) : -CUDART_INF_F;  // never fused with - m
            const float mnew = fmaxf(m[r4], warp_max(lg));
            if (mnew == -CUDART_INF_F) continue;  // warp-uniform
            const float corr = exp2f(m[r4] - mnew);
            const float p = exp2f(lg - mnew);
            l[r4] = l[r4] * corr + warp_sum(p);
            m[r4] = mnew;
#pragma unroll
            for (int k = 0; k < DPL; ++k) acc[r4][k] *= corr;
#pragma unroll 8
            for (int tt = 0; tt < kTileTok; ++tt) {
                const float pt = __shfl_sync(0xffffffffu, p, tt);
#pragma unroll
                for (int k = 0; k < DPL; ++k) acc[r4][k] = fmaf(pt, Vs[tt][lane + 32 * k], acc[r4][k]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int r4 = 0; r4 < kRowsPerWarp; ++r4) {
        const int r = rb * kRowsPerBlock + warp * kRowsPerWarp + r4;
        if (r >= R) continue;
        const long long base = ((long long)g * nsplit + split) * max_rows + r;
        if (lane == 0) {
            part_ml[2 * base] = m[r4];
            part_ml[2 * base + 1] = l[r4];
        }
#pragma unroll
        for (int k = 0; k < DPL; ++k) part_acc[base * D + lane + 32 * k] = acc[r4][k];
    }
}

template <int D>
__global__ void __launch_bounds__(D)
attend_combine_kernel(const float* __restrict__ part_acc, const float* __restrict__ part_ml,
                      int nsplit, long long head_stride, long long split_stride, int Hk, int Hq, int G,
                      const uint16_t* __restrict__ Q, const uint16_t* __restrict__ tK,
                      const uint16_t* __restrict__ tV, const int32_t* __restrict__ tlen,
                      int tail_max, float scale_log2, float* __restrict__ out) {
    __shared__ float x[D];
    __shared__ float red[D / 32];
    const int r = blockIdx.x, g = blockIdx.y, i = threadIdx.x;
    const int a = r / G, h = g * G + r % G;

    // merge the splits (log2 domain)
    float M = -CUDART_INF_F;
    for (int s = 0; s < nsplit; ++s) {
        const long long b = g * head_stride + s * split_stride + r;
        if (part_ml[2 * b + 1] > 0.f) M = fmaxf(M, part_ml[2 * b]);
    }
    float L = 0.f, acc = 0.f;
    for (int s = 0; s < nsplit; ++s) {
        const long long b = g * head_stride + s * split_stride + r;
        const float ls = part_ml[2 * b + 1];
        if (ls > 0.f) {
            const float w = exp2f(part_ml[2 * b] - M);
            L += ls * w;
            acc += part_acc[b * D + i] * w;
        }
    }
    // inverse rotation: H acc / D
    x[i] = acc;
    __syncthreads();
#pragma unroll
    for (int hh = 1; hh < D; hh <<= 1) {
        if (!(i & hh)) {
            const float u = x[i], v = x[i + hh];
            x[i] = u + v;
            x[i + hh] = u - v;
        }
        __syncthreads();
    }
    const float Opool = x[i] * (1.0f / (float)D);

    // private tail of agent a for kv head g
    float mt = -CUDART_INF_F, lt = 0.f, Ot = 0.f;
    if (tK != nullptr) {
        const int n = min(max(tlen[a], 0), tail_max);  // never read past the tail buffers
        const float q = bf2f(Q[((long long)a * Hq + h) * D + i]);
        const long long tb = ((long long)a * Hk + g) * tail_max;
        for (int t = 0; t < n; ++t) {
            float part = warp_sum(q * bf2f(tK[(tb + t) * D + i]));
            if ((i & 31) == 0) red[i / 32] = part;
            __syncthreads();
            float dot = 0.f;
#pragma unroll
            for (int w = 0; w < D / 32; ++w) dot += red[w];
            __syncthreads();
            const float lg = __fmul_rn(dot, scale_log2);
            const float mnew = fmaxf(mt, lg);
            const float corr = exp2f(mt - mnew), p = exp2f(lg - mnew);
            lt = lt * corr + p;
            Ot = Ot * corr + p * bf2f(tV[(tb + t) * D + i]);
            mt = mnew;
        }
    }
    const float Mf = fmaxf(M, mt);
    const float wp = (L > 0.f) ? exp2f(M - Mf) : 0.f;
    const float wt = (lt > 0.f) ? exp2f(mt - Mf) : 0.f;
    out[((long long)a * Hq + h) * D + i] = (Opool * wp + Ot * wt) / (L * wp + lt * wt);
}

// kvpool_merge_partials and the merge of kvpool_attend_ws: one warp per
// (row, KV head), lane = D/32 consecutive channels. The slices' (m, l) are
// read by the lanes at once with the first 20 slices' accumulators, the
// accumulators of any further slices four at a time; one
// inverse FWHT per row in registers and shuffles; then the agent's tail
// tokens (online softmax) and the final normalisation. Launched as a
// programmatic dependent of the kernel that wrote the partials. It releases
// its own dependents before its grid-dependency wait: the next layer's
// attention CTAs then start while this merge waits, and reach their own wait
// with their pool tiles already requested. Their wait still covers this
// kernel's completion, which follows the partials' writer; what they read
// before it (pool bytes) neither kernel writes.
template <int D>
__global__ void __launch_bounds__(512)
merge_rows_kernel(const float* __restrict__ part_acc, const float* __restrict__ part_ml, int nsplit, int R,
                  int Hk, int Hq, int G, const uint16_t* __restrict__ Q, const uint16_t* __restrict__ tK,
                  const uint16_t* __restrict__ tV, const int32_t* __restrict__ tlen, int tail_max,
                  float scale_log2, float* __restrict__ out, const float* __restrict__ tail_ml) {
    constexpr int EPL = D / 32;
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x % 32;
    const int r = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, g = blockIdx.y;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (r >= R) return;
    const long long stride = (long long)Hk * R;  // between slices
    const long long b0 = (long long)g * R + r;
    // one round trip: lane s's (m, l) of slice s and the accumulators of the
    // first kFirst slices are all requested before any is used
    constexpr int kFirst = 20;
    const float2 ml0 = lane < nsplit ? *reinterpret_cast<const float2*>(part_ml + 2 * (b0 + lane * stride))
                                     : make_float2(-CUDART_INF_F, 0.f);
    float v[kFirst][EPL];
#pragma unroll
    for (int u = 0; u < kFirst; ++u) {
        const float* src = part_acc + (b0 + (long long)u * stride) * D + lane * EPL;
        if (u < nsplit) {
            if constexpr (EPL == 4) {
                const float4 x = *reinterpret_cast<const float4*>(src);
                v[u][0] = x.x, v[u][1] = x.y, v[u][2] = x.z, v[u][3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2*>(src);
                v[u][0] = x.x, v[u][1] = x.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) v[u][e] = 0.f;
        }
    }
    float M = ml0.y > 0.f ? ml0.x : -CUDART_INF_F;
    for (int s = lane + 32; s < nsplit; s += 32) {
        const float2 ml = *reinterpret_cast<const float2*>(part_ml + 2 * (b0 + s * stride));
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    M = warp_max(M);
    float L = 0.f;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float w = ml0.y > 0.f ? exp2f(ml0.x - M) : 0.f;  // slice `lane`
    L += w * ml0.y;
#pragma unroll
    for (int u = 0; u < kFirst; ++u) {
        const float wu = __shfl_sync(full, w, u);  // 0 past nsplit and for empty slices
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = wu != 0.f ? fmaf(wu, v[u][e], acc[e]) : acc[e];
    }
    // slices from kFirst on (more than kFirst slices), four at a time
    for (int s0 = kFirst; s0 < nsplit; s0 += 4) {
        float ww[4], x[4][EPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int s = s0 + u;
            float wl = 0.f;
            if (s < nsplit && s >= 32) {  // slices below 32 have their weight in lane s
                const float2 ml = *reinterpret_cast<const float2*>(part_ml + 2 * (b0 + s * stride));
                wl = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
                if (lane == 0) L += wl * ml.y;  // counted once
            }
            ww[u] = s < 32 ? __shfl_sync(full, w, s & 31) : wl;
            if (s >= nsplit) ww[u] = 0.f;
            const float* src = part_acc + (b0 + (long long)s * stride) * D + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[u][e] = ww[u] != 0.f ? src[e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = ww[u] != 0.f ? fmaf(ww[u], x[u][e], acc[e]) : acc[e];
    }
    L = warp_sum(L);
    // inverse rotation H acc / D: channel lane * EPL + e
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
            const float other = __shfl_xor_sync(full, acc[e], o2);
            acc[e] = upper ? other - acc[e] : acc[e] + other;
        }
    }
    const int a = r / G, h = g * G + r % G;
    float mt = -CUDART_INF_F, lt = 0.f, ot[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) ot[e] = 0.f;
    if (tail_ml != nullptr) {
        // tails computed by the attention kernel: (m, l) here, the
        // unnormalised accumulator in the output row
        const float2 t = *reinterpret_cast<const float2*>(tail_ml + 2 * b0);
        mt = t.x;
        lt = t.y;
        if (lt > 0.f) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) ot[e] = out[((long long)a * Hq + h) * D + lane * EPL + e];
        }
    } else if (tK != nullptr) {
        // the agent's tail, 32 tokens at a time: lane = token for the logits
        // (the Q row in shared memory, read by every lane at once), then lane
        // = channels for P.V; online softmax over the chunks
        __shared__ float sq[16][D];
        const int wi = threadIdx.x / 32;
        const int n = min(max(tlen[a], 0), tail_max);  // never read past the tail buffers
#pragma unroll
        for (int e = 0; e < EPL; ++e) sq[wi][lane * EPL + e] = bf2f(Q[((long long)a * Hq + h) * D + lane * EPL + e]);
        __syncwarp();
        const long long tb = ((long long)a * Hk + g) * tail_max;
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int t = c0 + lane;
            float lg = -CUDART_INF_F;
            if (t < n) {
                const uint4* kr = reinterpret_cast<const uint4*>(tK + (tb + t) * D);
                float dot = 0.f;
#pragma unroll 8
                for (int cc = 0; cc < D / 8; ++cc) {
                    const uint4 u = kr[cc];
                    const float* qq = sq[wi] + cc * 8;
                    dot = fmaf(qq[0], bf2f(u.x & 0xFFFF), dot);
                    dot = fmaf(qq[1], bf2f(u.x >> 16), dot);
                    dot = fmaf(qq[2], bf2f(u.y & 0xFFFF), dot);
                    dot = fmaf(qq[3], bf2f(u.y >> 16), dot);
                    dot = fmaf(qq[4], bf2f(u.z & 0xFFFF), dot);
                    dot = fmaf(qq[5], bf2f(u.z >> 16), dot);
                    dot = fmaf(qq[6], bf2f(u.w & 0xFFFF), dot);
                    dot = fmaf(qq[7], bf2f(u.w >> 16), dot);
                }
                lg = __fmul_rn(dot, scale_log2);
            }
            const float mnew = fmaxf(mt, warp_max(lg));
            const float corr = exp2f(mt - mnew);  // 0 on the first chunk
            const float pt = t < n ? exp2f(lg - mnew) : 0.f;
            lt = lt * corr + warp_sum(pt);
#pragma unroll
            for (int e = 0; e < EPL; ++e) ot[e] *= corr;
            const int nk = min(32, n - c0);
            for (int k0 = 0; k0 < nk; k0 += 8) {  // eight V rows in flight at a time
                float pk[8];
                uint2 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    pk[u] = __shfl_sync(full, pt, (k0 + u) & 31);  // 0 past the tail
                    const uint16_t* vr = tV + (tb + c0 + k0 + u) * D + lane * EPL;
                    v[u] = make_uint2(0u, 0u);
                    if (k0 + u < nk) {
                        if constexpr (EPL == 4) v[u] = *reinterpret_cast<const uint2*>(vr);
                        else v[u].x = *reinterpret_cast<const uint32_t*>(vr);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    ot[0] = fmaf(pk[u], bf2f(v[u].x & 0xFFFF), ot[0]);
                    ot[1] = fmaf(pk[u], bf2f(v[u].x >> 16), ot[1]);
                    if constexpr (EPL == 4) {
                        ot[2] = fmaf(pk[u], bf2f(v[u].y & 0xFFFF), ot[2]);
                        ot[3] = fmaf(pk[u], bf2f(v[u].y >> 16), ot[3]);
                    }
                }
            }
            mt = mnew;
        }
    }
    const float Mf = fmaxf(M, mt);
    const float wp = (L > 0.f) ? exp2f(M - Mf) : 0.f;
    const float wt = (lt > 0.f) ? exp2f(mt - Mf) : 0.f;
    const float den = L * wp + lt * wt;
    float* orow = out + ((long long)a * Hq + h) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) orow[e] = (acc[e] * (1.0f / (float)D) * wp + ot[e] * wt) / den;
}

template <int D, int BITS>
cudaError_t run(const Shape& s, const LayerBufs& Lb, const AttendArgs& a, const AttendScratch& scr,
                cudaStream_t st) {
    const int ntile = (s.ctx + kTileTok - 1) / kTileTok;
    const int per = (ntile + scr.nsplit - 1) / scr.nsplit;
    const int tok_per_split = per * kTileTok;
    const int nsplit = (s.ctx + tok_per_split - 1) / tok_per_split;
    dim3 grid(nsplit, s.kv_heads, (a.rows + kRowsPerBlock - 1) / kRowsPerBlock);
    attend_split_kernel<D, BITS><<<grid, kWarps * 32, 0, st>>>(
        Lb.kq, Lb.vcodes, Lb.vnorm, Lb.kscale, Lb.kscales, s.ctx, s.ctx_pad, (const uint16_t*)a.Q, a.q_heads,
        a.group, a.rows, a.scale_log2, tok_per_split, scr.acc, scr.ml, nsplit, scr.max_rows,
        codebook(BITS));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attend_combine_kernel<D><<<dim3(a.rows, s.kv_heads), D, 0, st>>>(
        scr.acc, scr.ml, nsplit, (long long)nsplit * scr.max_rows, scr.max_rows, s.kv_heads, a.q_heads, a.group,
        (const uint16_t*)a.Q, (const uint16_t*)a.tailK, (const uint16_t*)a.tailV, a.tail_len,
        a.tail_max, a.scale_log2, a.out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_partials(int parts, const float* part_ml, const float* part_acc, int kv_heads,
                                  int head_dim, const AttendArgs& a, cudaStream_t st, int sm_count) {
    // 8 warps (rows) per CTA; 16 where that puts a grid of more than one
    // wave into one
    int wpc = 8;
    if (sm_count > 0 && (long long)((a.rows + 7) / 8) * kv_heads > sm_count &&
        (long long)((a.rows + 15) / 16) * kv_heads <= sm_count)
        wpc = 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.rows + wpc - 1) / wpc, kv_heads, 1);
    cfg.blockDim = dim3(32 * wpc, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = head_dim == 64 ? merge_rows_kernel<64> : merge_rows_kernel<128>;
    // The merge starts early, while the attention kernel still holds most
    // SMs: its CTAs would all land on the few SMs left free and share their
    // load bandwidth for the partial states. When the grid fits one wave and
    // the partial states are large (1 MiB or more), each CTA reserves more
    // than half of an SM's shared memory (unused), so at most one CTA runs
    // per SM and the rest start on the SMs the attention CTAs release. (With
    // small partial states the free SMs load them fast enough, and the CTAs
    // that would wait for a released SM only start later.)
    constexpr int kSpreadSmem = 120 * 1024;
    const size_t part_bytes = (size_t)parts * kv_heads * a.rows * (head_dim + 2) * sizeof(float);
    if (sm_count > 0 && (long long)cfg.gridDim.x * cfg.gridDim.y <= sm_count && part_bytes >= (size_t(1) << 20)) {
        // opted in once per instance (a static initialiser: thread-safe)
        static const cudaError_t opt64 =
            cudaFuncSetAttribute(merge_rows_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpreadSmem);
        static const cudaError_t opt128 =
            cudaFuncSetAttribute(merge_rows_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpreadSmem);
        const cudaError_t opt = head_dim == 64 ? opt64 : opt128;
        if (opt != cudaSuccess) return opt;
        cfg.dynamicSmemBytes = kSpreadSmem;
    }
    return cudaLaunchKernelEx(&cfg, kern, part_acc, part_ml, parts, a.rows, kv_heads, a.q_heads, a.group,
                              (const uint16_t*)a.Q, (const uint16_t*)a.tailK, (const uint16_t*)a.tailV, a.tail_len,
                              a.tail_max, a.scale_log2, a.out, (const float*)a.ws_tail_ml);
}

cudaError_t launch_attend_split(const Shape& s, const LayerBufs& L, const AttendArgs& a,
                                const AttendScratch& scr, cudaStream_t st) {
    if (s.head_dim == 64) {
        if (L.bits == 2) return run<64, 2>(s, L, a, scr, st);
        if (L.bits == 3) return run<64, 3>(s, L, a, scr, st);
        return run<64, 4>(s, L, a, scr, st);
    }
    if (L.bits == 2) return run<128, 2>(s, L, a, scr, st);
    if (L.bits == 3) return run<128, 3>(s, L, a, scr, st);
    return run<128, 4>(s, L, a, scr, st);
}

}  // namespace kvp
