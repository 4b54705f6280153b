// Local attention-error estimate of one layer over the agents' recent tokens.
//
// CoMixKV article (zicq.com), "online sensitivity estimation": a local
// attention-error bound from recently observed queries, keys and values tells
// how much a layer's cache suffers from fewer bits; sharp attention needs more
// precision than flat attention. The article prints no formula; the reading
// (float64 in oracle/allocator.py): a V head-vector coded at b bits has
// E|v - v_hat|^2 = D_b |v|^2 (Lloyd-Max distortion per rotated coordinate),
// so with independent errors the relative error of a query row's output is
// sqrt(D_b) * r, r = sqrt(sum_t p_t^2 |v_t|^2) / |sum_t p_t v_t|, p the
// softmax of the row's logits over the agent's recent tokens. The layer's
// sensitivity is the mean of r over all (agent, query head) rows; rows of an
// agent with no recent token count as 0.
//
// Kernels: one CTA per query row (logits, softmax weights, sum of p^2 |v|^2
// and |o| with unnormalised weights, in which r is the same), then one CTA
// that averages the rows in a fixed order (deterministic).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

constexpr int kSensThreads = 128;

__device__ __forceinline__ float bf(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

// CTA-wide reductions over kSensThreads threads through `red` (4 floats)
__device__ __forceinline__ float cta_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = v;
    __syncthreads();
    return (red[0] + red[1]) + (red[2] + red[3]);
}
__device__ __forceinline__ float cta_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = v;
    __syncthreads();
    return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

// grid: agents * q_heads rows; dynamic shared memory: T_max floats
template <int D>
__global__ void __launch_bounds__(kSensThreads)
row_ratio_kernel(const uint16_t* __restrict__ Q, const uint16_t* __restrict__ tK,
                 const uint16_t* __restrict__ tV, const int32_t* __restrict__ tlen, int T_max, int Hq,
                 int Hk, float scale, float* __restrict__ row_r) {
    extern __shared__ float w[];  // [T_max] logits, then weights
    __shared__ float qs[D];
    __shared__ float red[4];
    const int row = blockIdx.x, a = row / Hq, h = row % Hq, g = h / (Hq / Hk);
    const int tid = threadIdx.x;
    const int T = min(max(tlen[a], 0), T_max);
    for (int c = tid; c < D; c += kSensThreads) qs[c] = bf(Q[(long long)row * D + c]);
    __syncthreads();
    const long long base = ((long long)a * Hk + g) * T_max;
    // logits and their maximum
    float m = -CUDART_INF_F;
    for (int t = tid; t < T; t += kSensThreads) {
        const uint16_t* k = tK + (base + t) * D;
        float dot = 0.f;
        for (int c = 0; c < D; ++c) dot = fmaf(qs[c], bf(k[c]), dot);
        w[t] = dot * scale;
        m = fmaxf(m, w[t]);
    }
    m = cta_max(m, red);
    // unnormalised weights p_t = exp(l_t - m) and sum_t p_t^2 |v_t|^2
    float num = 0.f;
    for (int t = tid; t < T; t += kSensThreads) {
        const float p = __expf(w[t] - m);
        w[t] = p;
        const uint16_t* v = tV + (base + t) * D;
        float vv = 0.f;
        for (int c = 0; c < D; ++c) {
            const float x = bf(v[c]);
            vv = fmaf(x, x, vv);
        }
        num = fmaf(p * p, vv, num);
    }
    num = cta_sum(num, red);  // its barriers also publish w[]
    // |o|^2 with o = sum_t p_t v_t, thread = channel
    float oo = 0.f;
    for (int c = tid; c < D; c += kSensThreads) {
        float o = 0.f;
        for (int t = 0; t < T; ++t) o = fmaf(w[t], bf(tV[(base + t) * D + c]), o);
        oo = fmaf(o, o, oo);
    }
    oo = cta_sum(oo, red);
    if (tid == 0) row_r[row] = (T > 0 && oo > 0.f) ? sqrtf(num) / sqrtf(oo) : 0.f;
}

// one CTA: score = mean of rows[0..n), summed in a fixed order
__global__ void __launch_bounds__(kSensThreads) mean_kernel(const float* __restrict__ rows, int n,
                                                           float* __restrict__ score) {
    __shared__ float red[4];
    float s = 0.f;
    for (int i = threadIdx.x; i < n; i += kSensThreads) s += rows[i];
    s = cta_sum(s, red);
    if (threadIdx.x == 0) *score = s / (float)n;
}

}  // namespace

cudaError_t launch_sensitivity(const void* Q, int agents, int q_heads, int kv_heads, int head_dim,
                               const void* tK, const void* tV, const int32_t* tlen, int T_max, float scale,
                               float* row_r, float* score, cudaStream_t st) {
    const int rows = agents * q_heads;
    const size_t smem = (size_t)T_max * sizeof(float);
    if (head_dim == 64)
        row_ratio_kernel<64><<<rows, kSensThreads, smem, st>>>((const uint16_t*)Q, (const uint16_t*)tK,
                                                               (const uint16_t*)tV, tlen, T_max, q_heads,
                                                               kv_heads, scale, row_r);
    else
        row_ratio_kernel<128><<<rows, kSensThreads, smem, st>>>((const uint16_t*)Q, (const uint16_t*)tK,
                                                                (const uint16_t*)tV, tlen, T_max, q_heads,
                                                                kv_heads, scale, row_r);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    mean_kernel<<<1, kSensThreads, 0, st>>>(row_r, rows, score);
    return cudaGetLastError();
}

}  // namespace kvp
