// Write-once encode of one pool layer.
//
// PolyKV summary (gist.science, "PolyKV: A Shared Asymmetrically-Compressed
// KV Cache Pool for Multi-Agent LLM Inference"), section 2.B:
//   K: per-tensor linear quantisation to int8.
//   V: FWHT rotation of each head-vector, then the nearest Lloyd-Max centroid
//      for N(0,1) per rotated coordinate (3 bits; 2 or 4 bits per layer in the
//      CoMixKV article's mixed-precision setting).
//
// Two kernels:
//   encode_v_kmax: D/32 threads per head-vector, 32 coordinates each, loaded
//     straight from global memory with coalesced 16-byte loads; grid (token
//     chunks, kv heads). On the way it reduces max|K| over the same
//     coordinates of K and the largest norm of the layer (per CTA, then one
//     atomicMax per CTA only while the CTA's value is still larger).
//     Per vector: the norm by the pairwise tree (the first levels cross
//     threads by shuffles), the FWHT (stages h < 32 in registers, h = 32, 64
//     by shfl.xor), one float32 threshold per midpoint (m_j * n), the codes by
//     a branchless binary search over the sorted thresholds. The codes are
//     then regrouped through shared memory into the pool layout: per group of
//     32 tokens, one packed sequence per coordinate (the 32 tokens' codes in
//     token order, 4*BITS bytes), so that a reader holding one coordinate of
//     many tokens finds them in consecutive bytes.
//   encode_k_pack: s = max|K| / 127, q = clamp(rint(k / s), -127, 127), 16
//     elements per thread. k / s is formed as k * (1/s) and the correctly
//     rounded quotient is recomputed with an IEEE division only when the
//     product lies within 2^-15 of a half-integer, where the two could round
//     to different integers; elsewhere both give the same q.
// Every float operation that decides a code uses an explicit IEEE round-to-
// nearest intrinsic, in the fixed order of the definition, so the codes are
// reproducible bit for bit (no contraction into FMA, no approximate division).
#include <cuda_bf16.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

constexpr int kEncThreads = 256;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// number of thresholds below x (thresholds ascending): branchless binary search
template <int L>
__device__ __forceinline__ uint32_t bucket(float x, const float (&t)[16]) {
    if constexpr (L == 4) {
        const uint32_t b1 = x > t[1];
        const uint32_t b0 = x > (b1 ? t[2] : t[0]);
        return 2 * b1 + b0;
    } else if constexpr (L == 8) {
        const uint32_t b2 = x > t[3];
        const uint32_t b1 = x > (b2 ? t[5] : t[1]);
        const float t0 = b2 ? (b1 ? t[6] : t[4]) : (b1 ? t[2] : t[0]);
        const uint32_t b0 = x > t0;
        return 4 * b2 + 2 * b1 + b0;
    } else {
        const uint32_t b3 = x > t[7];
        const uint32_t b2 = x > (b3 ? t[11] : t[3]);
        const int base2 = 8 * b3 + 4 * b2;
        const float tm = (base2 == 0) ? t[1] : (base2 == 4) ? t[5] : (base2 == 8) ? t[9] : t[13];
        const uint32_t b1 = x > tm;
        const int base1 = base2 + 2 * b1;
        float tl = t[0];
#pragma unroll
        for (int k = 2; k < 16; k += 2) tl = (base1 == k) ? t[k] : tl;
        const uint32_t b0 = x > tl;
        return base1 + b0;
    }
}

// Raise *word to the maximum of `val` over the CTA: warp redux, then one
// thread per CTA, and an atomic only when the word is still smaller (the
// maximum stabilises after a few CTAs, so almost all CTAs skip the atomic).
__device__ __forceinline__ void cta_max_to(uint32_t val, uint32_t* word, uint32_t* red) {
    val = __reduce_max_sync(0xffffffffu, val);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = val;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
        for (int w = 0; w < (int)(blockDim.x / 32); ++w) m = max(m, red[w]);
        if (m > *reinterpret_cast<volatile uint32_t*>(word)) atomicMax(word, m);
    }
}

// grid: (token chunks, kv heads)
template <int D, int BITS>
__global__ void __launch_bounds__(kEncThreads)
encode_v_kmax_kernel(const uint4* __restrict__ K, const uint4* __restrict__ V, int ctx, int ctx_pad,
                     uint8_t* __restrict__ vcodes, float* __restrict__ vnorm,
                     uint32_t* __restrict__ scratch, int* __restrict__ status, Codebook cb) {
    constexpr int TPV = D / 32;          // threads per head-vector
    constexpr int L = 1 << BITS;
    __shared__ uint32_t red[2][kEncThreads / 32];
    constexpr int VPB = kEncThreads / TPV;  // head-vectors per block (a multiple of 32)
    __shared__ __align__(16) uint8_t codes8[VPB * D];
    const int tid = threadIdx.x, lane = tid % 32;
    const int lt = tid % TPV;            // this thread's 32-coordinate slice
    const int t = blockIdx.x * (kEncThreads / TPV) + tid / TPV;  // token
    const bool live = t < ctx;
    const long long v = (long long)blockIdx.y * ctx + t;         // input head-vector
    const unsigned gmask = 0xffffffffu;

    // 1. load 32 coordinates of V and K
    uint4 vv[4], kk[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        vv[c] = live ? __ldg(V + v * (D / 8) + lt * 4 + c) : make_uint4(0, 0, 0, 0);
        kk[c] = live ? __ldg(K + v * (D / 8) + lt * 4 + c) : make_uint4(0, 0, 0, 0);
    }
    uint32_t kmax = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t m = 0x7FFF7FFFu;
        const uint32_t a = __vmaxu2(__vmaxu2(kk[c].x & m, kk[c].y & m), __vmaxu2(kk[c].z & m, kk[c].w & m));
        kmax = max(kmax, max(a & 0xFFFFu, a >> 16));
    }
    // |bf16| bit patterns order like their values; Inf/NaN patterns exceed
    // every finite one, so a non-finite K survives the maximum.
    cta_max_to(kmax, &scratch[0], red[0]);

    float x[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {vv[c].x, vv[c].y, vv[c].z, vv[c].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[c * 8 + 2 * j] = bf_lo(w[j]);
            x[c * 8 + 2 * j + 1] = bf_hi(w[j]);
        }
    }

    // 2. norm: pairwise tree sq_i += sq_{i+w}, w = D/2, ..., 1 (squares exact)
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = __fmul_rn(x[i], x[i]);
    // levels w >= 32 pair slices lt and lt + w/32 (the lower slice keeps the sum)
#pragma unroll
    for (int w = D / 2; w >= 32; w >>= 1) {
        const int off = w / 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float o = __shfl_down_sync(gmask, s[i], off, TPV);
            s[i] = __fadd_rn(s[i], o);  // meaningful on slices lt < off
        }
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) s[i] = __fadd_rn(s[i], s[i + w]);
    }
    const float n = __shfl_sync(gmask, __fsqrt_rn(s[0]), lane - lt);  // slice 0 holds the sum
    cta_max_to(__float_as_uint(n), &scratch[1], red[1]);  // largest norm of the layer

    // 3. FWHT, stages h = 1, 2, ..., D/2, lower index first
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (!(i & h)) {
                const float a = x[i], b = x[i + h];
                x[i] = __fadd_rn(a, b);
                x[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int h = 32; h < D; h <<= 1) {
        const int off = h / 32;
        const bool upper = (lt & off) != 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float o = __shfl_xor_sync(gmask, x[i], off, TPV);
            // lower slice: own + partner; upper slice: partner (lower) - own
            x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
        }
    }

    // 4. thresholds m_j * n, 5. codes = number of thresholds exceeded (0 past the context)
    float tau[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) tau[j] = (j < L - 1) ? __fmul_rn(cb.m[j], n) : 0.f;
    uint32_t cw[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) cw[w] = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t code = live ? bucket<L>(x[i], tau) : 0u;
        cw[i / 4] |= code << (8 * (i % 4));
    }
    // this slice's codes as bytes [token][coordinate] in shared memory
    uint4* c8 = reinterpret_cast<uint4*>(codes8 + (tid / TPV) * D + lt * 32);
    c8[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    c8[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    if (live && lt == 0) {
        vnorm[(long long)blockIdx.y * ctx_pad + t] = n;
        if (!isfinite(n)) atomicOr(status, kStNonfinite);
    }
    __syncthreads();

    // 6. pool layout: one thread per (32-token group of this block, coordinate)
    //    packs the group's 32 codes of that coordinate, in token order
    {
        const int gq = tid / D, c = tid % D;
        uint32_t words[BITS + 1];
#pragma unroll
        for (int w = 0; w <= BITS; ++w) words[w] = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t code = codes8[(gq * 32 + j) * D + c];
            const int bit = j * BITS, w = bit / 32, off = bit % 32;
            words[w] |= code << off;
            if (off + BITS > 32) words[w + 1] |= code >> (32 - off);
        }
        const long long grp = ((long long)blockIdx.y * ctx_pad + (long long)blockIdx.x * VPB) / 32 + gq;
        uint32_t* out = reinterpret_cast<uint32_t*>(vcodes + (grp * D + c) * (4 * BITS));
#pragma unroll
        for (int w = 0; w < BITS; ++w) out[w] = words[w];
    }
}

// grid: (chunks of 16-element groups, kv heads)
template <int D>
__global__ void __launch_bounds__(256)
encode_k_pack_kernel(const uint4* __restrict__ K, int ctx, int ctx_pad, int8_t* __restrict__ kq,
                     const uint32_t* __restrict__ kabsmax, float* __restrict__ kscale,
                     int* __restrict__ status) {
    const uint32_t am = *kabsmax;
    const float s = (am == 0) ? 1.0f : __fdiv_rn(__uint_as_float(am << 16), 127.0f);
    const float r = __frcp_rn(s);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        *kscale = s;
        if (am >= 0x7F80u) atomicOr(status, kStNonfinite);
    }
    const int g = blockIdx.x * blockDim.x + threadIdx.x;  // 16-element group within the head
    if (g < ctx * (D / 16)) {
        const long long src = (long long)blockIdx.y * ctx * (D / 8) + 2LL * g;
        const uint4 a = __ldg(K + src), b = __ldg(K + src + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float k = (j & 1) ? bf_hi(w[j / 2]) : bf_lo(w[j / 2]);
            // k * (1/s) is within ~1.5 ulp of k / s; unless that lands within
            // 2^-15 of a half-integer both round to the same integer
            float y = __fmul_rn(k, r);
            const float fr = y - floorf(y);
            // (also taken when 1/s overflowed and y is not finite)
            if (!(fabsf(fr - 0.5f) > 3.0517578125e-05f)) y = __fdiv_rn(k, s);
            int q = __float2int_rn(y);  // ties to even
            q = max(-127, min(127, q));
            o[j / 4] |= (uint32_t)(q & 0xFF) << (8 * (j % 4));
        }
        const int t = g / (D / 16), c = g % (D / 16);
        *reinterpret_cast<uint4*>(kq + ((long long)blockIdx.y * ctx_pad + t) * D + c * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int D, int BITS>
cudaError_t run(const Shape& s, const LayerBufs& L, const void* K, const void* V, int* status,
                cudaStream_t st) {
    // the layer's two scratch words {max|K| bits, largest norm bits} are adjacent
    cudaError_t e = cudaMemsetAsync(L.kabsmax, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    constexpr int VPB = kEncThreads / (D / 32);
    const dim3 grid_v((s.ctx + VPB - 1) / VPB, s.kv_heads);
    encode_v_kmax_kernel<D, BITS><<<grid_v, kEncThreads, 0, st>>>(
        (const uint4*)K, (const uint4*)V, s.ctx, s.ctx_pad, L.vcodes, L.vnorm, L.kabsmax, status,
        codebook(BITS));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid_k((s.ctx * (D / 16) + 255) / 256, s.kv_heads);
    encode_k_pack_kernel<D><<<grid_k, 256, 0, st>>>((const uint4*)K, s.ctx, s.ctx_pad, L.kq, L.kabsmax,
                                                     L.kscale, status);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(256)
norm_max_kernel(const float* __restrict__ vnorm, int kv_heads, int ctx, int ctx_pad,
                uint32_t* __restrict__ vnmax) {
    uint32_t m = 0;
    const long long n = (long long)kv_heads * ctx;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const long long h = i / ctx, t = i - h * ctx;
        m = max(m, __float_as_uint(fabsf(vnorm[h * ctx_pad + t])));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0 && m) atomicMax(vnmax, m);
}

}  // namespace

cudaError_t launch_norm_max(const Shape& s, const LayerBufs& L, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(L.vnmax, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    norm_max_kernel<<<64, 256, 0, st>>>(L.vnorm, s.kv_heads, s.ctx, s.ctx_pad, L.vnmax);
    return cudaGetLastError();
}

cudaError_t launch_encode(const Shape& s, const LayerBufs& L, const void* K, const void* V,
                          int* status, cudaStream_t st) {
    if (s.head_dim == 64) {
        if (L.bits == 2) return run<64, 2>(s, L, K, V, status, st);
        if (L.bits == 3) return run<64, 3>(s, L, K, V, status, st);
        return run<64, 4>(s, L, K, V, status, st);
    }
    if (L.bits == 2) return run<128, 2>(s, L, K, V, status, st);
    if (L.bits == 3) return run<128, 3>(s, L, K, V, status, st);
    return run<128, 4>(s, L, K, V, status, st);
}

}  // namespace kvp
