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
//   encode_v_kmax: one thread per head-vector. The CTA stages 128 V rows
//     through shared memory with coalesced 16-byte loads, and on the way
//     reduces max|K| over the same 128 K rows (warp redux + one atomicMax per
//     warp on the layer's bf16-bits word). Each thread then computes the norm
//     (exact squares, pairwise tree), the FWHT in registers, one float32
//     threshold per midpoint (m_j * n) and the codes, and stores the packed
//     codes and the norm.
//   encode_k_pack: s = max|K| / 127, q = clamp(rint(k / s), -127, 127), 16
//     elements per thread with 16-byte loads and stores.
// Every float operation that decides a code uses an explicit IEEE round-to-
// nearest intrinsic, in the fixed order of the definition, so the codes are
// reproducible bit for bit (no contraction into FMA, no approximate division).
#include <cuda_bf16.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

constexpr int kEncThreads = 128;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D, int BITS>
__global__ void __launch_bounds__(kEncThreads)
encode_v_kmax_kernel(const uint4* __restrict__ K, const uint4* __restrict__ V, int nvec, int ctx,
                     int ctx_pad, uint8_t* __restrict__ vcodes, float* __restrict__ vnorm,
                     uint32_t* __restrict__ kabsmax, uint32_t* __restrict__ vnmax,
                     int* __restrict__ status, Codebook cb) {
    constexpr int CH = D / 8;          // 16-byte chunks per head-vector
    constexpr int ROW = D * 2 + 16;    // padded shared-memory row: conflict-free 16-byte reads
    constexpr int L = 1 << BITS;
    constexpr int VB = D * BITS / 8;   // packed bytes per head-vector
    constexpr int NW = VB / 4;
    __shared__ __align__(16) unsigned char srow[kEncThreads * ROW];

    const int tid = threadIdx.x;
    const long long v0 = (long long)blockIdx.x * kEncThreads;

    // 1. stage V rows; max |K| over the same rows
    uint32_t kmax = 0;
#pragma unroll 4
    for (int i = tid; i < kEncThreads * CH; i += kEncThreads) {
        const int r = i / CH, c = i % CH;
        const long long v = v0 + r;
        uint4 x = make_uint4(0, 0, 0, 0), k = make_uint4(0, 0, 0, 0);
        if (v < nvec) {
            x = __ldg(V + v * CH + c);
            k = __ldg(K + v * CH + c);
        }
        *reinterpret_cast<uint4*>(srow + r * ROW + c * 16) = x;
        const uint32_t m = 0x7FFF7FFFu;
        const uint32_t a = __vmaxu2(__vmaxu2(k.x & m, k.y & m), __vmaxu2(k.z & m, k.w & m));
        kmax = max(kmax, max(a & 0xFFFFu, a >> 16));
    }
    // |bf16| bit patterns order like their values; Inf/NaN patterns exceed
    // every finite one, so a non-finite K survives the maximum.
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if ((tid & 31) == 0 && kmax) atomicMax(kabsmax, kmax);
    __syncthreads();

    const long long v = v0 + tid;
    const bool live = v < nvec;
    const unsigned char* row = srow + tid * ROW;

    // 2. norm: sq_i = v_i^2 + v_{i+D/2}^2 (first tree level), then halves
    float s[D / 2];
#pragma unroll
    for (int c = 0; c < CH / 2; ++c) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + c * 16);
        const uint4 b = *reinterpret_cast<const uint4*>(row + (c + CH / 2) * 16);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a0 = bf_lo(aw[j]), a1 = bf_hi(aw[j]);
            const float b0 = bf_lo(bw[j]), b1 = bf_hi(bw[j]);
            s[c * 8 + 2 * j] = __fadd_rn(__fmul_rn(a0, a0), __fmul_rn(b0, b0));
            s[c * 8 + 2 * j + 1] = __fadd_rn(__fmul_rn(a1, a1), __fmul_rn(b1, b1));
        }
    }
#pragma unroll
    for (int w = D / 4; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) s[i] = __fadd_rn(s[i], s[i + w]);
    }
    const float n = __fsqrt_rn(s[0]);
    // largest norm of the layer (non-negative floats order like their bits)
    const uint32_t nmax = __reduce_max_sync(0xffffffffu, __float_as_uint(n));
    if ((tid & 31) == 0 && nmax) atomicMax(vnmax, nmax);
    if (!live) return;

    // 3. FWHT in registers, stages h = 1, 2, ..., D/2, lower index first
    float x[D];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + c * 16);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[c * 8 + 2 * j] = bf_lo(aw[j]);
            x[c * 8 + 2 * j + 1] = bf_hi(aw[j]);
        }
    }
#pragma unroll
    for (int h = 1; h < D; h <<= 1) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            if (!(i & h)) {
                const float a = x[i], b = x[i + h];
                x[i] = __fadd_rn(a, b);
                x[i + h] = __fsub_rn(a, b);
            }
        }
    }

    // 4. thresholds m_j * n, 5. codes = number of thresholds exceeded
    float tau[L - 1];
#pragma unroll
    for (int j = 0; j < L - 1; ++j) tau[j] = __fmul_rn(cb.m[j], n);
    uint32_t words[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) words[w] = 0;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        uint32_t code = 0;
#pragma unroll
        for (int j = 0; j < L - 1; ++j) code += (x[i] > tau[j]) ? 1u : 0u;
        const int bit = i * BITS, w = bit / 32, off = bit % 32;
        words[w] |= code << off;
        if (off + BITS > 32) words[w + 1] |= code >> (32 - off);
    }

    // 6. store codes and norm at the padded token position
    const long long head = v / ctx, t = v - head * ctx;
    const long long dst = head * ctx_pad + t;
    uint8_t* out = vcodes + dst * VB;
    if constexpr (VB % 16 == 0) {
#pragma unroll
        for (int q = 0; q < VB / 16; ++q)
            reinterpret_cast<uint4*>(out)[q] =
                make_uint4(words[4 * q], words[4 * q + 1], words[4 * q + 2], words[4 * q + 3]);
    } else {
#pragma unroll
        for (int q = 0; q < VB / 8; ++q)
            reinterpret_cast<uint2*>(out)[q] = make_uint2(words[2 * q], words[2 * q + 1]);
    }
    vnorm[dst] = n;
    if (!isfinite(n)) atomicOr(status, kStNonfinite);
}

template <int D>
__global__ void __launch_bounds__(256)
encode_k_pack_kernel(const uint4* __restrict__ K, long long n16, int ctx, int ctx_pad,
                     int8_t* __restrict__ kq, const uint32_t* __restrict__ kabsmax,
                     float* __restrict__ kscale, int* __restrict__ status) {
    const uint32_t am = *kabsmax;
    const float s = (am == 0) ? 1.0f : __fdiv_rn(__uint_as_float(am << 16), 127.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *kscale = s;
        if (am >= 0x7F80u) atomicOr(status, kStNonfinite);
    }
    for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < n16;
         g += (long long)gridDim.x * blockDim.x) {
        const uint4 a = __ldg(K + 2 * g), b = __ldg(K + 2 * g + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float k = (j & 1) ? bf_hi(w[j / 2]) : bf_lo(w[j / 2]);
            int q = __float2int_rn(__fdiv_rn(k, s));  // ties to even
            q = max(-127, min(127, q));
            o[j / 4] |= (uint32_t)(q & 0xFF) << (8 * (j % 4));
        }
        const long long e = g * 16, vec = e / D;
        const long long head = vec / ctx, t = vec - head * ctx;
        *reinterpret_cast<uint4*>(kq + (head * ctx_pad + t) * D + (e % D)) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int D, int BITS>
cudaError_t run(const Shape& s, const LayerBufs& L, const void* K, const void* V, int* status,
                cudaStream_t st) {
    const long long nvec = (long long)s.kv_heads * s.ctx;
    cudaError_t e = cudaMemsetAsync(L.kabsmax, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(L.vnmax, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    const unsigned grid_v = (unsigned)((nvec + kEncThreads - 1) / kEncThreads);
    encode_v_kmax_kernel<D, BITS><<<grid_v, kEncThreads, 0, st>>>(
        (const uint4*)K, (const uint4*)V, (int)nvec, s.ctx, s.ctx_pad, L.vcodes, L.vnorm,
        L.kabsmax, L.vnmax, status, codebook(BITS));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long n16 = nvec * D / 16;
    const unsigned grid_k = (unsigned)((n16 + 255) / 256);
    encode_k_pack_kernel<D><<<grid_k, 256, 0, st>>>((const uint4*)K, n16, s.ctx, s.ctx_pad, L.kq,
                                                     L.kabsmax, L.kscale, status);
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
