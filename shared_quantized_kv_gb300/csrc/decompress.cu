// Materialisation of one pool layer as bf16 K and V.
//
// PolyKV summary, section 2.A: each PooledAgent injects the decompressed K/V
// of every layer into its own cache; section 2.B: V is dequantised by
// centroid lookup followed by the inverse FWHT (H H = d I, so the inverse is
// H / d). This is the per-agent baseline path that direct attention over the
// pool avoids.
//
// One kernel, grid (blocks, kv heads):
//   V blocks: the block's code groups are unpacked into bytes [token]
//     [coordinate] in shared memory; then D/32 threads per head-vector, 32
//     coordinates each, look the centroids up in a shared-memory table, FWHT in
//     the encoder's stage order (h < 32 in registers, h = 32, 64 by
//     shfl.xor and one exact FMA), V_i = bf16(fl(fl(z_i * n) * (1/d))),
//     coalesced 16-byte stores.
//   K blocks: K = bf16(fl(q * s)), four 16-element groups per thread, loads
//     first, so that the V and K blocks fit one wave (the int8 to float
//     conversion by an integer add and one exact subtraction); s is the
//     layer's scale or, in block-scaled pools, the element's 32-block scale.
#include <cuda_bf16.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

constexpr int kDecThreads = 256;
constexpr int kKGroups = 4;  // K blocks: 16-element groups per thread (V and K blocks fit one wave)

// bf16 bits of (lo, hi), each rounded to nearest even, lo in the low half
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// the int8 in byte k of w as a float (exact: 1.5 * 2^23 + q has q in its low bits)
__device__ __forceinline__ float i8_to_f(uint32_t w, int k) {
    const int q = (int)(int8_t)((w >> (8 * k)) & 0xFF);
    return __fsub_rn(__int_as_float(0x4B400000 + q), 12582912.0f);
}

// One launch for both halves, grid (blocks, kv heads): the first nbv blocks of
// each head materialise V (D/32 threads per head-vector), the rest K (16
// elements per thread).
template <int D, int BITS>
__global__ void __launch_bounds__(kDecThreads)
decompress_kernel(const int8_t* __restrict__ kq, const float* __restrict__ kscale,
                  const float* __restrict__ kscales,
                  const uint8_t* __restrict__ vcodes, const float* __restrict__ vnorm, int ctx,
                  int ctx_pad, int nbv, uint4* __restrict__ Kout, uint4* __restrict__ Vout,
                  Codebook cb) {
    constexpr int TPV = D / 32;
    constexpr uint32_t MASK = (1u << BITS) - 1;
    const int tid = threadIdx.x;
    const long long head = blockIdx.y;
    if ((int)blockIdx.x >= nbv) {
        // ---- K = bf16(q * s): the layer's scale, or the scale of the 32-element
        //      block holding a 16-element group. kKGroups groups per thread,
        //      all loads in flight before any conversion.
        const int n16 = ctx * (D / 16);  // 16-element groups in the head
        const float s0 = kscales ? 1.0f : *kscale;
        uint4 q[kKGroups];
        float sc[kKGroups];
#pragma unroll
        for (int u = 0; u < kKGroups; ++u) {
            const int g = (blockIdx.x - nbv) * (kDecThreads * kKGroups) + u * kDecThreads + tid;
            const int t = g / (D / 16), c = g % (D / 16);
            q[u] = g < n16 ? __ldg(reinterpret_cast<const uint4*>(kq + (head * ctx_pad + t) * D + c * 16))
                           : make_uint4(0, 0, 0, 0);
            sc[u] = (kscales && g < n16) ? __ldg(kscales + (head * ctx_pad + t) * (D / 32) + c / 2) : s0;
        }
#pragma unroll
        for (int u = 0; u < kKGroups; ++u) {
            const int g = (blockIdx.x - nbv) * (kDecThreads * kKGroups) + u * kDecThreads + tid;
            if (g >= n16) break;
            const int t = g / (D / 16), c = g % (D / 16);
            const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float k0 = i8_to_f(w[j / 2], 2 * (j % 2)), k1 = i8_to_f(w[j / 2], 2 * (j % 2) + 1);
                o[j] = bf16x2_bits(__fmul_rn(k0, sc[u]), __fmul_rn(k1, sc[u]));
            }
            uint4* out = Kout + (head * ctx + t) * (D / 8) + 2 * c;
            out[0] = make_uint4(o[0], o[1], o[2], o[3]);
            out[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        return;
    }
    // ---- V = bf16(fl(fl(z * n) * (1/d))), z = FWHT(c[codes])
    // the block's code groups (pool layout: per 32 tokens, one sequence per
    // coordinate) are unpacked into bytes [token][coordinate] first
    constexpr int VPB = kDecThreads / TPV;  // head-vectors per block (a multiple of 32)
    __shared__ float cen[16];
    __shared__ __align__(16) uint8_t codes8[VPB * D];
    if (tid < 16) cen[tid] = cb.c[tid];
    const int lt = tid % TPV;
    const int t = blockIdx.x * VPB + tid / TPV;
    const bool live = t < ctx;
    const float n = live ? __ldg(vnorm + head * ctx_pad + t) : 0.f;  // in flight during the unpacking
    {
        const int gq = tid / D, c = tid % D;
        const long long grp = (head * ctx_pad + (long long)blockIdx.x * VPB) / 32 + gq;
        const uint32_t* in = reinterpret_cast<const uint32_t*>(vcodes + (grp * D + c) * (4 * BITS));
        uint32_t w[BITS + 1];
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[k] = __ldg(in + k);
        w[BITS] = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int bit = j * BITS;
            codes8[(gq * 32 + j) * D + c] = (uint8_t)(__funnelshift_r(w[bit / 32], w[bit / 32 + 1], bit % 32) & MASK);
        }
    }
    __syncthreads();
    const unsigned gmask = 0xffffffffu;
    const uint4* c8 = reinterpret_cast<const uint4*>(codes8 + (tid / TPV) * D + lt * 32);
    const uint4 ca = c8[0], cb8 = c8[1];
    const uint32_t cw[8] = {ca.x, ca.y, ca.z, ca.w, cb8.x, cb8.y, cb8.z, cb8.w};
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = cen[(cw[i / 4] >> (8 * (i % 4))) & 0xFF];
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
        // lower slice: own + partner; upper slice: partner - own (one
        // rounding either way, exactly the add or the subtraction)
        const float sg = (lt & off) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float o = __shfl_xor_sync(gmask, x[i], off, TPV);
            x[i] = __fmaf_rn(sg, x[i], o);
        }
    }
    if (!live) return;
    const float inv_d = 1.0f / (float)D;  // a power of two: exact
    uint4* out = Vout + (head * ctx + t) * (D / 8) + lt * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __fmul_rn(__fmul_rn(x[8 * q + 2 * j], n), inv_d);
            const float hi = __fmul_rn(__fmul_rn(x[8 * q + 2 * j + 1], n), inv_d);
            o[j] = bf16x2_bits(lo, hi);
        }
        out[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int D, int BITS>
cudaError_t run(const Shape& s, const LayerBufs& L, void* K_out, void* V_out, cudaStream_t st) {
    constexpr int VPB = kDecThreads / (D / 32);
    const int nbv = V_out ? (s.ctx + VPB - 1) / VPB : 0;
    const int nbk = K_out ? (s.ctx * (D / 16) + kDecThreads * kKGroups - 1) / (kDecThreads * kKGroups) : 0;
    if (nbv + nbk == 0) return cudaSuccess;
    decompress_kernel<D, BITS><<<dim3(nbv + nbk, s.kv_heads), kDecThreads, 0, st>>>(
        L.kq, L.kscale, L.kscales, L.vcodes, L.vnorm, s.ctx, s.ctx_pad, nbv, (uint4*)K_out, (uint4*)V_out,
        codebook(BITS));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decompress(const Shape& s, const LayerBufs& L, void* K_out, void* V_out,
                              cudaStream_t st) {
    if (s.head_dim == 64) {
        if (L.bits == 2) return run<64, 2>(s, L, K_out, V_out, st);
        if (L.bits == 3) return run<64, 3>(s, L, K_out, V_out, st);
        return run<64, 4>(s, L, K_out, V_out, st);
    }
    if (L.bits == 2) return run<128, 2>(s, L, K_out, V_out, st);
    if (L.bits == 3) return run<128, 3>(s, L, K_out, V_out, st);
    return run<128, 4>(s, L, K_out, V_out, st);
}

}  // namespace kvp
