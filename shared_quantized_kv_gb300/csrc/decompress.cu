// Materialisation of one pool layer as bf16 K and V.
//
// PolyKV summary, section 2.A: each PooledAgent injects the decompressed K/V
// of every layer into its own cache; section 2.B: V is dequantised by
// centroid lookup followed by the inverse FWHT (H H = d I, so the inverse is
// H / d). This is the per-agent baseline path that direct attention over the
// pool avoids.
//
//   decompress_v: one thread per head-vector: unpack the codes, look the
//     centroids up in a shared-memory table, FWHT in registers in the encoder's
//     stage order, V_i = bf16(fl(fl(z_i * n) * (1/d))), 16-byte stores.
//   decompress_k: K = bf16(fl(q * s)), 16 elements per thread.
#include <cuda_bf16.h>

#include "kvpool_internal.cuh"

namespace kvp {
namespace {

__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int D, int BITS>
__global__ void __launch_bounds__(128)
decompress_v_kernel(const uint8_t* __restrict__ vcodes, const float* __restrict__ vnorm, int nvec,
                    int ctx, int ctx_pad, uint4* __restrict__ Vout, Codebook cb) {
    constexpr int VB = D * BITS / 8;
    constexpr int NW = VB / 4;
    constexpr uint32_t MASK = (1u << BITS) - 1;
    __shared__ float cen[16];
    if (threadIdx.x < 16) cen[threadIdx.x] = cb.c[threadIdx.x];
    __syncthreads();
    const long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= nvec) return;
    const long long head = v / ctx, t = v - head * ctx;
    const long long src = head * ctx_pad + t;

    uint32_t words[NW];
    const uint8_t* in = vcodes + src * VB;
    if constexpr (VB % 16 == 0) {
#pragma unroll
        for (int q = 0; q < VB / 16; ++q) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(in) + q);
            words[4 * q] = u.x; words[4 * q + 1] = u.y; words[4 * q + 2] = u.z; words[4 * q + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < VB / 8; ++q) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(in) + q);
            words[2 * q] = u.x; words[2 * q + 1] = u.y;
        }
    }
    float x[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const int bit = i * BITS, w = bit / 32, off = bit % 32;
        uint32_t code = words[w] >> off;
        if (off + BITS > 32) code |= words[w + 1] << (32 - off);
        x[i] = cen[code & MASK];
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
    const float n = __ldg(vnorm + src);
    const float inv_d = 1.0f / (float)D;  // a power of two: exact
    uint4* out = Vout + v * (D / 8);
#pragma unroll
    for (int q = 0; q < D / 8; ++q) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __fmul_rn(__fmul_rn(x[8 * q + 2 * j], n), inv_d);
            const float hi = __fmul_rn(__fmul_rn(x[8 * q + 2 * j + 1], n), inv_d);
            o[j] = bf16_bits(lo) | (bf16_bits(hi) << 16);
        }
        out[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int D>
__global__ void __launch_bounds__(256)
decompress_k_kernel(const int8_t* __restrict__ kq, const float* __restrict__ kscale, long long n16,
                    int ctx, int ctx_pad, uint4* __restrict__ Kout) {
    const float s = *kscale;
    for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < n16;
         g += (long long)gridDim.x * blockDim.x) {
        const long long e = g * 16, vec = e / D;
        const long long head = vec / ctx, t = vec - head * ctx;
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(kq + (head * ctx_pad + t) * D + (e % D)));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int b0 = (int)(int8_t)((w[j / 2] >> (16 * (j % 2))) & 0xFF);
            const int b1 = (int)(int8_t)((w[j / 2] >> (16 * (j % 2) + 8)) & 0xFF);
            o[j] = bf16_bits(__fmul_rn((float)b0, s)) | (bf16_bits(__fmul_rn((float)b1, s)) << 16);
        }
        Kout[2 * g] = make_uint4(o[0], o[1], o[2], o[3]);
        Kout[2 * g + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

template <int D, int BITS>
cudaError_t run(const Shape& s, const LayerBufs& L, void* K_out, void* V_out, cudaStream_t st) {
    const long long nvec = (long long)s.kv_heads * s.ctx;
    if (V_out) {
        decompress_v_kernel<D, BITS><<<(unsigned)((nvec + 127) / 128), 128, 0, st>>>(
            L.vcodes, L.vnorm, (int)nvec, s.ctx, s.ctx_pad, (uint4*)V_out, codebook(BITS));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (K_out) {
        const long long n16 = nvec * D / 16;
        decompress_k_kernel<D><<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(
            L.kq, L.kscale, n16, s.ctx, s.ctx_pad, (uint4*)K_out);
        return cudaGetLastError();
    }
    return cudaSuccess;
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
