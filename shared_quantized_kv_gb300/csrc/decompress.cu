// Materialisation of pool layers as bf16 K and V.
//
// PolyKV summary, section 2.A: each PooledAgent injects the decompressed K/V
// of every layer into its own cache; section 2.B: V is dequantised by
// centroid lookup followed by the inverse FWHT (H H = d I, so the inverse is
// H / d). This is the per-agent baseline path that direct attention over the
// pool avoids.
//
// One kernel per V width for any number of layers (up to 32 per launch),
// grid (blocks, kv heads, layers):
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

#include <algorithm>

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
// the int8s in bytes k, k + 1 of w as floats (exact: 1.5 * 2^23 + q has q in
// its low bits); one paired subtraction
__device__ __forceinline__ float2 i8x2_to_f2(uint32_t w, int k) {
    const int q0 = (int)(int8_t)((w >> (8 * k)) & 0xFF), q1 = (int)(int8_t)((w >> (8 * k + 8)) & 0xFF);
    return __fadd2_rn(make_float2(__int_as_float(0x4B400000 + q0), __int_as_float(0x4B400000 + q1)),
                      make_float2(-12582912.0f, -12582912.0f));
}

// Centroids of the launch: c_BITS in entries [0, 2^BITS), or (layers of
// per-group widths) the tables of widths 2, 3, 4 at entries 0, 4, 12.
struct CenTable {
    float c[28];
};
__host__ __device__ constexpr int mix_base(int w) { return w == 2 ? 0 : (w == 3 ? 4 : 12); }

// one packed sequence of 32 codes of width B (4 * B bytes at `in`) into the
// bytes dst[0], dst[D], ..., dst[31 D], each plus `base`
template <int D, int B>
__device__ __forceinline__ void unpack_seq(const uint32_t* __restrict__ in, uint8_t* dst, uint32_t base) {
    constexpr uint32_t MASK = (1u << B) - 1;
    uint32_t w[B + 1];
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = __ldg(in + k);
    w[B] = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int bit = j * B;
        dst[j * D] = (uint8_t)(base + (__funnelshift_r(w[bit / 32], w[bit / 32 + 1], bit % 32) & MASK));
    }
}

// One launch for both halves of every layer of the launch, grid (blocks, kv
// heads, layers): the first nbv blocks of each head materialise V (D/32
// threads per head-vector), the next nbk K (16 elements per thread). MIX:
// layers of per-group V widths (each 32-token group read at its own width).
template <int D, int BITS, bool MIX>
__global__ void __launch_bounds__(kDecThreads, 5)  // five CTAs per SM: both halves in one wave
decompress_kernel(const __grid_constant__ DecBatch b, int ctx_pad, const __grid_constant__ CenTable ct) {
    constexpr int TPV = D / 32;
    constexpr int VPB = kDecThreads / TPV;  // head-vectors per V block (a multiple of 32)
    const DecLayer& Ly = b.L[blockIdx.z];
    const int tid = threadIdx.x;
    const long long head = blockIdx.y;
    const int ctx = Ly.len;
    const int8_t* __restrict__ kq = Ly.kq;
    const float* __restrict__ kscales = Ly.kscales;
    const int nbv = Ly.Vout ? (ctx + VPB - 1) / VPB : 0;
    const int nbk = Ly.Kout ? (ctx * (D / 16) + kDecThreads * kKGroups - 1) / (kDecThreads * kKGroups) : 0;
    if ((int)blockIdx.x >= nbv + nbk) return;  // a shorter layer of the launch
    if ((int)blockIdx.x >= nbv) {
        // ---- K = bf16(q * s): the layer's scale, or the scale of the 32-element
        //      block holding a 16-element group. kKGroups groups per thread,
        //      all loads in flight before any conversion.
        const int n16 = ctx * (D / 16);  // 16-element groups in the head
        const float s0 = kscales ? 1.0f : *Ly.kscale;
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
                const float2 k = i8x2_to_f2(w[j / 2], 2 * (j % 2));
                const float2 v = __fmul2_rn(k, make_float2(sc[u], sc[u]));
                o[j] = bf16x2_bits(v.x, v.y);
            }
            uint4* out = Ly.Kout + (head * ctx + t) * (D / 8) + 2 * c;
            out[0] = make_uint4(o[0], o[1], o[2], o[3]);
            out[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        return;
    }
    // ---- V = bf16(fl(fl(z * n) * (1/d))), z = FWHT(c[codes])
    // the block's code groups (pool layout: per 32 tokens, one sequence per
    // coordinate) are unpacked into bytes [token][coordinate] first
    __shared__ float cen[28];
    __shared__ __align__(16) uint8_t codes8[VPB * D];
    if (tid < 28) cen[tid] = ct.c[tid];
    const int lt = tid % TPV;
    const int t = blockIdx.x * VPB + tid / TPV;
    const bool live = t < ctx;
    const float n = live ? __ldg(Ly.vnorm + head * ctx_pad + t) : 0.f;  // in flight during the unpacking
    {
        const int gq = tid / D, c = tid % D;
        uint8_t* dst = codes8 + gq * 32 * D + c;
        if constexpr (MIX) {
            // the group's width (warp-uniform: a warp serves one group); a
            // group not written holds no live token
            const int gi = blockIdx.x * (VPB / 32) + gq;
            const int w = __ldg(Ly.gbits + gi);
            const unsigned char* grp = Ly.vcodes + head * Ly.vhead + (w ? __ldg(Ly.goff + gi) : 0u);
            if (w == 2) unpack_seq<D, 2>(reinterpret_cast<const uint32_t*>(grp + c * 8), dst, mix_base(2));
            else if (w == 3) unpack_seq<D, 3>(reinterpret_cast<const uint32_t*>(grp + c * 12), dst, mix_base(3));
            else if (w == 4) unpack_seq<D, 4>(reinterpret_cast<const uint32_t*>(grp + c * 16), dst, mix_base(4));
            else
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[j * D] = 0;
        } else {
            const long long grp = (head * ctx_pad + (long long)blockIdx.x * VPB) / 32 + gq;
            unpack_seq<D, BITS>(reinterpret_cast<const uint32_t*>(Ly.vcodes + (grp * D + c) * (4 * BITS)), dst, 0);
        }
    }
    __syncthreads();
    const unsigned gmask = 0xffffffffu;
    const uint4* c8 = reinterpret_cast<const uint4*>(codes8 + (tid / TPV) * D + lt * 32);
    const uint4 ca = c8[0], cb8 = c8[1];
    const uint32_t cw[8] = {ca.x, ca.y, ca.z, ca.w, cb8.x, cb8.y, cb8.z, cb8.w};
    // the float steps run on coordinate pairs (2i, 2i + 1): one instruction,
    // two IEEE round-to-nearest operations in the encoder's order
    float2 x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        x[i] = make_float2(cen[(cw[i / 2] >> (16 * (i % 2))) & 0xFF], cen[(cw[i / 2] >> (16 * (i % 2) + 8)) & 0xFF]);
    // FWHT stages h = 1 (inside each pair), 2 ... 16 (pairs i and i + h/2)
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = make_float2(__fadd_rn(x[i].x, x[i].y), __fsub_rn(x[i].x, x[i].y));
#pragma unroll
    for (int hp = 1; hp < 16; hp <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (!(i & hp)) {
                const float2 a = x[i], b = x[i + hp];
                x[i] = __fadd2_rn(a, b);
                x[i + hp] = __fadd2_rn(a, make_float2(-b.x, -b.y));  // a - b, exact negation
            }
        }
    }
#pragma unroll
    for (int h = 32; h < D; h <<= 1) {
        const int off = h / 32;
        // lower slice: own + partner; upper slice: partner - own (one
        // rounding either way, exactly the add or the subtraction)
        const float sg = (lt & off) ? -1.0f : 1.0f;
        const float2 sg2 = make_float2(sg, sg);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 o = make_float2(__shfl_xor_sync(gmask, x[i].x, off, TPV),
                                         __shfl_xor_sync(gmask, x[i].y, off, TPV));
            x[i] = __ffma2_rn(sg2, x[i], o);
        }
    }
    if (!live) return;
    const float inv_d = 1.0f / (float)D;  // a power of two: exact
    const float2 n2 = make_float2(n, n), d2 = make_float2(inv_d, inv_d);
    uint4* out = Ly.Vout + (head * ctx + t) * (D / 8) + lt * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 v = __fmul2_rn(__fmul2_rn(x[4 * q + j], n2), d2);
            o[j] = bf16x2_bits(v.x, v.y);
        }
        out[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int D, int BITS, bool MIX>
cudaError_t run(const Shape& s, const DecBatch& b, cudaStream_t st) {
    constexpr int VPB = kDecThreads / (D / 32);
    int gx = 0;
    for (int i = 0; i < b.n; ++i) {
        const int len = b.L[i].len;
        const int nbv = b.L[i].Vout ? (len + VPB - 1) / VPB : 0;
        const int nbk = b.L[i].Kout ? (len * (D / 16) + kDecThreads * kKGroups - 1) / (kDecThreads * kKGroups) : 0;
        gx = std::max(gx, nbv + nbk);
    }
    if (gx == 0) return cudaSuccess;
    CenTable ct = {};
    if (MIX) {
        for (int w = 2; w <= 4; ++w)
            for (int k = 0; k < (1 << w); ++k) ct.c[mix_base(w) + k] = codebook(w).c[k];
    } else {
        for (int k = 0; k < (1 << BITS); ++k) ct.c[k] = codebook(BITS).c[k];
    }
    decompress_kernel<D, BITS, MIX><<<dim3(gx, s.kv_heads, b.n), kDecThreads, 0, st>>>(b, s.ctx_pad, ct);
    return cudaGetLastError();
}

// bits 0: layers of per-group widths
template <int D>
cudaError_t run_bits(int bits, const Shape& s, const DecBatch& b, cudaStream_t st) {
    if (bits == 0) return run<D, 4, true>(s, b, st);
    if (bits == 2) return run<D, 2, false>(s, b, st);
    if (bits == 3) return run<D, 3, false>(s, b, st);
    return run<D, 4, false>(s, b, st);
}

}  // namespace

cudaError_t launch_decompress_layers(const Shape& s, const LayerBufs* L, const int* len, void* const* K_out,
                                     void* const* V_out, int n, cudaStream_t st) {
    for (int c0 = 0; c0 < n; c0 += kEncBatch) {
        const int nc = std::min(kEncBatch, n - c0);
        for (int bits = 0; bits <= 4; ++bits) {  // one launch per V width (0: per-group widths)
            if (bits == 1) continue;
            DecBatch b = {};
            for (int i = c0; i < c0 + nc; ++i) {
                if ((L[i].mixed ? 0 : L[i].bits) != bits) continue;
                DecLayer& d = b.L[b.n++];
                d.kq = L[i].kq;
                d.kscale = L[i].kscale;
                d.kscales = L[i].kscales;
                d.vcodes = L[i].vcodes;
                d.vnorm = L[i].vnorm;
                d.gbits = L[i].gbits;
                d.goff = L[i].goff;
                d.vhead = L[i].vhead;
                d.Kout = K_out ? static_cast<uint4*>(K_out[i]) : nullptr;
                d.Vout = V_out ? static_cast<uint4*>(V_out[i]) : nullptr;
                d.len = len[i];
            }
            if (b.n == 0) continue;
            const cudaError_t e = s.head_dim == 64 ? run_bits<64>(bits, s, b, st) : run_bits<128>(bits, s, b, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_decompress(const Shape& s, const LayerBufs& L, void* K_out, void* V_out, cudaStream_t st) {
    void* k[1] = {K_out};
    void* v[1] = {V_out};
    return launch_decompress_layers(s, &L, &s.ctx, K_out ? k : nullptr, V_out ? v : nullptr, 1, st);
}

}  // namespace kvp
