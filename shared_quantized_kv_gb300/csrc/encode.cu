// Write-once encode of pool layers.
//
// PolyKV summary (gist.science, "PolyKV: A Shared Asymmetrically-Compressed
// KV Cache Pool for Multi-Agent LLM Inference"), section 2.B:
//   K: per-tensor linear quantisation to int8.
//   V: FWHT rotation of each head-vector, then the nearest Lloyd-Max centroid
//      for N(0,1) per rotated coordinate (3 bits; 2 or 4 bits per layer in the
//      CoMixKV article's mixed-precision setting).
//
// Two kernels per layer. The max|K| kernel reduces slices of the K tensor to
// partial maxima and releases the encode kernel at once (programmatic
// dependent launch), so the encode kernel's V work runs beside it. In the
// encode kernel an item is 32 (head_dim 128) or 64 (head_dim 64) consecutive
// tokens of one KV head: 8 KB of K and 8 KB of V, brought into shared memory
// by bulk copies (one mbarrier per tile). CTA i takes items i, i + G, ...
// (G = grid size); the first item's copies are requested at launch (K and V
// are inputs no earlier kernel writes).
//   V, per item and head-vector, D/32 threads with 32 coordinates each: the
//     norm by the pairwise tree (the first levels cross threads by shuffles),
//     the FWHT (stages h < 32 in registers, h = 32, 64 by shfl.xor and one
//     exact FMA), one float32 threshold per midpoint (m_j * n), the codes by a
//     branchless binary search over the sorted thresholds, regrouped through
//     shared memory into the pool layout: per group of 32 tokens, one packed
//     sequence per coordinate (the 32 tokens' codes in token order, 4*BITS
//     bytes).
//   K: before its first K codes the kernel waits for the max|K| kernel and
//     reduces the partial maxima: s = max|K| / 127, and per element
//     q = clamp(rint(k / s), -127, 127) from the K tile: k / s is formed as
//     k * (1/s) and rounded by the 1.5 * 2^23 addition; where the product lies
//     within 2^-15 of a half-integer (the two could round to different
//     integers) the chunk's 8 elements are recomputed with IEEE divisions.
//     Block-scaled pools (one scale per 32 elements) take each block's scale
//     from its own maximum and run no max|K| kernel.
// A CTA's tiles (V of each of its items, then K of each) stream through two
// shared-memory buffers, two copies in flight: tile t + 2 is requested as
// soon as every thread has read tile t.
// Every float operation that decides a code uses an explicit IEEE round-to-
// nearest intrinsic, in the fixed order of the definition, so the codes are
// reproducible bit for bit (no contraction into FMA, no approximate division).
#include <cuda_bf16.h>

#include <algorithm>

#include "kvpool_internal.cuh"
#include "tc_ptx.cuh"

namespace kvp {
namespace {

constexpr int kEncThreads = 128;
constexpr uint64_t kEncWaitNs = 200ull * 1000 * 1000;  // bounded waits on the tile copies

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

// int8 codes of 8 bf16 values (one 16-byte chunk) as two little-endian words;
// the float steps run on element pairs (two IEEE round-to-nearest operations
// per instruction)
__device__ __forceinline__ uint2 quant8(uint4 u, float s, float r) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds |y| < 2^22 to an integer
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    const float2 r2 = make_float2(r, r), m2 = make_float2(kMagic, kMagic), nm2 = make_float2(-kMagic, -kMagic);
    uint32_t b[8];
    bool amb = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // k * (1/s) is within ~1.5 ulp of k / s; unless that lands within
        // 2^-15 of a half-integer both round to the same integer
        const float2 y = __fmul2_rn(make_float2(bf_lo(w[j]), bf_hi(w[j])), r2);
        const float2 t = __fadd2_rn(y, m2);                      // kMagic + rint(y), ties to even
        const float2 i = __fadd2_rn(t, nm2);                     // rint(y), exact
        const float2 e = __fadd2_rn(y, make_float2(-i.x, -i.y));  // y - rint(y), exact
        amb |= !(fabsf(e.x) < 0.499969482421875f);               // 0.5 - 2^-15 (also taken for NaN)
        amb |= !(fabsf(e.y) < 0.499969482421875f);
        b[2 * j] = __float_as_uint(t.x);  // low byte: rint(y) mod 256
        b[2 * j + 1] = __float_as_uint(t.y);
    }
    if (amb) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float k = (j & 1) ? bf_hi(w[j / 2]) : bf_lo(w[j / 2]);
            const int q = max(-127, min(127, __float2int_rn(__fdiv_rn(k, s))));
            b[j] = (uint32_t)q;
        }
    }
    const uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

// |bf16| bit patterns order like their values, and Inf/NaN patterns exceed
// every finite one, so a non-finite K survives the maximum.
__device__ __forceinline__ uint32_t absmax8(uint4 u) {
    const uint32_t m = 0x7FFF7FFFu;
    const uint32_t a = __vmaxu2(__vmaxu2(u.x & m, u.y & m), __vmaxu2(u.z & m, u.w & m));
    return max(a & 0xFFFFu, a >> 16);
}

// max|K| of each layer of the launch: CTA (b, l) reduces the b-th contiguous
// slice of layer l's K tensor (16-byte chunks) to a partial maximum. With
// several layers (NB > 1) the last CTA of a layer to finish (an arrival
// counter, re-armed by that CTA) reduces the partials and writes max|K|
// (bf16 bits), s = max|K| / 127 (1 when K is all zero) and 1/s; for one layer
// the encode kernel's CTAs reduce them themselves. It releases the encode
// kernel at once. For block-scaled layers it only sets *kscale = 1 and clears
// the maxima.
template <int NB>
__global__ void __launch_bounds__(256)
kmax_kernel(const __grid_constant__ EncBatchT<NB> b, long long nchunk, long long per_cta, int kb, int zero_vn,
            int* __restrict__ status) {
    ptx::grid_dep_launch();
    const EncLayer& L = b.L[blockIdx.y];
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    if (blockIdx.x == 0 && tid == 0) {
        if (zero_vn) L.maxima[1] = 0;  // raised by the encode kernel after its dependency wait
        if (kb) {
            L.maxima[0] = 0;
            *L.kscale = 1.0f;
        }
    }
    if (kb) return;
    __shared__ uint32_t red[8];
    __shared__ int last;
    const uint4* K = reinterpret_cast<const uint4*>(L.K);
    const long long c0 = (long long)blockIdx.x * per_cta;
    const long long c1 = min(nchunk, c0 + per_cta);
    uint32_t m = 0;
    for (long long base = c0 + tid; base < c1; base += 8 * 256) {
        uint4 u[8];  // all of a batch's loads in flight at once
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = (base + j * 256 < c1) ? __ldg(K + base + j * 256) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max(m, absmax8(u[j]));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int w = 1; w < 8; ++w) m = max(m, red[w]);
        L.kpart[blockIdx.x] = m;
        if constexpr (NB > 1) {
            __threadfence();  // the partial before the arrival
            last = atomicAdd(L.kpart + kKmaxCount, 1u) == gridDim.x - 1;
        }
    }
    if constexpr (NB == 1) return;
    __syncthreads();
    if (!last) return;
    __threadfence();
    uint32_t mm = 0;
    for (int i = tid; i < (int)gridDim.x; i += 256) mm = max(mm, *reinterpret_cast<volatile const uint32_t*>(L.kpart + i));
    mm = __reduce_max_sync(0xffffffffu, mm);
    __syncthreads();  // red[] is free again
    if (lane == 0) red[warp] = mm;
    __syncthreads();
    if (tid == 0) {
#pragma unroll
        for (int w = 0; w < 8; ++w) mm = max(mm, red[w]);
        const float s = (mm == 0) ? 1.0f : __fdiv_rn(__uint_as_float(mm << 16), 127.0f);
        L.maxima[0] = mm;
        *L.kscale = s;
        L.kpart[kKmaxInv] = __float_as_uint(__frcp_rn(s));
        L.kpart[kKmaxCount] = 0;  // re-armed for the layer's next compress
        if (mm >= 0x7F80u) atomicOr(status, kStNonfinite);
    }
}

// All items of the launch's layers (same V width), layer-major; CTA i takes
// items i, i + G, ... in two passes: first the V of every item (beside the
// max|K| kernel), then, after the dependency wait, the K of every item.
// KB: block-scaled K (one scale per 32 elements, written to kscales).
template <int D, int BITS, bool KB, int NB>
__global__ void __launch_bounds__(kEncThreads)
encode_kernel(const __grid_constant__ EncBatchT<NB> b, int ctx, int ctx_pad, int t_base, int items_per_head,
              int items_per_layer, int items, int nparts, int* __restrict__ status, Codebook cb) {
    constexpr int TPV = D / 32;              // threads per head-vector
    constexpr int VPI = kEncThreads / TPV;   // tokens per item (a multiple of 32)
    constexpr uint32_t kTile = VPI * D * 2;  // bytes of K (and of V) per item: 8 KB
    constexpr int kChunks = (int)(kTile / 16 / kEncThreads);  // 16-byte chunks per thread and tile
    constexpr int L = 1 << BITS;
    // the CTA's tiles, V of each of its items and then K of each, stream
    // through two buffers: tile t + 2 is requested once tile t has been read
    __shared__ __align__(128) unsigned char tiles[2][kTile];
    __shared__ __align__(16) uint8_t codes8[VPI * D];
    __shared__ uint32_t red[kEncThreads / 32];
    __shared__ __align__(8) uint64_t bars[2];  // one per buffer
    __shared__ uint32_t sDep[kEncThreads];
    extern __shared__ uint32_t snm[];  // per item of this CTA: float bits of its largest V norm
    const int tid = threadIdx.x, lane = tid % 32;
    const int lt = tid % TPV;  // this thread's 32-coordinate slice
    const int tl = tid / TPV;  // its token within the item
    const int G = (int)gridDim.x;
    const unsigned gmask = 0xffffffffu;
    const int m = (items - (int)blockIdx.x + G - 1) / G;  // items of this CTA (>= 1)

    auto item_l = [&](int it) { return it / items_per_layer; };
    auto item_h = [&](int it) { return (it % items_per_layer) / items_per_head; };
    auto item_t0 = [&](int it) { return (it % items_per_head) * VPI; };
    // K and V are inputs of the launch, written by no kernel that may still
    // run (the max|K| kernel before this one only reads K): the copies start
    // before the dependency wait
    auto item_bytes = [&](int it) { return (uint32_t)min(VPI, ctx - item_t0(it)) * D * 2; };
    auto item_src = [&](int it) { return ((long long)item_h(it) * ctx + item_t0(it)) * D; };
    // tile t < m: V of item blockIdx.x + t*G; tile m + k: K of item blockIdx.x + k*G
    auto issue_tile = [&](int t) {
        const bool isK = t >= m;
        const int it = (int)blockIdx.x + (isK ? t - m : t) * G;
        const uint32_t bar = ptx::smem_u32(&bars[t & 1]);
        const EncLayer& Ly = b.L[item_l(it)];
        ptx::mbar_expect_tx(bar, item_bytes(it));
        ptx::bulk_g2s(ptx::smem_u32(tiles[t & 1]), (isK ? Ly.K : Ly.V) + item_src(it), item_bytes(it), bar);
    };
    bool ok = true;
    auto wait_tile = [&](int t) {
        if (ok && !ptx::mbar_wait(ptx::smem_u32(&bars[t & 1]), (uint32_t)(t >> 1) & 1, kEncWaitNs)) ok = false;
    };
    // after every thread has read tile t (its dependency word stored, then a
    // barrier): the next tile for the buffer
    auto next_tile = [&](int t) {
        if (tid == 0 && ok && t + 2 < 2 * m) {
            ptx::fence_proxy_async();
            issue_tile(t + 2);
        }
    };
    if (tid == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
        ptx::mbar_init_fence();
        issue_tile(0);
        issue_tile(1);
    }
    __syncthreads();

    // ---- pass 1: V
    for (int it = blockIdx.x, k = 0; it < items; it += G, ++k) {
        const EncLayer& Ly = b.L[item_l(it)];
        const int h = item_h(it), t0 = item_t0(it);
        const int ntok = min(VPI, ctx - t0);
        wait_tile(k);
        const bool live = tl < ntok;
        float2 x[16];  // coordinates (2i, 2i + 1) of this thread's slice
        {
            uint32_t dep = 0;  // depends on every word this thread reads from the V tile
            const uint4* vs = reinterpret_cast<const uint4*>(tiles[k & 1] + tl * (D * 2) + lt * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 vv = vs[c];
                dep ^= vv.x ^ vv.y ^ vv.z ^ vv.w;
                const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) x[c * 4 + j] = make_float2(bf_lo(w[j]), bf_hi(w[j]));
            }
            // The next copy into the buffer overwrites the tile. A barrier does not
            // wait for shared-memory loads still in flight, and the copy
            // writes through the async proxy: every thread first stores a word
            // that depends on all its loads (so they have returned), and the
            // issuing thread fences the proxies before the copy.
            sDep[tid] = dep;
        }
        __syncthreads();
        next_tile(k);

        // The float steps below run on coordinate pairs (2i, 2i + 1): one
        // instruction, two IEEE round-to-nearest operations in the same order.
        // norm: pairwise tree sq_i += sq_{i+w}, w = D/2, ..., 1 (squares exact)
        float2 sq[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sq[i] = __fmul2_rn(x[i], x[i]);
        // levels w >= 32 pair slices lt and lt + w/32 (the lower slice keeps the sum)
#pragma unroll
        for (int w = D / 2; w >= 32; w >>= 1) {
            const int off = w / 32;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 o = make_float2(__shfl_down_sync(gmask, sq[i].x, off, TPV),
                                             __shfl_down_sync(gmask, sq[i].y, off, TPV));
                sq[i] = __fadd2_rn(sq[i], o);  // meaningful on slices lt < off
            }
        }
        // levels w = 16, ..., 2: element i + w is pair i/2 + w/2
#pragma unroll
        for (int w = 16; w >= 2; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w / 2; ++i) sq[i] = __fadd2_rn(sq[i], sq[i + w / 2]);
        }
        const float n = __shfl_sync(gmask, __fsqrt_rn(__fadd_rn(sq[0].x, sq[0].y)), lane - lt);  // slice 0 holds the sum
        const uint32_t nmax = __reduce_max_sync(gmask, live ? __float_as_uint(n) : 0u);
        if (lane == 0) red[tid / 32] = nmax;

        // FWHT, stages h = 1, 2, ..., D/2, lower index first; h = 1 inside
        // each pair, h = 2 ... 16 between pairs i and i + h/2
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
        for (int hh = 32; hh < D; hh <<= 1) {
            const int off = hh / 32;
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

        // thresholds m_j * n; codes = number of thresholds exceeded (0 past the context)
        float tau[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) tau[j] = (j < L - 1) ? __fmul_rn(cb.m[j], n) : 0.f;
        uint32_t cw[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) cw[w] = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t code = live ? bucket<L>((i & 1) ? x[i / 2].y : x[i / 2].x, tau) : 0u;
            cw[i / 4] |= code << (8 * (i % 4));
        }
        uint4* c8 = reinterpret_cast<uint4*>(codes8 + tl * D + lt * 32);
        c8[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        c8[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        if (live && lt == 0) Ly.vnorm[(long long)h * ctx_pad + t_base + t0 + tl] = n;
        __syncthreads();  // codes8 and red[] complete
        if (tid == 0) {
            uint32_t nm = red[0];
#pragma unroll
            for (int w = 1; w < kEncThreads / 32; ++w) nm = max(nm, red[w]);
            snm[k] = nm;  // flushed after the dependency wait, once the word is cleared
        }

        // pool layout: one thread per (32-token group of the item, coordinate)
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
            // only groups holding tokens of this encode: a group past its end
            // belongs to a later append (or lies past the head's codes)
            const int gl = t0 / 32 + gq;  // group within the encode
            if (gl * 32 < ctx) {
                uint32_t* out = reinterpret_cast<uint32_t*>(Ly.vcodes + h * Ly.vhead + Ly.voff +
                                                            ((long long)gl * D + c) * (4 * BITS));
#pragma unroll
                for (int w = 0; w < BITS; ++w) out[w] = words[w];
                if (Ly.gbits && h == 0 && c == 0) {  // the group's width and offset, once per layer
                    const int g = t_base / 32 + gl;
                    Ly.gbits[g] = (uint8_t)BITS;
                    Ly.goff[g] = (uint32_t)(Ly.voff + (long long)gl * D * 4 * BITS);
                }
            }
        }

    }

    // ---- pass 2: K. The max|K| kernel is complete: s and 1/s of every layer
    // are written and the largest-V-norm words cleared.
    ptx::grid_dep_wait();
    float s1 = 1.0f, r1 = 1.0f;  // one layer: s and 1/s from the partial maxima
    if constexpr (NB == 1 && !KB) {
        const EncLayer& Ly = b.L[0];
        uint32_t m = 0;
        for (int i = tid; i < nparts; i += kEncThreads) m = max(m, Ly.kpart[i]);
        m = __reduce_max_sync(gmask, m);
        __syncthreads();  // thread 0 may still read red[] of the last V item
        if (lane == 0) red[tid / 32] = m;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kEncThreads / 32; ++w) m = max(m, red[w]);
        s1 = (m == 0) ? 1.0f : __fdiv_rn(__uint_as_float(m << 16), 127.0f);
        r1 = __frcp_rn(s1);
        if (blockIdx.x == 0 && tid == 0) {
            *Ly.kscale = s1;
            Ly.maxima[0] = m;
            if (m >= 0x7F80u) atomicOr(status, kStNonfinite);
        }
    }
    for (int it = blockIdx.x, k = 0; it < items; it += G, ++k) {
        const int t = m + k;
        const unsigned char* sK = tiles[t & 1];
        const EncLayer& Ly = b.L[item_l(it)];
        const int h = item_h(it), t0 = item_t0(it);
        const int ntok = min(VPI, ctx - t0);
        if (tid == 0) {
            const uint32_t nm = snm[k];
            if (nm > *reinterpret_cast<volatile uint32_t*>(&Ly.maxima[1])) atomicMax(&Ly.maxima[1], nm);
            if (nm >= 0x7F800000u) atomicOr(status, kStNonfinite);
        }
        float s = s1, r = r1;
        if constexpr (!KB && NB > 1) {
            s = *Ly.kscale;
            r = __uint_as_float(Ly.kpart[kKmaxInv]);
        }
        // q = clamp(rint(k / s), -127, 127), 8 elements per 16-byte chunk
        wait_tile(t);
        {
            uint32_t dep = 0;
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int idx = tid + c * kEncThreads;
                const int row = idx / (D / 8);
                if constexpr (KB) {
                    // the 4 chunks of a 32-element block sit in lanes 4j..4j+3
                    // (same row); every lane takes part in the shuffles
                    const uint4 u = (row < ntok) ? reinterpret_cast<const uint4*>(sK)[idx] : make_uint4(0, 0, 0, 0);
                    uint32_t m = absmax8(u);
                    m = max(m, __shfl_xor_sync(gmask, m, 1));
                    m = max(m, __shfl_xor_sync(gmask, m, 2));
                    const float sb = (m == 0) ? 1.0f : __fdiv_rn(__uint_as_float(m << 16), 127.0f);
                    if (row < ntok) {
                        const uint2 q = quant8(u, sb, __frcp_rn(sb));
                        dep ^= q.x ^ u.x;
                        const long long tok_i = (long long)h * ctx_pad + t_base + t0 + row;
                        *reinterpret_cast<uint2*>(Ly.kq + tok_i * D + (idx % (D / 8)) * 8) = q;
                        if ((idx & 3) == 0) Ly.kscales[tok_i * (D / 32) + (idx % (D / 8)) / 4] = sb;
                        if (m >= 0x7F80u) atomicOr(status, kStNonfinite);
                    }
                } else if (row < ntok) {
                    const uint4 u = reinterpret_cast<const uint4*>(sK)[idx];
                    const uint2 q = quant8(u, s, r);
                    dep ^= q.x;
                    *reinterpret_cast<uint2*>(Ly.kq + ((long long)h * ctx_pad + t_base + t0 + row) * D +
                                              (idx % (D / 8)) * 8) = q;
                }
            }
            sDep[tid] = dep;  // as for the V tile
        }
        __syncthreads();
        next_tile(t);
    }
    if (tid == 0 && !ok) atomicOr(status, kStTimeout);
}

template <int D, int BITS, int NB>
cudaError_t run_encode(const Shape& s, const EncBatchT<NB>& b, int* status, int sm_count, int t_base, bool kb,
                       int nparts, cudaStream_t st) {
    constexpr int VPI = kEncThreads / (D / 32);
    auto kern = kb ? encode_kernel<D, BITS, true, NB> : encode_kernel<D, BITS, false, NB>;
    const int items_per_head = (s.ctx + VPI - 1) / VPI;
    const int items_per_layer = s.kv_heads * items_per_head;
    const long long items_ll = (long long)b.n * items_per_layer;
    if (items_ll > INT32_MAX) return cudaErrorInvalidValue;
    const int items = (int)items_ll;
    // grid: all CTAs resident; each keeps one word per item it takes
    int occ = 0, G = 0;
    size_t dyn = 0;
    for (int pass = 0; pass < 3; ++pass) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kEncThreads, dyn);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        G = std::min(items, occ * sm_count);
        const size_t need = (size_t)((items + G - 1) / G) * sizeof(uint32_t);
        if (need <= dyn) break;
        dyn = need;
    }
    if ((size_t)((items + G - 1) / G) * sizeof(uint32_t) > dyn) return cudaErrorInvalidConfiguration;
    if (dyn > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return e;
    }
    // starts while the max|K| kernel runs (programmatic dependent launch)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, 1, 1);
    cfg.blockDim = dim3(kEncThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, b, s.ctx, s.ctx_pad, t_base, items_per_head, items_per_layer, items,
                              nparts, status, codebook(BITS));
}

template <int D, int NB>
cudaError_t run_bits(int bits, const Shape& s, const EncBatchT<NB>& b, int* status, int sm_count, int t_base, bool kb,
                     int nparts, cudaStream_t st) {
    if (bits == 2) return run_encode<D, 2, NB>(s, b, status, sm_count, t_base, kb, nparts, st);
    if (bits == 3) return run_encode<D, 3, NB>(s, b, status, sm_count, t_base, kb, nparts, st);
    return run_encode<D, 4, NB>(s, b, status, sm_count, t_base, kb, nparts, st);
}

EncLayer enc_layer(const LayerBufs& L, const void* K, const void* V, long long voff) {
    EncLayer e;
    e.vhead = L.vhead;
    e.voff = voff;
    e.gbits = L.gbits;
    e.goff = L.goff;
    e.K = static_cast<const uint16_t*>(K);
    e.V = static_cast<const uint16_t*>(V);
    e.kq = L.kq;
    e.vcodes = L.vcodes;
    e.vnorm = L.vnorm;
    e.kscale = L.kscale;
    e.maxima = L.kabsmax;  // {max|K| bits, largest V norm bits}: adjacent words
    e.kpart = L.kpart;
    e.kscales = L.kscales;
    return e;
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

namespace {

// max|K| and encode launches for nc layers of a table of capacity NB
template <int NB>
cudaError_t launch_chunk(const Shape& s, const LayerBufs* L, const void* const* K, const void* const* V, int nc,
                         int* status, int sm_count, int t_base, long long voff, cudaStream_t st) {
    const bool kb = L[0].kscales != nullptr;
    // max|K| of every layer in one launch: about two CTAs per SM in all, so
    // that they are all running when the encode kernel starts
    EncBatchT<NB> all = {};
    all.n = nc;
    for (int i = 0; i < nc; ++i) all.L[i] = enc_layer(L[i], K[i], V[i], voff);
    const long long nchunk = (long long)s.kv_heads * s.ctx * (s.head_dim / 8);
    const int gx = kb ? 1 : std::max(1, std::min(kKmaxInv, (2 * sm_count + nc - 1) / nc));
    const long long per_cta = (nchunk + gx - 1) / gx;
    kmax_kernel<NB><<<dim3(gx, nc), 256, 0, st>>>(all, nchunk, per_cta, kb ? 1 : 0, t_base == 0 ? 1 : 0, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // one encode launch per V width among the layers
    for (int bits = 2; bits <= 4; ++bits) {
        EncBatchT<NB> sub = {};
        for (int i = 0; i < nc; ++i)
            if (L[i].bits == bits) sub.L[sub.n++] = all.L[i];
        if (sub.n == 0) continue;
        e = s.head_dim == 64 ? run_bits<64, NB>(bits, s, sub, status, sm_count, t_base, kb, gx, st)
                             : run_bits<128, NB>(bits, s, sub, status, sm_count, t_base, kb, gx, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_encode_layers(const Shape& s, const LayerBufs* L, const void* const* K, const void* const* V,
                                 int n, int* status, int sm_count, int t_base, long long voff,
                                 cudaStream_t st) {
    if (n < 1) return cudaErrorInvalidValue;
    const bool kb = L[0].kscales != nullptr;
    if ((t_base != 0 || voff != 0) && (!kb || n != 1 || t_base % 32 != 0)) return cudaErrorInvalidValue;
    for (int i = 0; i < n; ++i)
        if (L[i].vhead <= 0) return cudaErrorInvalidValue;
    if (n == 1) return launch_chunk<1>(s, L, K, V, 1, status, sm_count, t_base, voff, st);
    for (int c0 = 0; c0 < n; c0 += kEncBatch) {
        const int nc = std::min(kEncBatch, n - c0);
        const cudaError_t e =
            launch_chunk<kEncBatch>(s, L + c0, K + c0, V + c0, nc, status, sm_count, t_base, voff, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_encode(const Shape& s, const LayerBufs& L, const void* K, const void* V,
                          int* status, int sm_count, int t_base, long long voff, cudaStream_t st) {
    return launch_encode_layers(s, &L, &K, &V, 1, status, sm_count, t_base, voff, st);
}

}  // namespace kvp
