// Host side of the C-ABI: argument validation, the write-once state of each
// layer, the single device allocation of the pool, the library's own
// Lloyd-Max table, status reporting.
//
// Memory layout of a pool (one cudaMalloc, every region 256-byte aligned):
//   per layer l:  kq     int8  [Hk][ctx_pad][D]
//                 vcodes uint8 [Hk][ctx_pad/32][D][4*bits_l] (32-token groups)
//                 vnorm  f32   [Hk][ctx_pad]
//   kscale f32 [layers], per layer two u32 words {max|K| bf16 bits, largest
//   V norm float bits}, per layer 512 words of compress scratch (partial
//   maxima of max|K|, 1/s, the max|K| kernel's arrival counter), status int32. Block-scaled pools (kvpool_create_ex, k_block 32)
//   also hold per layer kscales f32 [Hk][ctx_pad][D/32].
// Attention needs no scratch: the CTAs of a cluster merge their context
// splits through distributed shared memory. Each layer also has a TMA tensor
// map of its kq (rows of head_dim bytes) for the attention kernel.
// ctx_pad rounds the token axis up to a multiple of 128 so tiles never leave a
// layer; the padding is zeroed once and never counted as tokens.
#include <math.h>

#include <cmath>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>
#include <new>
#include <vector>

#include "kvpool_internal.cuh"

// ----------------------------------------------------------- Lloyd-Max table
namespace kvp {
namespace {

// N(0,1) density and upper tail (double precision: the table is rounded to
// float32 in the end).
double npdf(double x) { return exp(-0.5 * x * x) * 0.3989422804014327; }
double ntail(double x) { return 0.5 * erfc(x * 0.7071067811865476); }

// Lloyd-Max quantiser for N(0,1) with `levels` (even) outputs. N(0,1) is
// symmetric, so only the positive half is solved, with cell edges 0 = e_0 <
// e_1 < ... < e_K = inf (K = levels/2): iterate
//   y_k = (pdf(e_{k-1}) - pdf(e_k)) / (tail(e_{k-1}) - tail(e_k)),
//   e_k = (y_k + y_{k+1}) / 2
// from equally spaced edges on [0, 3] until the edges stop moving.
void lloyd_max(int levels, double* pos /* K outputs */) {
    const int K = levels / 2;
    double e[9];
    e[0] = 0.0;
    for (int k = 1; k < K; ++k) e[k] = 3.0 * k / K;
    double y[8];
    for (int it = 0; it < 20000; ++it) {
        for (int k = 0; k < K; ++k) {
            const double hi_pdf = (k + 1 < K) ? npdf(e[k + 1]) : 0.0;
            const double hi_tail = (k + 1 < K) ? ntail(e[k + 1]) : 0.0;
            y[k] = (npdf(e[k]) - hi_pdf) / (ntail(e[k]) - hi_tail);
        }
        double moved = 0.0;
        for (int k = 1; k < K; ++k) {
            const double ne = 0.5 * (y[k - 1] + y[k]);
            moved = fmax(moved, fabs(ne - e[k]));
            e[k] = ne;
        }
        if (moved == 0.0) break;
    }
    for (int k = 0; k < K; ++k) pos[k] = y[k];
}

// float -> fp16 bits, round to nearest even (normal range; the table values
// are between 0.1 and 6)
uint16_t half_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const int e = (int)((x >> 23) & 0xFF) - 127 + 15;
    uint32_t mant = x & 0x7FFFFFu;
    if (e <= 0 || e >= 31) return (uint16_t)sign;  // not reached for the table
    uint32_t h = ((uint32_t)e << 10) | (mant >> 13);
    const uint32_t rest = mant & 0x1FFFu;
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1))) ++h;
    return (uint16_t)(sign | h);
}
double half_value(uint16_t h) {
    const int e = (h >> 10) & 0x1F;
    const double m = (double)(h & 0x3FF);
    const double v = ldexp(1.0 + m / 1024.0, e - 15);
    return (h & 0x8000) ? -v : v;
}

// Scale lam in [1, 2) minimising the largest relative fp16 rounding error of
// lam * c over the n positive centroids pos (the tables are antisymmetric).
float pick_lambda(const double* pos, int n) {
    double best = 1e30;
    float best_lam = 1.0f;
    for (int i = 0; i < (1 << 20); ++i) {
        const float lam = 1.0f + (float)i / (float)(1 << 20);
        double worst = 0.0;
        for (int k = 0; k < n; ++k) {
            const double v = (double)(float)((double)lam * pos[k]);
            const double e = fabs(half_value(half_bits((float)v)) - (double)lam * pos[k]) / ((double)lam * pos[k]);
            if (e > worst) worst = e;
            if (worst >= best) break;
        }
        if (worst < best) {
            best = worst;
            best_lam = lam;
        }
    }
    return best_lam;
}

Codebook g_books[5];
MixBook g_mix;
std::once_flag g_books_once;

void build_books() {
    double allpos[14];  // positive centroids of the three widths
    int npos = 0;
    double cen[5][16];
    for (int bits = 2; bits <= 4; ++bits) {
        Codebook& b = g_books[bits];
        const int L = 1 << bits, K = L / 2;
        double pos[8];
        lloyd_max(L, pos);
        double c[16];
        for (int k = 0; k < K; ++k) {
            c[K + k] = pos[k];
            c[K - 1 - k] = -pos[k];
        }
        for (int k = 0; k < 16; ++k) b.c[k] = (k < L) ? (float)c[k] : 0.0f;
        for (int k = 0; k < 16; ++k) b.m[k] = (k < L - 1) ? (float)(0.5 * (c[k] + c[k + 1])) : 0.0f;
        b.levels = L;
        b.bits = bits;
        b.lam = pick_lambda(c + K, K);
        for (int k = 0; k < 16; ++k)
            b.c16[k] = (k < L) ? half_bits((float)((double)b.lam * c[k])) : (uint16_t)0;
        for (int k = 0; k < 16; ++k) cen[bits][k] = k < L ? c[k] : 0.0;
        for (int k = 0; k < K; ++k) allpos[npos++] = c[K + k];
    }
    g_mix.lam = pick_lambda(allpos, npos);
    for (int bits = 2; bits <= 4; ++bits)
        for (int k = 0; k < 16; ++k)
            g_mix.c16[bits - 2][k] =
                k < (1 << bits) ? half_bits((float)((double)g_mix.lam * cen[bits][k])) : (uint16_t)0;
}

}  // namespace

const Codebook& codebook(int bits) {
    std::call_once(g_books_once, build_books);
    return g_books[bits];
}

const MixBook& mixbook() {
    std::call_once(g_books_once, build_books);
    return g_mix;
}

// Mean squared error of the Lloyd-Max quantiser for N(0,1) at `bits` bits,
// in closed form per cell: E[(X - y)^2; a < X < b] = P (1 + y^2)
// - 2 y (pdf(a) - pdf(b)) + (a pdf(a) - b pdf(b)); twice the positive half.
double lm_distortion(int bits) {
    const int L = 1 << bits, K = L / 2;
    double y[8];
    lloyd_max(L, y);
    double total = 0.0;
    for (int k = 0; k < K; ++k) {
        const double a = (k == 0) ? 0.0 : 0.5 * (y[k - 1] + y[k]);
        const bool last = k + 1 == K;
        const double b = last ? 0.0 : 0.5 * (y[k] + y[k + 1]);
        const double P = ntail(a) - (last ? 0.0 : ntail(b));
        const double pa = npdf(a), pb = last ? 0.0 : npdf(b);
        total += P * (1.0 + y[k] * y[k]) - 2.0 * y[k] * (pa - pb) + (a * pa - (last ? 0.0 : b * pb));
    }
    return 2.0 * total;
}


}  // namespace kvp

// ---------------------------------------------------------------- the pool
struct kvpool {
    int layers = 0, kv_heads = 0, head_dim = 0, ctx = 0, ctx_pad = 0, max_rows = 0;
    int device = 0, sm_count = 0;
    int k_block = 0;  // 0: one K scale per layer; 32: one per 32 elements
    std::vector<int> bits;  // per layer: the width fixed at create (the largest a group may take)
    std::vector<size_t> off_kq, off_vc, off_vn, off_ks, off_gt;
    // block-scaled pools: the width of every written 32-token group of a layer
    // (its device copy, with the groups' byte offsets, is written by the
    // encode kernel)
    std::vector<std::vector<uint8_t>> gw;
    std::vector<unsigned char> compressed;
    std::vector<int> len;  // tokens the layer holds: ctx once compressed; grows by appends
    // Per stream: the layer that this pool's most recent launch on it wrote,
    // -1 for none, kWroteMany for several (a multi-layer compress). An attend
    // may read its layer before the grid-dependency wait (programmatic
    // dependent launch) unless the launch right before it on the same stream
    // wrote that layer. The kernels that write a layer (the encode) never
    // release their dependents before they finish, so once any later launch
    // has started, the writer is complete; only a writer launched right
    // before the attend can be finishing as the attend starts.
    static constexpr int kWroteMany = -2;
    std::unordered_map<void*, int> last_write;
    std::mutex mu;  // last_write: attends may come from several host threads
    void wrote(void* stream, int layer) {
        std::lock_guard<std::mutex> g(mu);
        last_write[stream] = layer;
    }
    bool may_read_early(void* stream, int layer) {
        std::lock_guard<std::mutex> g(mu);
        auto it = last_write.find(stream);
        return it == last_write.end() || (it->second != layer && it->second != kWroteMany);
    }
    std::vector<CUtensorMap> kmaps;
    unsigned char* base = nullptr;
    size_t bytes = 0;
    float* kscale = nullptr;
    uint32_t* kabsmax = nullptr;
    uint32_t* kpart = nullptr;
    int* status = nullptr;

    kvp::Shape shape() const { return {kv_heads, head_dim, ctx, ctx_pad}; }
    // the layer's current tokens (attend, decompress, export read [0, len))
    kvp::Shape shape_of(int l) const { return {kv_heads, head_dim, len[l], ctx_pad}; }
    int groups() const { return ctx_pad / 32; }
    // 1 when the layer's written groups do not all have its create width
    int mixed(int l) const {
        for (uint8_t b : gw[l])
            if (b != bits[l]) return 1;
        return 0;
    }
    // byte offset within a KV head's codes of the layer's group g (g <= groups written)
    long long group_offset(int l, int g) const {
        long long o = 0;
        for (int i = 0; i < g; ++i) o += (long long)head_dim * 4 * gw[l][i];
        return o;
    }
    kvp::LayerBufs layer(int l) const {
        kvp::LayerBufs L{reinterpret_cast<int8_t*>(base + off_kq[l]), base + off_vc[l],
                         reinterpret_cast<float*>(base + off_vn[l]), kscale + l, kabsmax + 2 * l, bits[l],
                         kabsmax + 2 * l + 1, &kmaps[l], kpart + (size_t)l * kvp::kKmaxParts,
                         k_block ? reinterpret_cast<float*>(base + off_ks[l]) : nullptr};
        L.vhead = (long long)ctx_pad * head_dim * bits[l] / 8;
        if (k_block) {
            L.gbits = base + off_gt[l];
            L.goff = reinterpret_cast<uint32_t*>(base + off_gt[l] + align_groups());
            L.mixed = mixed(l);
        }
        return L;
    }
    // group table of a layer: widths [groups] (u8), then offsets [groups] (u32)
    size_t align_groups() const { return ((size_t)groups() + 255) & ~size_t(255); }
    size_t group_table_bytes() const { return align_groups() + (size_t)groups() * 4; }
};

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int map_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KVPOOL_OK;
    if (e == cudaErrorMemoryAllocation) return KVPOOL_ERR_OOM;
    return KVPOOL_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// cuTensorMapEncodeTiled, fetched from the driver at run time (the library
// does not link libcuda).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);
EncodeTiled tensor_map_encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// kq of one layer as a 2-D tensor of Hk*ctx_pad rows of D bytes; boxes of 128
// rows land in shared memory with the 128-byte (D = 128) or 64-byte (D = 64)
// swizzle that the attention kernel reads.
bool make_kmap(CUtensorMap* map, void* kq, int D, long long rows) {
    EncodeTiled enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)D};
    const cuuint32_t box[2] = {(cuuint32_t)D, 128};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kq, gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_layer(const kvpool* p, int layer) {
    if (!p || layer < 0 || layer >= p->layers) return KVPOOL_ERR_INVALID_ARG;
    return KVPOOL_OK;
}

}  // namespace

extern "C" {

int kvpool_codebook(int bits, float* centroids, float* midpoints) {
    if (bits < 2 || bits > 4) return KVPOOL_ERR_INVALID_ARG;
    const kvp::Codebook& b = kvp::codebook(bits);
    for (int k = 0; k < b.levels; ++k) {
        if (centroids) centroids[k] = b.c[k];
        if (midpoints && k < b.levels - 1) midpoints[k] = b.m[k];
    }
    return KVPOOL_OK;
}

int kvpool_create(kvpool_t** out, int layers, int kv_heads, int head_dim, int ctx,
                  const uint8_t* bits_per_layer, int max_rows) {
    return kvpool_create_ex(out, layers, kv_heads, head_dim, ctx, bits_per_layer, max_rows, 0);
}

int kvpool_create_ex(kvpool_t** out, int layers, int kv_heads, int head_dim, int ctx,
                     const uint8_t* bits_per_layer, int max_rows, int k_block) {
    if (!out) return KVPOOL_ERR_INVALID_ARG;
    if (k_block != 0 && k_block != 32) return KVPOOL_ERR_INVALID_ARG;
    *out = nullptr;
    if (layers < 1 || kv_heads < 1 || ctx < 1 || (head_dim != 64 && head_dim != 128))
        return KVPOOL_ERR_INVALID_ARG;
    if (max_rows == 0) max_rows = 512;
    if (max_rows < 1 || max_rows > 1024) return KVPOOL_ERR_INVALID_ARG;
    if ((long long)kv_heads * ctx > (1LL << 31) / 128) return KVPOOL_ERR_INVALID_ARG;
    if (bits_per_layer)
        for (int l = 0; l < layers; ++l)
            if (bits_per_layer[l] < 2 || bits_per_layer[l] > 4) return KVPOOL_ERR_INVALID_ARG;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return KVPOOL_ERR_UNSUPPORTED;
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return map_cuda(e);
    if (prop.major * 10 + prop.minor != 103) return KVPOOL_ERR_UNSUPPORTED;

    kvpool* p = new (std::nothrow) kvpool;
    if (!p) return KVPOOL_ERR_OOM;
    p->layers = layers;
    p->kv_heads = kv_heads;
    p->head_dim = head_dim;
    p->ctx = ctx;
    p->ctx_pad = (ctx + kvp::kTokenPad - 1) / kvp::kTokenPad * kvp::kTokenPad;
    p->max_rows = max_rows;
    p->k_block = k_block;
    p->device = dev;
    p->sm_count = prop.multiProcessorCount;
    p->bits.resize(layers);
    p->compressed.assign(layers, 0);
    p->len.assign(layers, 0);
    p->gw.resize(layers);
    size_t off = 0;
    const size_t nvec = (size_t)kv_heads * p->ctx_pad;
    for (int l = 0; l < layers; ++l) {
        p->bits[l] = bits_per_layer ? bits_per_layer[l] : 3;
        p->off_kq.push_back(off);
        off = align256(off + nvec * head_dim);
        p->off_vc.push_back(off);
        off = align256(off + nvec * head_dim * p->bits[l] / 8);
        p->off_vn.push_back(off);
        off = align256(off + nvec * 4);
        p->off_ks.push_back(off);
        if (k_block) off = align256(off + nvec * (head_dim / k_block) * 4);
        p->off_gt.push_back(off);
        if (k_block) off = align256(off + p->group_table_bytes());
    }
    const size_t off_scale = off;
    off = align256(off + 4 * (size_t)layers);
    const size_t off_absmax = off;  // per layer {max|K| bits, largest V norm bits}
    off = align256(off + 8 * (size_t)layers);
    const size_t off_kpart = off;  // per layer: compress scratch (partial maxima, 1/s, arrival counter)
    off = align256(off + 4 * (size_t)kvp::kKmaxParts * layers);
    const size_t off_status = off;
    off = align256(off + 4);
    p->bytes = off;
    e = cudaMalloc(reinterpret_cast<void**>(&p->base), p->bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return map_cuda(e);
    }
    e = cudaMemset(p->base, 0, p->bytes);
    if (e != cudaSuccess) {
        cudaFree(p->base);
        delete p;
        return map_cuda(e);
    }
    p->kscale = reinterpret_cast<float*>(p->base + off_scale);
    p->kabsmax = reinterpret_cast<uint32_t*>(p->base + off_absmax);
    p->kpart = reinterpret_cast<uint32_t*>(p->base + off_kpart);
    p->status = reinterpret_cast<int*>(p->base + off_status);
    p->kmaps.resize(layers);
    for (int l = 0; l < layers; ++l) {
        if (!make_kmap(&p->kmaps[l], p->base + p->off_kq[l], head_dim, (long long)nvec)) {
            cudaFree(p->base);
            delete p;
            return KVPOOL_ERR_UNSUPPORTED;
        }
    }
    kvp::codebook(2);  // derive the tables now, not inside a stream capture
    *out = p;
    return KVPOOL_OK;
}

void kvpool_destroy(kvpool_t* p) {
    if (!p) return;
    cudaDeviceSynchronize();
    cudaFree(p->base);
    delete p;
}

int kvpool_compress(kvpool_t* p, int layer, const void* K, const void* V, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!K || !V || !aligned16(K) || !aligned16(V)) return KVPOOL_ERR_INVALID_ARG;
    if (p->compressed[layer]) return KVPOOL_ERR_STATE;
    cudaError_t e = kvp::launch_encode(p->shape(), p->layer(layer), K, V, p->status, p->sm_count, 0, 0,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return map_cuda(e);
    p->compressed[layer] = 1;
    p->len[layer] = p->ctx;
    if (p->k_block) p->gw[layer].assign((p->ctx + 31) / 32, (uint8_t)p->bits[layer]);
    p->wrote(stream, layer);
    return KVPOOL_OK;
}

int kvpool_compress_layers(kvpool_t* p, int n, const int* layers, const void* const* K, const void* const* V,
                           void* stream) {
    if (!p || n < 1 || !layers || !K || !V) return KVPOOL_ERR_INVALID_ARG;
    std::vector<char> seen(p->layers, 0);
    for (int i = 0; i < n; ++i) {
        const int l = layers[i];
        if (l < 0 || l >= p->layers || seen[l]) return KVPOOL_ERR_INVALID_ARG;
        seen[l] = 1;
        if (!K[i] || !V[i] || !aligned16(K[i]) || !aligned16(V[i])) return KVPOOL_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i)
        if (p->compressed[layers[i]]) return KVPOOL_ERR_STATE;
    std::vector<kvp::LayerBufs> L(n);
    for (int i = 0; i < n; ++i) L[i] = p->layer(layers[i]);
    cudaError_t e = kvp::launch_encode_layers(p->shape(), L.data(), K, V, n, p->status, p->sm_count, 0, 0,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return map_cuda(e);
    for (int i = 0; i < n; ++i) {
        p->compressed[layers[i]] = 1;
        p->len[layers[i]] = p->ctx;
        if (p->k_block) p->gw[layers[i]].assign((p->ctx + 31) / 32, (uint8_t)p->bits[layers[i]]);
    }
    p->wrote(stream, n == 1 ? layers[0] : kvpool::kWroteMany);
    return KVPOOL_OK;
}

int kvpool_append(kvpool_t* p, int layer, const void* K, const void* V, int n, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    return kvpool_append_bits(p, layer, K, V, n, p->bits[layer], stream);
}

int kvpool_append_bits(kvpool_t* p, int layer, const void* K, const void* V, int n, int bits, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!K || !V || !aligned16(K) || !aligned16(V) || n < 1) return KVPOOL_ERR_INVALID_ARG;
    if (!p->k_block) return KVPOOL_ERR_UNSUPPORTED;
    if (bits < 2 || bits > p->bits[layer]) return KVPOOL_ERR_INVALID_ARG;
    const int len = p->len[layer];
    if (len % 32 != 0) return KVPOOL_ERR_STATE;  // a ragged append closed the layer
    if ((long long)len + n > p->ctx) return KVPOOL_ERR_INVALID_ARG;
    const kvp::Shape s{p->kv_heads, p->head_dim, n, p->ctx_pad};
    kvp::LayerBufs L = p->layer(layer);
    L.bits = bits;  // the width these tokens are coded at
    const long long voff = p->group_offset(layer, len / 32);
    cudaError_t e = kvp::launch_encode(s, L, K, V, p->status, p->sm_count, len, voff,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return map_cuda(e);
    p->len[layer] = len + n;
    p->compressed[layer] = 1;
    p->gw[layer].resize((len + n + 31) / 32, (uint8_t)bits);
    p->wrote(stream, layer);
    return KVPOOL_OK;
}

int kvpool_layer_widths(const kvpool_t* p, int layer, uint8_t* widths, int max_groups) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (max_groups < 0 || (max_groups > 0 && !widths)) return KVPOOL_ERR_INVALID_ARG;
    const int ng = (p->len[layer] + 31) / 32;
    for (int g = 0; g < ng && g < max_groups; ++g)
        widths[g] = p->k_block ? p->gw[layer][g] : (uint8_t)p->bits[layer];
    return ng;
}

int kvpool_layer_len(const kvpool_t* p, int layer) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    return p->len[layer];
}

namespace {

// Validation shared by the attend calls: fills a (no slice, no partial mode).
int attend_args(kvpool_t* p, int layer, const void* Q, int agents, int q_heads, const kvpool_tail_t* tail,
                float* out, float softmax_scale, void* stream, kvp::AttendArgs& a) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!Q || !out || agents < 1 || q_heads < p->kv_heads || q_heads % p->kv_heads)
        return KVPOOL_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(out)) return KVPOOL_ERR_INVALID_ARG;
    if (!(softmax_scale >= 0.0f) || isinf(softmax_scale)) return KVPOOL_ERR_INVALID_ARG;
    const int group = q_heads / p->kv_heads;
    if ((long long)agents * group > p->max_rows) return KVPOOL_ERR_INVALID_ARG;
    if (tail && (tail->T_max < 0 || (tail->T_max > 0 && (!tail->K || !tail->V || !tail->len))))
        return KVPOOL_ERR_INVALID_ARG;
    if (tail && tail->T_max > 0 && (!aligned16(tail->K) || !aligned16(tail->V) ||
                                    (reinterpret_cast<uintptr_t>(tail->len) & 3)))
        return KVPOOL_ERR_INVALID_ARG;
    if (!p->compressed[layer]) return KVPOOL_ERR_STATE;
    a = kvp::AttendArgs{};
    a.Q = Q;
    a.agents = agents;
    a.q_heads = q_heads;
    a.group = group;
    a.rows = agents * group;
    const bool has_tail = tail && tail->T_max > 0;
    a.tailK = has_tail ? tail->K : nullptr;
    a.tailV = has_tail ? tail->V : nullptr;
    a.tail_len = has_tail ? tail->len : nullptr;
    a.tail_max = has_tail ? tail->T_max : 0;
    a.out = out;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)p->head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.early = p->may_read_early(stream, layer) ? 1 : 0;
    a.t0 = 0;
    a.t1 = p->len[layer];
    return KVPOOL_OK;
}

// Workspace of kvpool_attend_ws for rows query rows per KV head: the most
// slices per (KV head, row group) one wave of CTAs can hold, and the byte
// offset of the accumulators (after the (m, l) pairs).
struct WsLayout {
    long long nslice_max;
    size_t acc_off, tail_off, bytes;
};
WsLayout ws_layout(const kvpool* p, long long rows, int group) {
    // row groups as the tensor-core launcher forms them (at most 64 rows in
    // all: groups of <= 64 rows; else <= 128), whole agents each
    const bool spread = rows <= 64;
    const long long RW = ((spread ? 64 : 128) / group) * group;
    WsLayout w{0, 0, 0, 0};
    if (RW < 1) return w;
    const long long jobs = (long long)p->kv_heads * ((rows + RW - 1) / RW);
    const long long ntiles = (p->ctx + kvp::kTokenPad - 1) / kvp::kTokenPad;
    w.nslice_max = std::min(ntiles, (long long)p->sm_count / jobs);
    if (w.nslice_max < 1) return w;
    const size_t per = (size_t)p->kv_heads * rows;  // partial rows per slice
    w.acc_off = align256((size_t)w.nslice_max * per * 2 * sizeof(float));
    // then the rows' tail (m, l), for calls with tails
    w.tail_off = align256(w.acc_off + (size_t)w.nslice_max * per * p->head_dim * sizeof(float));
    w.bytes = w.tail_off + per * 2 * sizeof(float);
    return w;
}

}  // namespace

int kvpool_attend(kvpool_t* p, int layer, const void* Q, int agents, int q_heads,
                  const kvpool_tail_t* tail, float* out, float softmax_scale, void* stream) {
    kvp::AttendArgs a;
    const int rc = attend_args(p, layer, Q, agents, q_heads, tail, out, softmax_scale, stream, a);
    if (rc) return rc;
    const cudaError_t e = kvp::launch_attend_tc(p->shape_of(layer), p->layer(layer), a, p->status, p->sm_count,
                                                static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) p->wrote(stream, -1);
    return map_cuda(e);
}

size_t kvpool_attend_ws_bytes(const kvpool_t* p, int agents, int q_heads) {
    if (!p || agents < 1 || q_heads < p->kv_heads || q_heads % p->kv_heads) return 0;
    const int group = q_heads / p->kv_heads;
    if ((long long)agents * group > p->max_rows) return 0;
    return ws_layout(p, (long long)agents * group, group).bytes;
}

int kvpool_attend_ws(kvpool_t* p, int layer, const void* Q, int agents, int q_heads, const kvpool_tail_t* tail,
                     float* out, float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
    kvp::AttendArgs a;
    const int rc = attend_args(p, layer, Q, agents, q_heads, tail, out, softmax_scale, stream, a);
    if (rc) return rc;
    const WsLayout w = ws_layout(p, a.rows, a.group);
    if (w.bytes == 0) return KVPOOL_ERR_UNSUPPORTED;  // more row groups than one wave of CTAs
    if (!workspace || !aligned16(workspace) || workspace_bytes < w.bytes) return KVPOOL_ERR_INVALID_ARG;
    // slices of the context, one CTA each, their partial states into the
    // workspace (and each slice's share of the agents' tails); then the
    // log-sum-exp merge with the tails and the inverse FWHT
    kvp::AttendArgs pa = a;
    if (a.tailK != nullptr) {
        pa.ws_tail_ml = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + w.tail_off);
        a.ws_tail_ml = pa.ws_tail_ml;
    }
    pa.part_ml = static_cast<float*>(workspace);
    pa.part_acc = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + w.acc_off);
    pa.ws_ctas = p->sm_count;  // one wave of CTAs
    pa.ws_nslice_max = (int)w.nslice_max;
    int nslice = 0;
    pa.ws_nslice = &nslice;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = kvp::launch_attend_tc(p->shape_of(layer), p->layer(layer), pa, p->status, p->sm_count, st);
    if (e == cudaSuccess && (nslice < 1 || nslice > w.nslice_max)) e = cudaErrorInvalidValue;
    if (e == cudaSuccess)
        e = kvp::launch_merge_partials(nslice, pa.part_ml, pa.part_acc, p->kv_heads, p->head_dim, a, st,
                                       p->sm_count);
    if (e == cudaSuccess) p->wrote(stream, -1);
    return map_cuda(e);
}

int kvpool_attend_partial(kvpool_t* p, int layer, const void* Q, int agents, int q_heads, int t_begin,
                          int t_end, float* part_ml, float* part_acc, float softmax_scale, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!Q || !part_ml || !part_acc || agents < 1 || q_heads < p->kv_heads || q_heads % p->kv_heads)
        return KVPOOL_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(part_acc) || (reinterpret_cast<uintptr_t>(part_ml) & 7))
        return KVPOOL_ERR_INVALID_ARG;
    if (!(softmax_scale >= 0.0f) || isinf(softmax_scale)) return KVPOOL_ERR_INVALID_ARG;
    const int group = q_heads / p->kv_heads;
    if ((long long)agents * group > p->max_rows) return KVPOOL_ERR_INVALID_ARG;
    if (!p->compressed[layer]) return KVPOOL_ERR_STATE;
    if (t_begin < 0 || t_begin % kvp::kTokenPad != 0 || t_end <= t_begin || t_end > p->len[layer])
        return KVPOOL_ERR_INVALID_ARG;
    kvp::AttendArgs a{};
    a.Q = Q;
    a.agents = agents;
    a.q_heads = q_heads;
    a.group = group;
    a.rows = agents * group;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)p->head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.early = p->may_read_early(stream, layer) ? 1 : 0;
    a.t0 = t_begin;
    a.t1 = t_end;
    a.part_ml = part_ml;
    a.part_acc = part_acc;
    const cudaError_t e = kvp::launch_attend_tc(p->shape_of(layer), p->layer(layer), a, p->status, p->sm_count,
                                                static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) p->wrote(stream, -1);
    return map_cuda(e);
}

int kvpool_merge_partials(int parts, const float* part_ml, const float* part_acc, int kv_heads, int head_dim,
                          const void* Q, int agents, int q_heads, const kvpool_tail_t* tail, float* out,
                          float softmax_scale, void* stream) {
    if (parts < 1 || parts > 4096 || !part_ml || !part_acc || !Q || !out || agents < 1 || kv_heads < 1 ||
        (head_dim != 64 && head_dim != 128) || q_heads < kv_heads || q_heads % kv_heads)
        return KVPOOL_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(part_ml) & 7) ||
        (reinterpret_cast<uintptr_t>(part_acc) & 3))
        return KVPOOL_ERR_INVALID_ARG;
    if (!(softmax_scale >= 0.0f) || isinf(softmax_scale)) return KVPOOL_ERR_INVALID_ARG;
    if (tail && (tail->T_max < 0 || (tail->T_max > 0 && (!tail->K || !tail->V || !tail->len))))
        return KVPOOL_ERR_INVALID_ARG;
    const long long rows = (long long)agents * (q_heads / kv_heads);
    if (rows > 65535 || (long long)kv_heads > 65535) return KVPOOL_ERR_INVALID_ARG;
    kvp::AttendArgs a{};
    a.Q = Q;
    a.agents = agents;
    a.q_heads = q_heads;
    a.group = q_heads / kv_heads;
    a.rows = (int)rows;
    const bool has_tail = tail && tail->T_max > 0;
    a.tailK = has_tail ? tail->K : nullptr;
    a.tailV = has_tail ? tail->V : nullptr;
    a.tail_len = has_tail ? tail->len : nullptr;
    a.tail_max = has_tail ? tail->T_max : 0;
    a.out = out;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    return map_cuda(kvp::launch_merge_partials(parts, part_ml, part_acc, kv_heads, head_dim, a,
                                               static_cast<cudaStream_t>(stream)));
}

int kvpool_decompress(kvpool_t* p, int layer, void* K_out, void* V_out, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if ((!K_out && !V_out) || !aligned16(K_out) || !aligned16(V_out)) return KVPOOL_ERR_INVALID_ARG;
    if (!p->compressed[layer]) return KVPOOL_ERR_STATE;
    const cudaError_t e = kvp::launch_decompress(p->shape_of(layer), p->layer(layer), K_out, V_out,
                                                 static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) p->wrote(stream, -1);
    return map_cuda(e);
}

int kvpool_decompress_layers(kvpool_t* p, int n, const int* layers, void* const* K_out, void* const* V_out,
                             void* stream) {
    if (!p || n < 1 || !layers || (!K_out && !V_out)) return KVPOOL_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const int l = layers[i];
        if (l < 0 || l >= p->layers) return KVPOOL_ERR_INVALID_ARG;
        if (K_out && (!K_out[i] || !aligned16(K_out[i]))) return KVPOOL_ERR_INVALID_ARG;
        if (V_out && (!V_out[i] || !aligned16(V_out[i]))) return KVPOOL_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i)
        if (!p->compressed[layers[i]]) return KVPOOL_ERR_STATE;
    std::vector<kvp::LayerBufs> L(n);
    std::vector<int> len(n);
    for (int i = 0; i < n; ++i) {
        L[i] = p->layer(layers[i]);
        len[i] = p->len[layers[i]];
    }
    const cudaError_t e = kvp::launch_decompress_layers(p->shape(), L.data(), len.data(), K_out, V_out, n,
                                                        static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) p->wrote(stream, -1);
    return map_cuda(e);
}

size_t kvpool_pool_bytes(const kvpool_t* p) {
    if (!p) return 0;
    size_t total = 0;
    const size_t nvec = (size_t)p->kv_heads * p->ctx;
    for (int l = 0; l < p->layers; ++l) {
        total += nvec * p->head_dim + nvec * p->head_dim * p->bits[l] / 8 + 4 * nvec + 4;
        if (p->k_block) total += nvec * (p->head_dim / p->k_block) * 4;
    }
    return total;
}

size_t kvpool_device_bytes(const kvpool_t* p) { return p ? p->bytes : 0; }

int kvpool_status(kvpool_t* p, void* stream) {
    if (!p) return KVPOOL_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return map_cuda(e);
    int st = 0;
    e = cudaMemcpy(&st, p->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return map_cuda(e);
    if (st) {
        e = cudaMemset(p->status, 0, sizeof(int));
        if (e != cudaSuccess) return map_cuda(e);
    }
    if (st & kvp::kStNonfinite) return KVPOOL_ERR_NONFINITE;
    if (st & kvp::kStTimeout) return KVPOOL_ERR_TIMEOUT;
    return KVPOOL_OK;
}

int kvpool_reset_layer(kvpool_t* p, int layer) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    p->compressed[layer] = 0;
    p->len[layer] = 0;
    p->gw[layer].clear();
    return KVPOOL_OK;
}

int kvpool_layer_view(const kvpool_t* p, int layer, kvpool_layer_view_t* v) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!v) return KVPOOL_ERR_INVALID_ARG;
    const kvp::LayerBufs L = p->layer(layer);
    v->kq = L.kq;
    v->vcodes = L.vcodes;
    v->vnorm = L.vnorm;
    v->kscale = L.kscale;
    v->ctx = p->ctx;
    v->ctx_padded = p->ctx_pad;
    v->bits = L.bits;
    v->compressed = p->compressed[layer];
    v->kscales = L.kscales;
    v->k_block = p->k_block;
    v->len = p->len[layer];
    v->group_bits = L.gbits;
    v->group_off = L.goff;
    v->mixed = L.mixed;
    return KVPOOL_OK;
}

namespace {

// Move one layer between the padded pool layout and a dense caller layout.
int copy_layer(const kvpool* p, int layer, bool to_pool, void* kq, void* vc, void* vn,
               void* ks, cudaStream_t st) {
    const kvp::LayerBufs L = p->layer(layer);
    const size_t rows = (size_t)p->kv_heads;
    const int T = to_pool ? p->ctx : p->len[layer];  // tokens moved
    const size_t kw = (size_t)T * p->head_dim, kp = (size_t)p->ctx_pad * p->head_dim;
    const size_t vb = (size_t)p->head_dim * L.bits / 8;
    // V codes travel in whole 32-token groups (the pool layout); a layer of
    // per-group widths moves each head's written groups back to back
    const size_t vw = (p->k_block && !to_pool) ? (size_t)p->group_offset(layer, (T + 31) / 32)
                                               : (size_t)((T + 31) / 32 * 32) * vb;
    const size_t vp = (size_t)L.vhead;
    const size_t nw = (size_t)T * 4, np_ = (size_t)p->ctx_pad * 4;
    cudaError_t e = cudaSuccess;
    if (kq && e == cudaSuccess)
        e = to_pool ? cudaMemcpy2DAsync(L.kq, kp, kq, kw, kw, rows, cudaMemcpyDefault, st)
                    : cudaMemcpy2DAsync(kq, kw, L.kq, kp, kw, rows, cudaMemcpyDefault, st);
    if (vc && e == cudaSuccess)
        e = to_pool ? cudaMemcpy2DAsync(L.vcodes, vp, vc, vw, vw, rows, cudaMemcpyDefault, st)
                    : cudaMemcpy2DAsync(vc, vw, L.vcodes, vp, vw, rows, cudaMemcpyDefault, st);
    if (vn && e == cudaSuccess)
        e = to_pool ? cudaMemcpy2DAsync(L.vnorm, np_, vn, nw, nw, rows, cudaMemcpyDefault, st)
                    : cudaMemcpy2DAsync(vn, nw, L.vnorm, np_, nw, rows, cudaMemcpyDefault, st);
    if (ks && e == cudaSuccess)
        e = to_pool ? cudaMemcpyAsync(L.kscale, ks, 4, cudaMemcpyDefault, st)
                    : cudaMemcpyAsync(ks, L.kscale, 4, cudaMemcpyDefault, st);
    return map_cuda(e);
}

}  // namespace

int kvpool_export_layer(const kvpool_t* p, int layer, void* kq, void* vcodes, void* vnorm,
                        void* kscale, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!p->compressed[layer]) return KVPOOL_ERR_STATE;
    return copy_layer(p, layer, false, kq, vcodes, vnorm, kscale, static_cast<cudaStream_t>(stream));
}

int kvpool_import_layer(kvpool_t* p, int layer, const void* kq, const void* vcodes,
                        const void* vnorm, const void* kscale, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (p->k_block) return KVPOOL_ERR_UNSUPPORTED;
    if (!kq || !vcodes || !vnorm || !kscale) return KVPOOL_ERR_INVALID_ARG;
    if (p->compressed[layer]) return KVPOOL_ERR_STATE;
    rc = copy_layer(p, layer, true, const_cast<void*>(kq), const_cast<void*>(vcodes),
                    const_cast<void*>(vnorm), const_cast<void*>(kscale),
                    static_cast<cudaStream_t>(stream));
    if (rc != KVPOOL_OK) return rc;
    rc = map_cuda(kvp::launch_norm_max(p->shape(), p->layer(layer), static_cast<cudaStream_t>(stream)));
    p->wrote(stream, layer);
    if (rc == KVPOOL_OK) {
        p->compressed[layer] = 1;
        p->len[layer] = p->ctx;
    }
    return rc;
}

int kvpool_import_layer_blocks(kvpool_t* p, int layer, const void* kq, const void* vcodes, const void* vnorm,
                               const void* kscales, const uint8_t* widths, int len, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!p->k_block) return KVPOOL_ERR_UNSUPPORTED;
    if (!kq || !vcodes || !vnorm || !kscales || len < 1 || len > p->ctx) return KVPOOL_ERR_INVALID_ARG;
    if (p->compressed[layer] || p->len[layer] != 0) return KVPOOL_ERR_STATE;
    const int ng = (len + 31) / 32;
    std::vector<uint8_t> w(ng);
    std::vector<uint32_t> off(ng);
    size_t head_bytes = 0;  // the layer's code bytes per KV head
    for (int g = 0; g < ng; ++g) {
        w[g] = widths ? widths[g] : (uint8_t)p->bits[layer];
        if (w[g] < 2 || w[g] > p->bits[layer]) return KVPOOL_ERR_INVALID_ARG;
        off[g] = (uint32_t)head_bytes;
        head_bytes += (size_t)p->head_dim * 4 * w[g];
    }
    const kvp::LayerBufs L = p->layer(layer);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t rows = (size_t)p->kv_heads, D = (size_t)p->head_dim, T = (size_t)len, Tp = (size_t)p->ctx_pad;
    const size_t nb = D / (size_t)p->k_block;  // block scales per token
    static const float kOne = 1.0f;  // the per-layer scale of a block-scaled layer
    cudaError_t e = cudaMemcpy2DAsync(L.kq, Tp * D, kq, T * D, T * D, rows, cudaMemcpyDefault, st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(L.vcodes, (size_t)L.vhead, vcodes, head_bytes, head_bytes, rows, cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaMemcpy2DAsync(L.vnorm, Tp * 4, vnorm, T * 4, T * 4, rows, cudaMemcpyDefault, st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(L.kscales, Tp * nb * 4, kscales, T * nb * 4, T * nb * 4, rows, cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.kscale, &kOne, sizeof(float), cudaMemcpyHostToDevice, st);
    // the group table (pageable host memory: staged before the calls return)
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.gbits, w.data(), (size_t)ng, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.goff, off.data(), (size_t)ng * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = kvp::launch_norm_max({p->kv_heads, p->head_dim, len, p->ctx_pad}, L, st);
    p->wrote(stream, layer);
    if (e != cudaSuccess) return map_cuda(e);
    p->gw[layer] = w;
    p->len[layer] = len;
    p->compressed[layer] = 1;
    return KVPOOL_OK;
}

int kvpool_export_kscales(const kvpool_t* p, int layer, float* kscales, void* stream) {
    int rc = check_layer(p, layer);
    if (rc) return rc;
    if (!kscales) return KVPOOL_ERR_INVALID_ARG;
    if (!p->k_block) return KVPOOL_ERR_UNSUPPORTED;
    if (!p->compressed[layer]) return KVPOOL_ERR_STATE;
    const kvp::LayerBufs L = p->layer(layer);
    const size_t per = (size_t)(p->head_dim / p->k_block) * 4;  // bytes per token
    const size_t T = (size_t)p->len[layer];
    return map_cuda(cudaMemcpy2DAsync(kscales, T * per, L.kscales, (size_t)p->ctx_pad * per,
                                      T * per, (size_t)p->kv_heads, cudaMemcpyDefault,
                                      static_cast<cudaStream_t>(stream)));
}

int kvpool_sensitivity(const void* Q, int agents, int q_heads, const kvpool_tail_t* recent, int kv_heads,
                       int head_dim, float softmax_scale, float* row_r, float* score, void* stream) {
    if (!Q || !recent || !row_r || !score || agents < 1 || kv_heads < 1 || q_heads < kv_heads ||
        q_heads % kv_heads || (head_dim != 64 && head_dim != 128))
        return KVPOOL_ERR_INVALID_ARG;
    if (recent->T_max < 0 || recent->T_max > 12288 ||
        (recent->T_max > 0 && (!recent->K || !recent->V || !recent->len)))
        return KVPOOL_ERR_INVALID_ARG;
    if (!(softmax_scale >= 0.0f) || isinf(softmax_scale)) return KVPOOL_ERR_INVALID_ARG;
    if (recent->T_max == 0) {  // no recent token: every row counts 0
        cudaError_t e = cudaMemsetAsync(score, 0, sizeof(float), static_cast<cudaStream_t>(stream));
        return map_cuda(e);
    }
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
    return map_cuda(kvp::launch_sensitivity(Q, agents, q_heads, kv_heads, head_dim, recent->K, recent->V,
                                            recent->len, recent->T_max, scale, row_r, score,
                                            static_cast<cudaStream_t>(stream)));
}

int kvpool_allocate_bits(int layers, const double* sens, const int64_t* cost, int64_t budget, uint8_t* bits) {
    if (layers < 1 || !sens || !cost || !bits || budget < 0) return KVPOOL_ERR_INVALID_ARG;
    int64_t g = 0;
    for (int l = 0; l < layers; ++l) {
        if (cost[l] < 1 || !(sens[l] >= 0.0) || std::isinf(sens[l])) return KVPOOL_ERR_INVALID_ARG;
        int64_t a = g, b = cost[l];
        while (b) {
            const int64_t t = a % b;
            a = b;
            b = t;
        }
        g = a;
    }
    // integer units: every cost is a multiple of g
    std::vector<int64_t> c(layers), rest(layers + 1, 0);
    for (int l = 0; l < layers; ++l) c[l] = cost[l] / g;
    for (int l = layers - 1; l >= 0; --l) rest[l] = rest[l + 1] + 2 * c[l];
    const int64_t B = budget / g;
    if (rest[0] > B) return KVPOOL_ERR_INVALID_ARG;  // even 2 bits everywhere do not fit
    const int64_t need = std::min<int64_t>(B, 4 * rest[0] / 2);  // more units than 4 bits everywhere never matter
    if ((int64_t)(layers + 1) * (need + 1) > (int64_t)1 << 26) return KVPOOL_ERR_UNSUPPORTED;
    const double D[3] = {kvp::lm_distortion(2), kvp::lm_distortion(3), kvp::lm_distortion(4)};
    // err/bytes/choice of layers l.. with u units left (u in [0, need])
    const size_t W = (size_t)need + 1;
    std::vector<double> err((size_t)(layers + 1) * W, 0.0);
    std::vector<int64_t> by((size_t)(layers + 1) * W, 0);
    std::vector<uint8_t> pick((size_t)layers * W, 0);
    for (int l = layers - 1; l >= 0; --l) {
        for (int64_t u = 0; u <= need; ++u) {
            bool have = false;
            double be = 0.0;
            int64_t bb = 0;
            uint8_t bbits = 0;
            for (int b = 2; b <= 4; ++b) {
                const int64_t cc = c[l] * b;
                if (cc + rest[l + 1] > u) continue;
                const double s2 = sens[l] * sens[l];
                const double e = D[b - 2] * s2 + err[(size_t)(l + 1) * W + (size_t)(u - cc)];
                const int64_t y = cc + by[(size_t)(l + 1) * W + (size_t)(u - cc)];
                if (!have || e < be || (e == be && y < bb)) {
                    have = true;
                    be = e;
                    bb = y;
                    bbits = (uint8_t)b;
                }
            }
            err[(size_t)l * W + u] = be;
            by[(size_t)l * W + u] = bb;
            pick[(size_t)l * W + u] = bbits;
        }
    }
    int64_t u = need;
    for (int l = 0; l < layers; ++l) {
        const uint8_t b = pick[(size_t)l * W + u];
        bits[l] = b;
        u -= c[l] * b;
    }
    return KVPOOL_OK;
}

const char* kvpool_strerror(int code) {
    switch (code) {
        case KVPOOL_OK: return "ok";
        case KVPOOL_ERR_INVALID_ARG: return "invalid argument";
        case KVPOOL_ERR_STATE: return "layer state: compress is write-once, attend/decompress need a compressed layer";
        case KVPOOL_ERR_CUDA: return "CUDA runtime error";
        case KVPOOL_ERR_OOM: return "device allocation failed";
        case KVPOOL_ERR_NONFINITE: return "non-finite K maximum or V norm";
        case KVPOOL_ERR_TIMEOUT: return "a bounded device wait expired";
        case KVPOOL_ERR_UNSUPPORTED: return "unsupported device or shape (needs sm_103)";
        default: return "unknown error";
    }
}

}  // extern "C"
