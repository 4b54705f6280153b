// kvpool_attend_noalloc: decode attention over a compressed layer that the
// caller holds, without allocating any device memory.
//
// Some callers cannot call cudaMalloc: engines that reserve all device memory
// at start-up and hand out slices themselves (a stray cudaMalloc fails or
// breaks their accounting), and latency-critical callers for which the
// implicit device-wide synchronisation of cudaMalloc would stall concurrent
// work. For them this entry point runs the same split-context attention as
// kvpool_attend, with the split partials kept in the fixed array below instead
// of in memory owned by a kvpool_t.
#include <math.h>

#include <mutex>

#include "kvpool_internal.cuh"

namespace {

// Split scratch of the attention: every GPU that loads the library holds
// these bytes until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_attend_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_attend_scratch, per device

// Device address of the scratch on the current device, looked up once per
// device. In host code `g_attend_scratch` names a host-side stand-in, so the
// address must come from cudaGetSymbolAddress with that device current.
int scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attend_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KVPOOL_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVPOOL_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int kvpool_attend_noalloc(const int8_t* kq, const uint8_t* vcodes, const float* vnorm,
                                     const float* kscale, const float* kscales, int kv_heads,
                                     int head_dim, int ctx, int bits, const void* Q, int agents, int q_heads,
                                     const kvpool_tail_t* tail, float* out, float softmax_scale,
                                     void* stream) {
    if (!kq || !vcodes || !vnorm || !kscale || !Q || !out) return KVPOOL_ERR_INVALID_ARG;
    if (!aligned(kq, 16) || !aligned(vcodes, 16) || !aligned(vnorm, 4) || !aligned(kscale, 4) ||
        !aligned(Q, 16) || !aligned(out, 16) || !aligned(kscales, 4))
        return KVPOOL_ERR_INVALID_ARG;
    if ((head_dim != 64 && head_dim != 128) || bits < 2 || bits > 4 || kv_heads < 1 || ctx < 1 ||
        agents < 1 || q_heads < kv_heads || q_heads % kv_heads)
        return KVPOOL_ERR_INVALID_ARG;
    if (!(softmax_scale >= 0.0f) || isinf(softmax_scale)) return KVPOOL_ERR_INVALID_ARG;
    if (tail && (tail->T_max < 0 || (tail->T_max > 0 && (!tail->K || !tail->V || !tail->len))))
        return KVPOOL_ERR_INVALID_ARG;
    const int group = q_heads / kv_heads;
    const long long rows = (long long)agents * group;
    if ((long long)kv_heads * ctx > (1LL << 31) / 128 || rows > 4096) return KVPOOL_ERR_INVALID_ARG;

    // split count as kvpool_create picks it, then shrunk to fit the scratch
    const size_t per_split = (size_t)kv_heads * rows * (head_dim + 2) * sizeof(float) + 512;
    const long long fit = (long long)(kNoallocScratchBytes / per_split);
    if (fit < 1) return KVPOOL_ERR_INVALID_ARG;  // kv_heads*rows*(head_dim+2)*4 B exceeds 8 MiB

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVPOOL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVPOOL_ERR_UNSUPPORTED;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVPOOL_ERR_CUDA;
    if (major * 10 + minor != 103) return KVPOOL_ERR_UNSUPPORTED;
    void* base = nullptr;
    int rc = scratch_address(dev, &base);
    if (rc != KVPOOL_OK) return rc;

    const int ntile = (ctx + 31) / 32;
    long long nsplit = (2LL * sms + kv_heads - 1) / kv_heads;
    if (nsplit > ntile) nsplit = ntile;
    if (nsplit > fit) nsplit = fit;
    if (nsplit < 1) nsplit = 1;

    // carve: acc f32 [Hk][nsplit][rows][D], then ml f32 [Hk][nsplit][rows][2]
    const size_t acc_bytes = (size_t)kv_heads * nsplit * rows * head_dim * sizeof(float);
    const size_t ml_off = (acc_bytes + 255) & ~size_t(255);
    kvp::AttendScratch scr;
    scr.acc = static_cast<float*>(base);
    scr.ml = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + ml_off);
    scr.nsplit = (int)nsplit;
    scr.max_rows = (int)rows;

    kvp::Shape shape{kv_heads, head_dim, ctx, (ctx + kvp::kTokenPad - 1) / kvp::kTokenPad * kvp::kTokenPad};
    kvp::LayerBufs layer{const_cast<int8_t*>(kq), const_cast<uint8_t*>(vcodes),
                         const_cast<float*>(vnorm), const_cast<float*>(kscale), nullptr, bits,
                         nullptr};
    layer.kscales = const_cast<float*>(kscales);  // block-scaled K: one scale per 32 elements
    kvp::AttendArgs a{};
    a.Q = Q;
    a.agents = agents;
    a.q_heads = q_heads;
    a.group = group;
    a.rows = (int)rows;
    const bool has_tail = tail && tail->T_max > 0;
    a.tailK = has_tail ? tail->K : nullptr;
    a.tailV = has_tail ? tail->V : nullptr;
    a.tail_len = has_tail ? tail->len : nullptr;
    a.tail_max = has_tail ? tail->T_max : 0;
    a.out = out;
    a.t0 = 0;
    a.t1 = ctx;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    const cudaError_t e =
        kvp::launch_attend_split(shape, layer, a, scr, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVPOOL_OK : KVPOOL_ERR_CUDA;
}
