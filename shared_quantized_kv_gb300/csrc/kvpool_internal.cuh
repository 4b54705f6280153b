// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (the encode entry point is fetched at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvpool.h"

namespace kvp {

// The token axis of every pool layer is padded to a multiple of this.
constexpr int kTokenPad = 128;

// Device status bits (kernels OR them in; the host maps them to error codes).
enum : int { kStNonfinite = 1, kStTimeout = 2 };

// Float32 Lloyd-Max table of one V bit width, passed to kernels by value.
struct Codebook {
    float c[16];  // centroids, ascending (levels used)
    float m[16];  // midpoints (levels - 1 used)
    int levels;
    int bits;
    // Tensor-core operand table: fp16 bits of lam * c[k]. The scale lam in
    // [1, 2) is chosen so that every lam * c[k] lies as close as possible to
    // an fp16 value (the attention kernel divides its output by lam).
    uint16_t c16[16];
    float lam;
};

// Host: the library's own table for `bits` in {2,3,4} (derived once).
const Codebook& codebook(int bits);

// Most CTAs of the max|K| kernel that runs ahead of the encode kernel: one
// partial maximum (bf16 bits of |k|) per CTA, kept per layer.
constexpr int kKmaxParts = 512;

// Device buffers of one layer.
struct LayerBufs {
    int8_t* kq;        // [Hk][ctx_pad][D]
    uint8_t* vcodes;   // [Hk][ctx_pad/32][D][4*bits]: per 32-token group, one code sequence per coordinate
    float* vnorm;      // [Hk][ctx_pad]
    float* kscale;     // 1 float
    uint32_t* kabsmax; // 1 word: bf16 bits of max|K| (scratch of the encode)
    int bits;
    uint32_t* vnmax;   // 1 word right after kabsmax: float bits of the largest V norm
    const CUtensorMap* kmap;  // TMA map of kq as rows of D bytes (128 / 64-byte swizzle), or null
    uint32_t* kpart;          // [kKmaxParts] partial maxima of max|K| (compress scratch)
    float* kscales;           // block-scaled K: [Hk][ctx_pad][D/32], one scale per 32 elements; else null
};

struct Shape {
    int kv_heads, head_dim, ctx, ctx_pad;
};

// ---- encode (write-once compress of one layer)
// s.ctx is the token count of K and V; t_base the pool token they start at
// (non-zero only for appends to block-scaled layers, a multiple of 32).
cudaError_t launch_encode(const Shape& s, const LayerBufs& L, const void* K, const void* V,
                          int* status, int sm_count, int t_base, cudaStream_t st);

// ---- decompress
cudaError_t launch_decompress(const Shape& s, const LayerBufs& L, void* K_out, void* V_out,
                              cudaStream_t st);

// ---- attend
struct AttendArgs {
    const void* Q;       // bf16 [A][Hq][D]
    int agents, q_heads, group, rows;  // rows = agents * group
    const void* tailK;   // bf16 [A][Hk][T_max][D] or null
    const void* tailV;
    const int32_t* tail_len;
    int tail_max;
    float* out;          // f32 [A][Hq][D]
    float scale_log2;    // softmax scale * log2(e)
    int early;           // 1: the launch right before this one on its stream did not write the layer
};

struct AttendScratch {
    float* acc;   // [Hk][nsplit][max_rows][D]
    float* ml;    // [Hk][nsplit][max_rows][2]
    int nsplit;
    int max_rows;
};

// CUDA-core split-context attention with partials in `scr` (any device memory).
cudaError_t launch_attend_split(const Shape& s, const LayerBufs& L, const AttendArgs& a,
                                const AttendScratch& scr, cudaStream_t st);

// Tensor-core cluster attention (no scratch memory).
cudaError_t launch_attend_tc(const Shape& s, const LayerBufs& L, const AttendArgs& a, int* status,
                             int sm_count, cudaStream_t st);

// Local attention-error estimate of one layer (see sensitivity.cu): r per
// (agent, query head) row into row_r, their mean into *score.
cudaError_t launch_sensitivity(const void* Q, int agents, int q_heads, int kv_heads, int head_dim,
                               const void* tK, const void* tV, const int32_t* tlen, int T_max, float scale,
                               float* row_r, float* score, cudaStream_t st);

// Mean squared error of the library's Lloyd-Max quantiser for N(0,1).
double lm_distortion(int bits);

// Largest V norm of a layer (for layers loaded with kvpool_import_layer).
cudaError_t launch_norm_max(const Shape& s, const LayerBufs& L, cudaStream_t st);

}  // namespace kvp
