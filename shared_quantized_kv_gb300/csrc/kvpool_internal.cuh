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

// Tensor-core operand tables of the three widths under one scale lam (layers
// whose groups have different widths: the attention kernel divides its output
// by one lam), c16[b - 2][k] = fp16 bits of lam * c_b[k].
struct MixBook {
    uint16_t c16[3][16];
    float lam;
};
const MixBook& mixbook();

// Compress scratch of a layer: kKmaxParts words. Words [0, kKmaxInv) take the
// max|K| kernel's partial maxima (bf16 bits of |k|, one per CTA); kKmaxInv
// the float bits of 1/s; kKmaxCount the kernel's arrival counter (0 between
// launches; the pool is created zeroed).
constexpr int kKmaxParts = 512;
constexpr int kKmaxInv = kKmaxParts - 2;
constexpr int kKmaxCount = kKmaxParts - 1;

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
    uint32_t* kpart;          // [kKmaxParts] compress scratch (see kKmaxParts)
    float* kscales;           // block-scaled K: [Hk][ctx_pad][D/32], one scale per 32 elements; else null
    // Per-group V widths (block-scaled pools, whose layers grow by appends):
    // gbits[g] the width of 32-token group g (0: not written), goff[g] the
    // byte offset of its codes within a KV head (null for per-tensor pools);
    // KV head h's codes start at h * vhead (ctx_pad * D * bits / 8, bits the
    // width fixed at create, the largest a group may take). mixed = 1 when the
    // written groups do not all have width `bits`: attend and decompress then
    // take the per-group path.
    uint8_t* gbits;
    uint32_t* goff;
    long long vhead;
    int mixed;
};

struct Shape {
    int kv_heads, head_dim, ctx, ctx_pad;
};

// ---- encode (write-once compress)
// One layer of a multi-layer encode launch (kernel parameter, by value).
struct EncLayer {
    const uint16_t* K;  // bf16 [Hk][ctx][D] inputs
    const uint16_t* V;
    int8_t* kq;
    uint8_t* vcodes;
    float* vnorm;
    float* kscale;
    uint32_t* maxima;   // {bf16 bits of max|K|, float bits of the largest V norm}
    uint32_t* kpart;    // kKmaxParts words of compress scratch
    float* kscales;     // block-scaled K, else null
    // V codes of token group g of the encode (g = 0 at its first token) start
    // at vcodes + h * vhead + voff + g * D * 4 * bits; block-scaled pools also
    // record each group's width and offset in gbits / goff (else null)
    long long vhead, voff;
    uint8_t* gbits;
    uint32_t* goff;
};
// Most layers per launch of the multi-layer kernels.
constexpr int kEncBatch = 32;
// A launch's layer table; one-layer calls pass the one-entry form (a smaller
// parameter block, and the encode kernel reduces the partial maxima itself)
template <int NB>
struct EncBatchT {
    int n;
    EncLayer L[NB];
};
using EncBatch = EncBatchT<kEncBatch>;

// s.ctx is the token count of K and V; t_base the pool token they start at
// (non-zero only for appends to block-scaled layers, a multiple of 32) and
// voff the byte offset of its group within a KV head's codes; L.bits is the
// width the tokens are coded at.
cudaError_t launch_encode(const Shape& s, const LayerBufs& L, const void* K, const void* V,
                          int* status, int sm_count, int t_base, long long voff, cudaStream_t st);
// n layers (all of one pool, so one k-scaling mode) in a few launches per
// kEncBatch of them: one max|K| kernel over all, then one encode kernel per V
// width. t_base != 0 or voff != 0 only with n = 1.
cudaError_t launch_encode_layers(const Shape& s, const LayerBufs* L, const void* const* K, const void* const* V,
                                 int n, int* status, int sm_count, int t_base, long long voff,
                                 cudaStream_t st);

// ---- decompress
// One layer of a multi-layer decompress launch (kernel parameter, by value).
struct DecLayer {
    const int8_t* kq;
    const float* kscale;
    const float* kscales;  // block-scaled K, else null
    const uint8_t* vcodes;
    const float* vnorm;
    const uint8_t* gbits;  // per-group widths (kernels of mixed layers), else unused
    const uint32_t* goff;
    long long vhead;       // bytes per KV head of the codes
    uint4* Kout;           // bf16 [Hk][len][D], or null
    uint4* Vout;
    int len;               // tokens the layer holds
};
struct DecBatch {
    int n;
    DecLayer L[kEncBatch];
};

cudaError_t launch_decompress(const Shape& s, const LayerBufs& L, void* K_out, void* V_out,
                              cudaStream_t st);
// n layers, one launch per V width and kEncBatch layers; len[i] tokens of
// layer i; K_out or V_out may be null (that half for none of the layers).
cudaError_t launch_decompress_layers(const Shape& s, const LayerBufs* L, const int* len, void* const* K_out,
                                     void* const* V_out, int n, cudaStream_t st);

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
    // context slice [t0, t1) of the layer's tokens (the whole layer: 0, len)
    int t0, t1;
    // partial mode: the slice's per-row (m, l) and rotated accumulator instead
    // of the output (see kvpool_attend_partial); null otherwise
    float* part_ml;      // [Hk][rows][2]
    float* part_acc;     // [Hk][rows][D]
    // workspace mode of the tensor-core kernel (ws_ctas > 0, partial mode
    // only): the context in slices of one CTA each, at most ws_ctas CTAs;
    // part_ml / part_acc then hold [nslice][Hk][rows] and *ws_nslice gets
    // nslice
    int ws_ctas;
    int ws_nslice_max;  // the workspace holds at most this many slices
    int* ws_nslice;
    // workspace mode with tails: the slices' CTAs compute the agents' tails
    // (accumulators into `out`, (m, l) here, [Hk][rows][2]) and the merge
    // joins them; null otherwise (the merge computes the tails itself)
    float* ws_tail_ml;
};

// Log-sum-exp merge of `parts` partial results laid out [parts][Hk][rows]
// (see kvpool_merge_partials), one inverse FWHT per row, the agents' tails,
// and the final normalisation into a.out. sm_count > 0 (the workspace path)
// shapes the grid for that many SMs: CTAs of 16 warps where that fits a grid
// of more than one wave into one, and for a one-wave grid over 1 MiB of
// partial states a shared-memory reservation that spreads the CTAs one per
// SM (see attend.cu).
cudaError_t launch_merge_partials(int parts, const float* part_ml, const float* part_acc, int kv_heads,
                                  int head_dim, const AttendArgs& a, cudaStream_t st, int sm_count = 0);

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
