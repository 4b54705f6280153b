/*
 * kvpool -- a shared, asymmetrically quantized KV-cache pool for multi-agent
 * decode on one GB300 GPU (sm_103a).
 *
 * The method (PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool for
 * Multi-Agent LLM Inference, gist.science summary, section 2): the full KV
 * state of a shared document is computed once, compressed, and stored as ONE
 * write-once / read-many object that every agent reads (section 2.A,
 * SharedKVPool / PooledAgent). Keys are quantised per tensor to int8; values
 * are rotated per head-vector by the fast Walsh-Hadamard transform and mapped
 * to Lloyd-Max centroids for N(0,1), 3 bits by default (section 2.B). The
 * CoMixKV article (zicq.com, "CoMixKV ... Qwen3显存降低32.08%") gives 2 to 4
 * bits per layer and keeps the most recent states at native precision; here
 * each layer has its own V bit width in {2, 3, 4} and every agent may bring a
 * private bf16 recent-token tail to attention.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Return value: KVPOOL_OK (0) or a negative KVPOOL_ERR_* code. Argument and
 *    state errors are reported synchronously and enqueue nothing.
 *  - Errors found by a kernel (a non-finite K maximum or V norm, an expired
 *    bounded wait) are recorded in a device status word. They are sticky and
 *    are returned (and cleared) by kvpool_status().
 *  - All device work is asynchronous on the caller's stream (`stream` is a
 *    cudaStream_t passed as void*; NULL is the legacy default stream). Device
 *    pointers passed in must stay valid until that work completes; the library
 *    keeps no caller pointer after a call returns.
 *  - The pool owns all of its device memory, allocated once by
 *    kvpool_create(); compress, attend and decompress allocate nothing.
 *  - bf16 tensors are raw IEEE bfloat16 bit patterns, row-major, contiguous,
 *    16-byte aligned. head_dim is 64 or 128.
 *  - After a layer is compressed its pool bytes are read-only, so concurrent
 *    kvpool_attend / kvpool_decompress calls on different streams are safe.
 *    A single pool must not be compressed from two host threads at once.
 */
#ifndef KVPOOL_H
#define KVPOOL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    KVPOOL_OK = 0,
    KVPOOL_ERR_INVALID_ARG = -1, /* null pointer, bad size, layer out of range  */
    KVPOOL_ERR_STATE = -2,       /* write-once violated / layer not compressed   */
    KVPOOL_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed         */
    KVPOOL_ERR_OOM = -4,         /* device allocation failed in kvpool_create    */
    KVPOOL_ERR_NONFINITE = -5,   /* K maximum or a V norm was Inf/NaN (device)   */
    KVPOOL_ERR_TIMEOUT = -6,     /* a bounded device wait expired (device)       */
    KVPOOL_ERR_UNSUPPORTED = -7  /* no sm_103a device, or a shape not supported  */
};

typedef struct kvpool kvpool_t;

/* A private recent-token tail per agent, kept at bf16 (CoMixKV article,
 * incremental quantisation: recent states stay at native precision). Agent a
 * attends over the pool followed by its first len[a] tail tokens, in one
 * softmax. */
typedef struct {
    const void* K;      /* bf16 [agents][kv_heads][T_max][head_dim], device    */
    const void* V;      /* bf16 [agents][kv_heads][T_max][head_dim], device    */
    const int32_t* len; /* int32 [agents], device, each in [0, T_max]          */
    int T_max;          /* capacity of the tail buffers, >= 0                  */
} kvpool_tail_t;

/* Device-side view of one compressed layer (for inspection and tests). The
 * token axis is padded to `ctx_padded`; padding is zero and never read as a
 * token. Pointers stay owned by the pool.
 *
 * V code layout: per KV head, the tokens form groups of 32; a group holds, for
 * each rotated coordinate i in order, the codes of its 32 tokens in token order
 * packed little-endian (8 codes in 3 bytes at 3 bits, 4 per byte at 2 bits, 2
 * per byte low nibble first at 4 bits): 4*bits bytes per coordinate,
 * head_dim*4*bits bytes per group. Token slots past ctx in the last group hold
 * code 0. (PolyKV summary, section 2.B, fixes the packing; the grouping is this
 * library's, so that one thread reading one coordinate of many tokens finds
 * them in consecutive bytes.) */
typedef struct {
    const int8_t* kq;      /* int8 [kv_heads][ctx_padded][head_dim]            */
    const uint8_t* vcodes; /* uint8 [kv_heads][ctx_padded/32][head_dim][4*bits] */
    const float* vnorm;    /* float [kv_heads][ctx_padded]                     */
    const float* kscale;   /* one float: the layer's K scale s = max|K| / 127  */
    int ctx;
    int ctx_padded;
    int bits;
    int compressed;        /* 1 once kvpool_compress succeeded for the layer   */
    const float* kscales;  /* block-scaled pools (kvpool_create_ex, k_block 32):
                              float [kv_heads][ctx_padded][head_dim/32], one
                              scale per 32 elements (*kscale is then 1); NULL
                              for per-tensor pools                            */
    int k_block;           /* 0 (per-tensor scale) or 32                       */
    int len;               /* tokens the layer holds: ctx once compressed or
                              imported; appends (kvpool_append) grow it         */
    const uint8_t* group_bits; /* block-scaled pools: uint8 [ctx_padded/32],
                              device, the V width of each 32-token group
                              (entries from ceil(len/32) on are not
                              meaningful); NULL for per-tensor pools         */
    const uint32_t* group_off; /* block-scaled pools: uint32 [ctx_padded/32],
                              device, the byte offset of each written group
                              within its KV head's codes; NULL otherwise      */
    int mixed;             /* 1 if the written groups do not all have width
                              `bits` (kvpool_append_bits); the layout is then
                              the per-group one of kvpool_append_bits         */
} kvpool_layer_view_t;

/* Create a pool for `layers` layers of a shared context of `ctx` tokens with
 * `kv_heads` KV heads of size `head_dim` (64 or 128). bits_per_layer: host
 * array [layers] of V bit widths, each 2, 3 or 4 (NULL: 3 for every layer).
 * max_rows: the most query rows that may share one KV head in kvpool_attend
 * (agents x GQA group), 1..1024 (0: 512).
 * Allocates all device memory on the current device. Source: PolyKV summary,
 * section 2.A (one shared object, O(1) in the number of agents). */
int kvpool_create(kvpool_t** out, int layers, int kv_heads, int head_dim, int ctx,
                  const uint8_t* bits_per_layer, int max_rows);

/* kvpool_create with a choice of K scaling. k_block = 0 is kvpool_create (one
 * scale per layer's K tensor). k_block = 32 gives every block of 32
 * consecutive elements of a K head-vector its own float32 scale: s_b =
 * max|k| / 127 over the block (float32 division; 1 for an all-zero block),
 * q = clamp(round-half-even(k / s_b), -127, 127) with a float32 division,
 * K_hat = q * s_b. This is the "q8_0" reading of the PolyKV summary's section
 * 2.B (which names both a per-tensor scale and q8_0); the scales are float32,
 * not q8_0's fp16, because a bf16 K can exceed the fp16 range. The pool then
 * holds head_dim/32 scales per token and head (kvpool_layer_view_t.kscales).
 * Attention over such a pool runs on the tensor cores like that of a
 * per-tensor pool and needs no scratch: K^ is formed from each block's
 * quantised values and scale as a pair of fp16 operands (about 22 significant
 * bits), the token's power-of-two range factor applied to its logit exactly.
 * kvpool_export_layer exports such a layer with *kscale = 1 and
 * kvpool_export_kscales copies its block scales; such layers are loaded with
 * kvpool_import_layer_blocks (kvpool_import_layer returns
 * KVPOOL_ERR_UNSUPPORTED for these pools). Other k_block values:
 * KVPOOL_ERR_INVALID_ARG. */
int kvpool_create_ex(kvpool_t** out, int layers, int kv_heads, int head_dim, int ctx,
                     const uint8_t* bits_per_layer, int max_rows, int k_block);

/* Copy the block scales of one compressed layer of a block-scaled pool to
 * `kscales` (host or device), float [kv_heads][ctx][head_dim/32], on
 * `stream`. KVPOOL_ERR_UNSUPPORTED for per-tensor pools, KVPOOL_ERR_STATE if
 * the layer is not compressed. */
int kvpool_export_kscales(const kvpool_t* pool, int layer, float* kscales, void* stream);

/* Incremental pool append (CoMixKV article: aged recent-state blocks are
 * quantised into new pool blocks; earlier blocks are never rewritten) for
 * block-scaled pools: encode n new tokens K, V bf16 [kv_heads][n][head_dim]
 * (device, 16-byte aligned) as tokens [len, len + n) of the layer, exactly as
 * kvpool_compress encodes each token (with block-scaled K every stored byte
 * depends on its own token only, so the layer equals the encode of all its
 * tokens at once). A layer starts empty (len 0, also after
 * kvpool_reset_layer); kvpool_compress on an empty block-scaled layer is the
 * append of all ctx tokens. Attend, decompress and export read tokens
 * [0, len) (decompress writes [kv_heads][len][head_dim]). Before an append
 * len must be a multiple of 32 (an append of a length that is not a multiple
 * of 32 closes the layer: KVPOOL_ERR_STATE), and len + n <= ctx
 * (KVPOOL_ERR_INVALID_ARG). Per-tensor pools: KVPOOL_ERR_UNSUPPORTED (one K
 * scale cannot take new tokens without re-encoding the old ones). */
int kvpool_append(kvpool_t* pool, int layer, const void* K, const void* V, int n, void* stream);

/* kvpool_append with the V codes of the n new tokens at width `bits` (2, 3
 * or 4, at most the layer's width fixed at create, which sets the layer's
 * reserved size). CoMixKV article, incremental quantisation strategy: a
 * width newly chosen by the allocator (kvpool_allocate_bits) applies only to
 * blocks quantised afterwards; earlier blocks keep their width and bytes.
 * The unit is the 32-token group: every group has one width, and per KV head
 * the groups' codes follow each other in token order with no gap (group g at
 * byte sum_{g' < g} head_dim * 4 * b_{g'} of the head's codes, which start at
 * h * ctx_padded * head_dim * bits_create / 8), each group in the uniform
 * layout of kvpool_layer_view_t at its own width. Attend, partial attend and
 * decompress read every group at its width; kvpool_export_layer writes each
 * head's groups back to back (kv_heads * sum_g head_dim * 4 * b_g bytes; see
 * kvpool_layer_widths). Errors as kvpool_append, and KVPOOL_ERR_INVALID_ARG
 * for a width outside [2, create width]. */
int kvpool_append_bits(kvpool_t* pool, int layer, const void* K, const void* V, int n, int bits,
                       void* stream);

/* Widths of the 32-token groups layer `layer` holds: writes the width of
 * group g (tokens [32 g, 32 g + 32)) to widths[g] for g < max_groups (host
 * array; may be NULL when max_groups is 0) and returns the number of groups,
 * ceil(kvpool_layer_len / 32), or a negative error code. Per-tensor pools and
 * layers filled by kvpool_compress report the layer's width for every group. */
int kvpool_layer_widths(const kvpool_t* pool, int layer, uint8_t* widths, int max_groups);

/* Tokens layer `layer` holds (see kvpool_append), or a negative error code. */
int kvpool_layer_len(const kvpool_t* pool, int layer);

/* Local attention-error estimate of one layer from recently observed queries,
 * keys and values (CoMixKV article, online sensitivity estimation: no
 * calibration set, no trial quantisation). The article prints no formula; the
 * one used: a V head-vector coded at b bits has E|v - v_hat|^2 = D_b |v|^2
 * (D_b the Lloyd-Max distortion of N(0,1)), so a query row's relative output
 * error is sqrt(D_b) * r with r = sqrt(sum_t p_t^2 |v_t|^2) / |sum_t p_t v_t|
 * over the agent's recent tokens (p the softmax of the row's logits, scaled
 * by softmax_scale, 0 meaning 1/sqrt(head_dim)). Writes r of every (agent,
 * query head) row to row_r (device float [agents * q_heads]) and their mean,
 * the layer's sensitivity s, to *score (device float); an agent with no
 * recent token contributes 0. Q: bf16 [agents][q_heads][head_dim]; recent:
 * the agents' recent tokens in the kvpool_tail_t layout (T_max <= 12288).
 * Asynchronous on `stream`; needs no pool. */
int kvpool_sensitivity(const void* Q, int agents, int q_heads, const kvpool_tail_t* recent, int kv_heads,
                       int head_dim, float softmax_scale, float* row_r, float* score, void* stream);

/* Joint V bit widths (CoMixKV article: the controller combines sensitivity,
 * capacity and byte-level cost and picks every layer's width within one
 * budget). Host only. Chooses bits[l] in {2, 3, 4} minimising
 * sum_l D_{bits[l]} * sens[l]^2 subject to sum_l cost[l] * bits[l] <= budget,
 * exactly (dynamic programming over the costs in units of their greatest
 * common divisor); among allocations of equal error the one of fewer bytes,
 * then the one with the smaller width at the first layer where they differ.
 * cost[l] >= 1: the layer's V bytes per bit of width (kv_heads * tokens *
 * head_dim / 8 for a pool layer). KVPOOL_ERR_INVALID_ARG when even 2 bits
 * everywhere exceed the budget, KVPOOL_ERR_UNSUPPORTED when the table would
 * exceed 2^26 entries. The widths apply to layers created later
 * (kvpool_create) or, in block-scaled pools, to the blocks appended later
 * (kvpool_append_bits, up to each layer's create width). */
int kvpool_allocate_bits(int layers, const double* sens, const int64_t* cost, int64_t budget, uint8_t* bits);

/* Free all device memory of the pool. Waits for the device first. NULL is a
 * no-op. */
void kvpool_destroy(kvpool_t* pool);

/* Write-once encode of one layer. K, V: bf16 [kv_heads][ctx][head_dim], device.
 * K: s = max|K| / 127 (float32; s = 1 when K is all zero), q = clamp(round-
 * half-even(k / s), -127, 127). V, per head-vector v: n = |v| (float32,
 * pairwise tree), u = H v (unnormalised FWHT, stages 1, 2, 4, ...), code_i =
 * #{ j : u_i > fl(m_j * n) } for the float32 Lloyd-Max midpoints m_j, codes
 * bit-packed little-endian. Source: PolyKV summary, section 2.B. Returns
 * KVPOOL_ERR_STATE if the layer was already compressed (see
 * kvpool_reset_layer). A non-finite K or V norm is reported by kvpool_status
 * as KVPOOL_ERR_NONFINITE. */
int kvpool_compress(kvpool_t* pool, int layer, const void* K, const void* V, void* stream);

/* Write-once encode of n layers in one call: the same pool bytes as
 * kvpool_compress(pool, layers[i], K[i], V[i], stream) for every i, with one
 * max|K| kernel for all of them and one encode kernel per V width among them
 * (per 32 layers), so that a whole shared context is written with a few
 * launches (PolyKV summary, section 2.A: the pool is built once for every
 * layer of the shared context). layers, K, V: host arrays [n]; K[i], V[i]:
 * device pointers, as for kvpool_compress. KVPOOL_ERR_INVALID_ARG for n < 1,
 * a null or misaligned pointer, a layer out of range or named twice;
 * KVPOOL_ERR_STATE if any of the layers is already compressed. On either
 * error nothing is launched and no layer changes state. */
int kvpool_compress_layers(kvpool_t* pool, int n, const int* layers, const void* const* K, const void* const* V,
                           void* stream);

/* Decode attention of `agents` agents over one compressed layer.
 * Q: bf16 [agents][q_heads][head_dim], device; q_heads a multiple of
 * kv_heads; query head h reads KV head h / (q_heads / kv_heads).
 * tail: NULL for none. out: float32 [agents][q_heads][head_dim], device.
 * softmax_scale: 0 means 1/sqrt(head_dim).
 * Every agent's rows attend over the dequantised pool (K = q*s, V = n*H c/d)
 * followed by the agent's tail tokens, in one softmax. agents * group must not
 * exceed the pool's max_rows. Source: PolyKV summary, section 2.A (every agent
 * reads the same pool) and 2.B (dequantisation: centroid lookup + inverse
 * FWHT). */
int kvpool_attend(kvpool_t* pool, int layer, const void* Q, int agents, int q_heads,
                  const kvpool_tail_t* tail, float* out, float softmax_scale, void* stream);

/* kvpool_attend through a caller-provided workspace (device memory of at
 * least kvpool_attend_ws_bytes(pool, agents, q_heads) bytes, 16-byte
 * aligned; its contents need no initialisation and are scratch afterwards):
 * the context is cut into more slices than kvpool_attend's clusters can hold
 * (one CTA each, enough to fill every SM once), their partial states (the
 * kvpool_attend_partial quantities) go to the workspace, the slices' CTAs
 * also compute the agents' tails (each slice a share of the agents), and a
 * second kernel merges all of it as kvpool_merge_partials does. Same
 * arguments, result and errors as kvpool_attend, plus
 * KVPOOL_ERR_INVALID_ARG for a missing, misaligned or short workspace and
 * KVPOOL_ERR_UNSUPPORTED when the (KV head, row group) pairs alone exceed
 * one wave of CTAs. Calls that overlap on the GPU must not share a
 * workspace. Source: the PolyKV summary's attention over the shared pool
 * (section 2.A), split over the context with the log-sum-exp merge of
 * softmax partial sums. */
int kvpool_attend_ws(kvpool_t* pool, int layer, const void* Q, int agents, int q_heads,
                     const kvpool_tail_t* tail, float* out, float softmax_scale, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Bytes of workspace kvpool_attend_ws needs for `agents` agents with q_heads
 * query heads over any layer of the pool (0 for invalid arguments). */
size_t kvpool_attend_ws_bytes(const kvpool_t* pool, int agents, int q_heads);

/* Context split (one pool's context over several calls, ranks or GPUs):
 * the attention state of every (agent, query head) row over the pool tokens
 * [t_begin, t_end) of a compressed layer, instead of the finished output.
 * For row r = a * G + j of KV head g (G = q_heads / kv_heads, query head
 * g * G + j of agent a) it writes part_ml[g][r] = (m, l) and part_acc[g][r][:]
 * = acc with, over the slice's tokens t and logits x_t = softmax_scale *
 * log2(e) * <q, K_t> (log2 units): l = sum_t 2^(x_t - m) and acc =
 * sum_t 2^(x_t - m) n_t c[codes_t] in the rotated domain (the slice's
 * output is H acc / (head_dim * l), H the Sylvester Hadamard matrix); m is
 * a reference within a few units of the slice's largest logit. part_ml:
 * float [kv_heads][agents * G][2], 8-byte aligned; part_acc: float
 * [kv_heads][agents * G][head_dim], 16-byte aligned; device. t_begin a
 * multiple of 128, 0 <= t_begin < t_end <= kvpool_layer_len. No tail:
 * the agents' private tails join in kvpool_merge_partials. Per-tensor and
 * block-scaled pools. Source: the PolyKV
 * summary's attention over the shared pool (section 2.A), split over the
 * context; the merge below is the log-sum-exp combination of softmax
 * partial sums. */
int kvpool_attend_partial(kvpool_t* pool, int layer, const void* Q, int agents, int q_heads, int t_begin,
                          int t_end, float* part_ml, float* part_acc, float softmax_scale, void* stream);

/* Merge `parts` results of kvpool_attend_partial (slices of one context, in
 * any order), each agent's private bf16 tail (NULL for none) and the final
 * normalisation into out (float [agents][q_heads][head_dim], device):
 * o = H (sum_s 2^(m_s - M) acc_s) / head_dim joined with the tail tokens in
 * one softmax, divided by the total weight. part_ml: float [parts][kv_heads]
 * [agents * G][2]; part_acc: float [parts][kv_heads][agents * G][head_dim]
 * (the parts' buffers back to back), device. A part whose l is not
 * positive (an empty slice) counts for nothing; its m and accumulator are
 * not used. Q, tail, softmax_scale as in kvpool_attend. Needs no pool. */
int kvpool_merge_partials(int parts, const float* part_ml, const float* part_acc, int kv_heads, int head_dim,
                          const void* Q, int agents, int q_heads, const kvpool_tail_t* tail, float* out,
                          float softmax_scale, void* stream);

/* Materialise one layer as bf16: K_out = bf16(q*s), V_out_i = bf16(fl(z_i*n)
 * * (1/d)) with z = FWHT(c[codes]) in float32. K_out, V_out: bf16
 * [kv_heads][len][head_dim], device (len = kvpool_layer_len: ctx unless the
 * layer was built by appends). This is the per-agent decompression of
 * the PolyKV summary, section 2.A (each agent injects the decompressed KV into
 * its own cache). */
int kvpool_decompress(kvpool_t* pool, int layer, void* K_out, void* V_out, void* stream);

/* kvpool_decompress of n layers in one launch per V width (per 32 layers):
 * layer layers[i] into K_out[i], V_out[i] (bf16 [kv_heads][len][head_dim],
 * device). layers, K_out, V_out: host arrays [n]; K_out or V_out may be NULL
 * (that half for none of the layers, not both), and then every entry of the
 * other must be a device pointer. KVPOOL_ERR_INVALID_ARG for n < 1, a layer
 * out of range, a null or misaligned output; KVPOOL_ERR_STATE if a layer is
 * not compressed (nothing is launched). */
int kvpool_decompress_layers(kvpool_t* pool, int n, const int* layers, void* const* K_out, void* const* V_out,
                             void* stream);

/* Compressed bytes held for the shared context: per layer, int8 K, packed V,
 * float32 norms and the float32 K scale (padding excluded). Independent of
 * the number of agents (PolyKV summary, section 4: the pool is O(1) in agents). */
size_t kvpool_pool_bytes(const kvpool_t* pool);

/* All device bytes the pool allocated (pool with padding, scratch, status). */
size_t kvpool_device_bytes(const kvpool_t* pool);

/* Synchronise `stream`, then return and clear the device status word
 * (KVPOOL_OK or the first device-side error recorded). */
int kvpool_status(kvpool_t* pool, void* stream);

/* Re-arm the write-once guard of one layer so it can be compressed again. */
int kvpool_reset_layer(kvpool_t* pool, int layer);

/* Fill *view with the device pointers and sizes of one layer. */
int kvpool_layer_view(const kvpool_t* pool, int layer, kvpool_layer_view_t* view);

/* Allocation-free variant of kvpool_attend, for callers that cannot call
 * cudaMalloc: an engine that reserved all device memory up front and hands
 * out slices itself (a cudaMalloc would fail or break its accounting), or a
 * latency-critical caller that cannot afford the device-wide synchronisation
 * cudaMalloc implies. The pages have no counterpart; this is an interface
 * convenience only.
 *
 * Inputs and outputs are the caller's: one compressed layer in the pool's
 * uniform layout (every group at width `bits`; layers of per-group widths,
 * kvpool_layer_view_t.mixed = 1, are not supported here and give wrong
 * results; the library cannot tell from these pointers), as
 * kvpool_layer_view describes it (token axis padded to
 * ctx_padded = ctx rounded up to a multiple of 128): kq int8
 * [kv_heads][ctx_padded][head_dim], vcodes uint8 [kv_heads][ctx_padded/32]
 * [head_dim][4*bits], vnorm float [kv_heads][ctx_padded], kscale one float;
 * kscales: NULL for a per-tensor layer, or a block-scaled layer's scales
 * float [kv_heads][ctx_padded][head_dim/32] (kvpool_layer_view_t.kscales;
 * *kscale, 1 in such a layer's view, multiplies every block scale);
 * Q, tail, out, softmax_scale and stream as in kvpool_attend. The result
 * equals kvpool_attend's on the same layer within float rounding.
 *
 * The split-context scratch is a fixed 8 MiB array inside the library, held
 * by every GPU that loads it until the process exits. A call needs
 * kv_heads * agents * (q_heads/kv_heads) * (head_dim + 2) * 4 bytes of it
 * per context split; calls that do not fit even one split (or with more than
 * 4096 query rows per KV head) return KVPOOL_ERR_INVALID_ARG. The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress with
 * that device current); make that first call before any stream capture. All
 * calls share the one array, so calls that overlap on the GPU (different
 * streams, or other host threads) race and must be serialised by the caller;
 * every byte a call reads from the array it has written first. Returns
 * KVPOOL_ERR_UNSUPPORTED on a device other than sm_103. */
int kvpool_attend_noalloc(const int8_t* kq, const uint8_t* vcodes, const float* vnorm,
                          const float* kscale, const float* kscales, int kv_heads, int head_dim,
                          int ctx, int bits,
                          const void* Q, int agents, int q_heads, const kvpool_tail_t* tail,
                          float* out, float softmax_scale, void* stream);

/* Copy the stored bytes of one compressed layer, token padding removed, to
 * caller buffers in host or device memory (any of the four may be NULL):
 * kq int8 [kv_heads][ctx][head_dim], vcodes uint8 [kv_heads][ceil(ctx/32)]
 * [head_dim][4*bits] (whole 32-token groups, see kvpool_layer_view_t; a layer
 * of per-group widths: uint8 [kv_heads][sum_g head_dim * 4 * b_g], see
 * kvpool_append_bits), vnorm float [kv_heads][ctx], kscale one float.
 * Asynchronous on
 * `stream` (host buffers should be pinned). This is the quantised-cache handoff
 * of the QKVShare blog (mhpn.cn, section 3.1: the sender packs the quantised
 * cache with its scales; the receiver loads it instead of recomputing). */
int kvpool_export_layer(const kvpool_t* pool, int layer, void* kq, void* vcodes, void* vnorm,
                        void* kscale, void* stream);

/* Load one layer from the four buffers kvpool_export_layer writes (same
 * kv_heads, ctx, head_dim and bits). Write-once like kvpool_compress:
 * KVPOOL_ERR_STATE if the layer already holds data. All four are required. */
int kvpool_import_layer(kvpool_t* pool, int layer, const void* kq, const void* vcodes,
                        const void* vnorm, const void* kscale, void* stream);

/* Load one layer of a block-scaled pool (kvpool_create_ex, k_block 32) from
 * what kvpool_export_layer, kvpool_export_kscales and kvpool_layer_widths
 * give for a layer of another block-scaled pool with the same kv_heads and
 * head_dim: len tokens (1..ctx); kq int8 [kv_heads][len][head_dim]; vcodes
 * the layer's code groups, per KV head back to back (kv_heads *
 * sum_g head_dim * 4 * widths[g] bytes: kvpool_export_layer's layout);
 * vnorm float [kv_heads][len]; kscales float [kv_heads][len][head_dim/32];
 * widths: host uint8 [ceil(len/32)], each from 2 to this layer's create
 * width (NULL: every group at the create width). The four buffers may be
 * host or device memory; the copies are asynchronous on `stream` (host
 * buffers should be pinned). Write-once: KVPOOL_ERR_STATE if the layer holds
 * tokens. Afterwards the layer holds len tokens and takes appends if len is a
 * multiple of 32. KVPOOL_ERR_UNSUPPORTED for per-tensor pools (they use
 * kvpool_import_layer). Source: the QKVShare blog (mhpn.cn), section 3.1:
 * the sender packs the quantised cache with its scales, and the receiver
 * loads it. */
int kvpool_import_layer_blocks(kvpool_t* pool, int layer, const void* kq, const void* vcodes, const void* vnorm,
                               const void* kscales, const uint8_t* widths, int len, void* stream);

/* Copy the library's float32 Lloyd-Max table for `bits` (2, 3 or 4) to host
 * arrays: 2^bits centroids (ascending) and 2^bits - 1 midpoints. The library
 * derives it on the host, once, in double precision. */
int kvpool_codebook(int bits, float* centroids, float* midpoints);

/* Static description of an error code. */
const char* kvpool_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVPOOL_H */
