/*
 * gattn.h -- C ABI of the GB300 (sm_103a) gated full-attention layer library.
 *
 * One thing runs here: the Qwen3.5-family full-attention decoder layer at
 * decode and speculative-verify time, for B sequences of R new rows each
 * (R = q_len: 1..4 for decode and the pages' verify rows, up to 32 for wider
 * verify rows and short prefill chunks, with B*R <= 32):
 *
 *   q_full = Wq x  (doubled q_proj: per head h the rows [h*2d, h*2d+d) are the
 *                   query and [h*2d+d, (h+1)*2d) the output gate)
 *   k = Wk x,  v = Wv x
 *   q = RoPE(RMSNorm(query, q_norm)),  k = RoPE(RMSNorm(k, k_norm))
 *   cache[cache_pos + r] = bf16(k), bf16(v)
 *   attn = causal GQA softmax(q k^T / sqrt(d)) v over t <= cache_pos + r
 *   out = Wo (attn * sigmoid(gate))
 *
 * Sources: "feat(engine): stage D6 - qwen3_5 dense full-attn deltas" (Summary:
 * doubled q_proj -> split queries/gate -> o_proj(attn * sigmoid(gate)); Audit
 * table: partial_rotary_factor, has_qk_norm); Atlas "spark_model/forward/
 * qwen3_5/mod.rs" (Qwen35ForwardConfig, q_total = num_heads*head_dim*2,
 * LayerKvCache: caller pre-allocates, KV-append at cache_pos, attention over
 * cache_pos+1); DS4Server issue 113 "Reproduction and boundary" (the verify
 * head-chunk plan); TensorFold issue 503 "Option C" (generic affine row decoder,
 * 2-8 bit, groups 32/64/128).
 *
 * Optional parts, each on the same kernels: the decoder block around the layer
 * (input RMSNorm, residual add, post-attention RMSNorm: gattn_layer_step_block;
 * Atlas mod.rs module doc, FullAttentionLayer input_ln / post_ln), Turbo4
 * quantized caches (Bf16KTurbo4V and symmetric Turbo4: gattn_kv_register_turbo4v,
 * gattn_kv_register_turbo4; Atlas mod.rs MetalKvDtype, LayerKvCache) and
 * attention masks (gattn_layer_set_mask; DS4Server issue 113, broadcast and
 * head-specific masks of the verify route).
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device addresses, (host) host memory.
 *   - Weights, caches, x, out and cache_pos are BORROWED: the library never
 *     frees them.  The library OWNS its handles, its repacked weights, its
 *     scratch and its TMA descriptors (freed by the matching destroy call).
 *   - A status other than GATTN_OK leaves a message for gattn_last_error()
 *     (thread-local, valid until the next call on the same thread).
 *   - Streams are cudaStream_t values passed as gattn_stream (0 = legacy default).
 *   - Inadmissible configurations are rejected at create time, never silently
 *     at step time.
 */
#ifndef GATTN_H
#define GATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gattn_stream; /* same type as cudaStream_t */

typedef enum gattn_status {
    GATTN_OK = 0,
    GATTN_E_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    GATTN_E_UNSUPPORTED = 2,   /* admissible on the pages but not built here */
    GATTN_E_CUDA = 3,          /* a CUDA runtime/driver call failed */
    GATTN_E_DEVICE_RANGE = 4,  /* a kernel saw cache_pos + q_len > capacity */
    GATTN_E_STATE = 5,         /* call out of order (e.g. step before set_weights) */
    GATTN_E_DEVICE_TIMEOUT = 6 /* a bounded device wait gave up (kernel returned early) */
} gattn_status;

enum { GATTN_DTYPE_F32 = 0, GATTN_DTYPE_BF16 = 1 };
enum { GATTN_PROJ_Q = 0, GATTN_PROJ_K = 1, GATTN_PROJ_V = 2, GATTN_PROJ_O = 3 };

/*
 * Layer configuration (mirrors the config fields of Qwen35ForwardConfig).
 *   hidden                 Hd, width of x and out; Hd % 128 == 0 and Hd <= 16384
 *   num_heads, num_kv_heads H, Hk (H % Hk == 0, gqa = H / Hk; query head h uses KV head h / gqa);
 *                          H * d % 128 == 0 and H * d <= 16384
 *   head_dim               d; d % 64 == 0 and d <= 256 in this library
 *   partial_rotary_factor  prf in (0, 1]; rotary dims rd = trunc(d * prf), even and >= 2
 *   rope_theta             base of inv_freq_i = theta^(-2i/rd)
 *   rms_eps                QK-RMSNorm epsilon (inside the square root)
 *   bits, group_size       default code width {2,3,4,5,6,8} and group {32,64,128}
 *   proj_bits[4], proj_group[4]  per projection q,k,v,o; 0 = the default
 *   x_dtype                GATTN_DTYPE_F32 or GATTN_DTYPE_BF16 (out is always bf16)
 *   max_batch, max_q_len   upper bounds for step(); max_batch*max_q_len <= 32 (<= 16 for
 *                          fp32 x)
 *   head_chunk             1 = the verify head-chunk plan is on (the pages'
 *                          default), 0 = off; both routes give the same result
 */
typedef struct gattn_cfg {
    int32_t hidden;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    float partial_rotary_factor;
    float rope_theta;
    float rms_eps;
    int32_t bits;
    int32_t group_size;
    int32_t proj_bits[4];
    int32_t proj_group[4];
    int32_t x_dtype;
    int32_t max_batch;
    int32_t max_q_len;
    int32_t head_chunk;
} gattn_cfg;

/*
 * Packed affine weights of one projection in the interchange layout, all (device):
 *   packed  uint32 [N][K*bits/32]: row n is an LSB-first bitstream, code k at
 *           bits [k*bits, (k+1)*bits) of the row's little-endian words
 *   scales  bf16   [N][K/group]
 *   biases  bf16   [N][K/group]      weight = scale * code + bias
 * N x K: q = (2*H*d) x Hd, k = v = (Hk*d) x Hd, o = Hd x (H*d).
 */
typedef struct gattn_proj {
    const uint32_t *packed;
    const uint16_t *scales;
    const uint16_t *biases;
} gattn_proj;

typedef struct gattn_weights {
    gattn_proj proj[4];        /* q, k, v, o */
    const uint16_t *q_norm;    /* bf16 [d] (device) */
    const uint16_t *k_norm;    /* bf16 [d] (device) */
} gattn_weights;

/*
 * A caller-owned bf16 KV cache (device), element (b, kv_head, token, j) of K at
 *   k + b*stride_batch + kv_head*stride_head + token*stride_token + j
 * and the same for V (same strides).  Strides are in elements; each must be a
 * multiple of 8 (16 bytes) and the base pointers 16-byte aligned.
 * [B][Hk][cap][d] is stride_token = d, stride_head = cap*d, stride_batch = Hk*cap*d;
 * the token-major [B][cap][Hk*d] layout is stride_token = Hk*d, stride_head = d.
 */
typedef struct gattn_kv_desc {
    void *k;
    void *v;
    int32_t batch;       /* sequences held */
    int32_t capacity;    /* tokens per sequence */
    int64_t stride_token;
    int64_t stride_head;
    int64_t stride_batch;
} gattn_kv_desc;

/* Intermediate taps of the last step (device, fp32), each may be NULL:
 *   y     [B*R][2*H*d + 2*Hk*d]  projection outputs q_full | k | v before the norm
 *   attn  [B*R][H*d]             attention output before the gate */
typedef struct gattn_taps {
    float *y;
    float *attn;
} gattn_taps;

typedef struct gattn_layer gattn_layer;
typedef struct gattn_kv gattn_kv;

/* Validate a configuration without touching a GPU.  Same rules as create(). */
gattn_status gattn_cfg_validate(const gattn_cfg *cfg);

/* Rotary dims the layer uses: trunc(head_dim * partial_rotary_factor), computed
 * in double ("rope dims" of the qwen3_5 deltas page); -1 if cfg is NULL. */
int32_t gattn_rotary_dims(const gattn_cfg *cfg);

/* Create a layer on the current CUDA device: validates cfg, allocates scratch
 * (sized by max_batch/max_q_len) and the repacked-weight buffers.  *out owned
 * by the caller, release with gattn_layer_destroy.  Errors: those of
 * gattn_cfg_validate (GATTN_E_INVALID_ARG, GATTN_E_UNSUPPORTED; *out = NULL),
 * GATTN_E_CUDA when an allocation or device query fails (nothing leaks). */
gattn_status gattn_layer_create(const gattn_cfg *cfg, gattn_layer **out);

/* Repack the interchange weights (TensorFold issue 503 "Option C" affine rows,
 * layout of gattn_proj) into the library's device tile layout (same bytes per
 * step); copies q_norm and k_norm.  Runs and synchronizes on `stream`; the
 * caller may free the interchange buffers after it returns.  Errors:
 * GATTN_E_INVALID_ARG for a NULL layer, weights or buffer; GATTN_E_CUDA when a
 * launch or copy fails.  May be called again to replace the weights. */
gattn_status gattn_layer_set_weights(gattn_layer *layer, const gattn_weights *w, gattn_stream stream);

/* Register a cache for this layer (Atlas qwen3_5 forward page, LayerKvCache:
 * the caller pre-allocates, the step appends at cache_pos): checks sizes and
 * alignment and encodes the TMA tensor maps once.  *out is owned by the
 * caller (gattn_kv_destroy); the cache memory is borrowed and must outlive the
 * registration, and the registration must not outlive the layer.  Errors:
 * GATTN_E_INVALID_ARG for a NULL or misaligned pointer, batch <= 0, capacity
 * < 16, a stride that is not a positive multiple of 8, or a layout the TMA
 * encoder rejects; GATTN_E_CUDA when the encoder cannot be found. */
gattn_status gattn_kv_register(gattn_layer *layer, const gattn_kv_desc *desc, gattn_kv **out);

/*
 * A caller-owned Bf16KTurbo4V cache (device): the "safer-asym" format of the
 * Atlas qwen3_5 forward page (MetalKvDtype::Bf16KTurbo4V, LayerKvCache with a
 * V-side scale buffer): K raw bf16, V in a Walsh-Hadamard-rotated basis as
 * 4-bit Lloyd-Max codebook indices plus one FP8 E4M3 scale per group of 16.
 *   K       bf16, element (b, kv_head, token, j) at
 *           k + b*k_stride_batch + kv_head*k_stride_head + token*k_stride_token + j
 *           (strides in elements, multiples of 8)
 *   v_codes uint8, the row of (b, kv_head, token) -- d/2 bytes, code j in the
 *           low (j even) or high (j odd) nibble of byte j/2 -- at
 *           v_codes + b*code_stride_batch + kv_head*code_stride_head + token*(d/2)
 *   v_scales uint8 E4M3, d/16 bytes per row, at
 *           v_scales + b*scale_stride_batch + kv_head*scale_stride_head + token*(d/16)
 * Code and scale strides are in bytes, multiples of 16; rows of one
 * (b, kv_head) are consecutive.  Pointers 16-byte aligned; capacity a
 * multiple of 16; head_dim a power of two from 64 to 256.  A V row is
 * dequantized as H (s * c(code)) / sqrt(d) (H the Sylvester Hadamard matrix,
 * c the levels of gattn_turbo4_codebook); the step quantizes its new V rows
 * from their bf16 values (gattn_turbo4_quantize_device states how) and
 * applies the inverse rotation once to each attention output row.
 */
typedef struct gattn_kv_turbo4v_desc {
    void *k;
    void *v_codes;
    void *v_scales;
    int32_t batch;
    int32_t capacity;
    int64_t k_stride_token, k_stride_head, k_stride_batch;
    int64_t code_stride_head, code_stride_batch;
    int64_t scale_stride_head, scale_stride_batch;
} gattn_kv_turbo4v_desc;

/* Register a Bf16KTurbo4V cache (as gattn_kv_register).  GATTN_E_INVALID_ARG
 * for a bad pointer, stride, capacity or head_dim. */
gattn_status gattn_kv_register_turbo4v(gattn_layer *layer, const gattn_kv_turbo4v_desc *desc,
                                       gattn_kv **out);

/*
 * A caller-owned symmetric Turbo4 cache (device; MetalKvDtype::Turbo4 of the
 * Atlas qwen3_5 forward page: K and V both WHT-rotated 4-bit Lloyd-Max codes
 * with E4M3 group-of-16 scales).  K and V planes have the layout of the V
 * planes of gattn_kv_turbo4v_desc (one set of code and scale strides for
 * both).  The step quantizes its new K rows from the bf16 values of the
 * normed, rotary-embedded keys, and its new V rows as for Bf16KTurbo4V; the
 * attention rotates each q row once (q' = H q / sqrt(d)) so the scores are
 * q' . dequantized key rows in the rotated basis.  Same rules as
 * gattn_kv_register_turbo4v (no bf16 K).
 */
typedef struct gattn_kv_turbo4_desc {
    void *k_codes;
    void *k_scales;
    void *v_codes;
    void *v_scales;
    int32_t batch;
    int32_t capacity;
    int64_t code_stride_head, code_stride_batch;
    int64_t scale_stride_head, scale_stride_batch;
} gattn_kv_turbo4_desc;

gattn_status gattn_kv_register_turbo4(gattn_layer *layer, const gattn_kv_turbo4_desc *desc,
                                      gattn_kv **out);

/* The Turbo4 codebook as the kernels use it (host, no GPU): the 16 levels of
 * the Lloyd-Max quantizer of N(0, 1), ascending, rounded to fp32, and the 15
 * decision thresholds between them (midpoints taken in double, then rounded;
 * the middle one is 0).  Computed once per process by Lloyd's iteration (the
 * pages name the codebook, Atlas MetalKvDtype::Turbo4, but print no values).
 * GATTN_E_INVALID_ARG for a NULL array. */
gattn_status gattn_turbo4_codebook(float levels[16], float thresholds[15]);

/*
 * Quantize `rows` bf16 rows of `d` values (device, [rows][d]) into Turbo4
 * codes (device, [rows][d/2]) and E4M3 scales (device, [rows][d/16]), as the
 * step does for its new V rows; enqueued on `stream`, no synchronization.
 * Per row: y = H v * fp32(1/sqrt(d)) (butterfly stages h = 1, 2, 4, ... in
 * fp32); per group of 16: ss = pairwise fp32 sum of y_i^2, u_i = y_i /
 * sqrt(ss/16), code_i = number of thresholds below u_i, scale = E4M3 (nearest,
 * ties to even, saturating at 448) of sqrt(ss / pairwise sum of level^2); a
 * zero group gets codes 0 and scale 0.  d a power of two from 64 to 256.
 * GATTN_E_INVALID_ARG for rows < 0, a NULL pointer with rows > 0 or another
 * d; GATTN_E_CUDA when the launch fails.  rows == 0 launches nothing.
 */
gattn_status gattn_turbo4_quantize_device(const void *v_bf16, int64_t rows, int32_t d,
                                          void *codes, void *scales, gattn_stream stream);

/*
 * One layer step, enqueued on `stream` with no host synchronization and no
 * allocation (capturable into a CUDA graph).
 *   x          (device) [batch][q_len][hidden], cfg.x_dtype
 *   kv         registered cache holding sequences 0..batch-1
 *   cache_pos  (device) int32 [batch]: first new position of each sequence;
 *              the new rows go to cache_pos[b] .. cache_pos[b]+q_len-1 and
 *              row r attends positions 0 .. cache_pos[b]+r
 *   out        (device) bf16 [batch][q_len][hidden]
 * A sequence with cache_pos < 0 or cache_pos + q_len > capacity is skipped on
 * the device (its cache is untouched and its out rows are zero) and the next
 * gattn_layer_poll_status() returns GATTN_E_DEVICE_RANGE.  One step at a time
 * per layer handle: steps of one handle on different streams race on its scratch.
 * Errors (nothing is launched): GATTN_E_INVALID_ARG for a NULL argument, a
 * cache registered with another layer, batch outside [1, min(max_batch, cache
 * batch)] or q_len outside [1, max_q_len]; GATTN_E_STATE before
 * gattn_layer_set_weights; GATTN_E_UNSUPPORTED for a step the set mask does not
 * take (gattn_layer_set_mask);
 * GATTN_E_CUDA when a launch fails.
 */
gattn_status gattn_layer_step(gattn_layer *layer, const void *x, gattn_kv *kv,
                              const int32_t *cache_pos, int32_t batch, int32_t q_len,
                              void *out, gattn_stream stream);

/*
 * gattn_layer_step from host buffers: copies x and cache_pos into the layer's
 * own device staging buffers, enqueues the step on `stream` after those
 * copies, and the copy of its output rows into out_host after the step, then
 * returns (no host synchronization: out_host holds the result once `stream`
 * has reached it).
 *   x_host          (host) [batch][q_len][hidden], cfg.x_dtype
 *   cache_pos_host  (host) int32 [batch], as cache_pos of gattn_layer_step
 *   out_host        (host) bf16 [batch][q_len][hidden]
 * The input copies run on a stream of the layer's own, ordered before the
 * step but not after earlier work on `stream`: x_host and cache_pos_host must
 * hold the step's inputs when the call is made (not be written by work still
 * pending on `stream`), and stay unchanged until the stream has passed the
 * step.  out_host is written by a copy on `stream` after the step.  Pinned
 * (page-locked) memory makes the copies asynchronous.  The staging buffers
 * (two input slots used in turn, allocated with the layer for the largest
 * step it admits) belong to the handle, like its scratch.  Errors: those of
 * gattn_layer_step, checked before anything is enqueued; GATTN_E_CUDA when a
 * copy or a launch fails.
 */
gattn_status gattn_layer_step_host(gattn_layer *layer, const void *x_host, gattn_kv *kv,
                                   const int32_t *cache_pos_host, int32_t batch, int32_t q_len,
                                   void *out_host, gattn_stream stream);

/* Synchronize `stream`, then read and clear the layer's device status word:
 * GATTN_OK, GATTN_E_DEVICE_RANGE or GATTN_E_DEVICE_TIMEOUT (GATTN_E_INVALID_ARG
 * for a NULL layer, GATTN_E_CUDA when the synchronization or read fails). */
gattn_status gattn_layer_poll_status(gattn_layer *layer, gattn_stream stream);

/* Ask the next steps to also write the taps (layout of gattn_taps; borrowed
 * device buffers; NULL or all-NULL turns them off).  GATTN_E_INVALID_ARG for a
 * NULL layer.  Test instrumentation, not part of the layer's computation. */
gattn_status gattn_layer_set_taps(gattn_layer *layer, const gattn_taps *taps);

/*
 * An attention mask for the following steps (DS4Server issue 113: the verify
 * route's broadcast and head-specific masks), device bytes, borrowed:
 *   byte mask[b*stride_batch + hm*stride_head + r*stride_row + t]
 * nonzero = row r of sequence b may attend cache position t; hm = 0 for a
 * broadcast mask (heads == 1), the query head for a head-specific one
 * (heads == num_heads).  A mask replaces the causal rule: row r attends the
 * marked positions t < cache_pos[b] + q_len (positions >= `positions` are not
 * attended and never read); a row with no position left gives a zero attention
 * row.  Strides in bytes; stride_row >= positions.  The step refuses
 * (GATTN_E_UNSUPPORTED) a head-specific mask when the head-chunked verify route
 * applies (it hands the mask unchanged to every head chunk, where only a
 * broadcast mask fits).  The contents may
 * change between steps (read at run time, graph-capturable).
 */
typedef struct gattn_mask {
    const uint8_t *mask;
    int32_t heads;
    int32_t positions;
    int64_t stride_row, stride_head, stride_batch;
} gattn_mask;

/* Set (or with NULL / mask->mask == NULL clear) the attention mask of the
 * following steps.  GATTN_E_INVALID_ARG for a NULL layer, heads other than 1
 * or num_heads, positions <= 0, stride_row < positions or a negative stride. */
gattn_status gattn_layer_set_mask(gattn_layer *layer, const gattn_mask *mask);

/* Free a layer and everything it owns (NULL is a no-op).  Call it after the
 * layer's last step has finished on the GPU and after destroying the caches
 * registered with it; borrowed buffers are left alone. */
void gattn_layer_destroy(gattn_layer *layer);
/* Free a cache registration (NULL is a no-op); the cache memory is the
 * caller's and is left alone. */
void gattn_kv_destroy(gattn_kv *kv);

/* Thread-local message of the last failed call on this thread ("" if none). */
const char *gattn_last_error(void);

/*
 * Host quantizer + packer for synthetic weights (host): per (row, group)
 *   bias = bf16(min w), scale = bf16((max w - min w)/(2^bits - 1)),
 *   code = clamp(nearest-even((w - bias)/scale), 0, 2^bits - 1), code = 0 if scale == 0,
 * all arithmetic in double with ties-to-even bf16 rounding, written into the
 * interchange layout above.  w float [N][K]; packed [N][K*bits/32];
 * scales/biases [N][K/group].  Requires K % group == 0 and K*bits % 32 == 0.
 */
gattn_status gattn_pack_affine_host(const float *w, int64_t N, int64_t K, int32_t bits,
                                    int32_t group, uint32_t *packed, uint16_t *scales,
                                    uint16_t *biases);

/* Decode interchange codes on the GPU (device in/out): codes uint8 [N][K],
 * enqueued on `stream`.  GATTN_E_INVALID_ARG for a NULL pointer, negative
 * sizes, bits outside 1..8 or K*bits not a multiple of 32. */
gattn_status gattn_unpack_codes_device(const uint32_t *packed, int64_t N, int64_t K, int32_t bits,
                                       uint8_t *codes, gattn_stream stream);

/* Dequantize one projection of a layer FROM ITS REPACKED DEVICE LAYOUT with the
 * same register unpack the projection kernels use: w (device) float [N][K],
 * w = fp32(scale*code + bias) (exact: scale*code has <= 16 significant bits).
 * Allocates a temporary device buffer and synchronizes `stream`.  Errors:
 * GATTN_E_INVALID_ARG (NULL, proj outside 0..3), GATTN_E_STATE before
 * gattn_layer_set_weights, GATTN_E_CUDA. */
gattn_status gattn_layer_dequant_device(gattn_layer *layer, int32_t proj, float *w,
                                        gattn_stream stream);

/*
 * Same result as gattn_layer_dequant_device (bit for bit), for callers that
 * cannot allocate device memory or synchronize at the point of the call: code
 * recording a CUDA graph in global capture mode, code whose framework owns the
 * whole device memory budget, latency-sensitive paths.  It allocates nothing:
 * its staging buffer is a fixed 16 MiB device array inside the library (held
 * on every GPU that loads it, until exit), and it returns without waiting for
 * the GPU (w is ready once `stream` reaches that point).
 *   - Limit: the 128-row blocks spanning the projection times K must fit in
 *     4 Mi floats; larger projections fail with GATTN_E_UNSUPPORTED and a
 *     message naming the sizes.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress), and so does the first call after the device's
 *     context was created anew (e.g. after cudaDeviceReset); make those
 *     calls before any stream capture.
 *   - A sticky CUDA error of the context is returned as GATTN_E_CUDA; an
 *     error left by an earlier, unrelated launch is neither reported nor
 *     cleared.
 *   - Every call shares the one array: calls that can overlap on the GPU (on
 *     different streams, or different layers at once) race on it.
 * The pages have no counterpart of this entry point (it is a library utility).
 */
gattn_status gattn_layer_dequant_device_static(gattn_layer *layer, int32_t proj, float *w,
                                               gattn_stream stream);

/*
 * The verify head-chunk plan (DS4Server issue 113, "Reproduction and boundary"):
 * when enabled and q_len*gqa > 32 and q_len <= 32, the query heads of each KV
 * group are split into chunks of max(1, min(gqa, 32/q_len)) heads (the last
 * chunk of a group holds the remainder), in head order; otherwise each KV
 * group is one chunk.  Writes up to `cap` chunks (first head, head count) and
 * returns the chunk count, or -1 for bad arguments.
 */
int32_t gattn_head_chunk_plan(int32_t q_len, int32_t num_heads, int32_t num_kv_heads,
                              int32_t enabled, int32_t *chunk_first_head, int32_t *chunk_len,
                              int32_t cap);


/*
 * Decoder-block variant of gattn_layer_step: the steps on either side of the
 * layer in forward_full_attention (Atlas spark_model/forward/qwen3_5/mod.rs,
 * module doc and FullAttentionLayer: input_ln, post_ln, norm -> projections ->
 * attention -> residual + post-norm -> MLP).  Per row of x:
 *   h          = x / sqrt(mean(x^2) + rms_eps) * input_ln     (RMSNorm)
 *   out        = bf16(x + layer(h))                           (residual stream)
 *   out_normed = bf16(RMSNorm(out) * post_ln)                 (the MLP's input;
 *                computed from the stored bf16 row of out)
 * Arguments: x is the raw hidden state [batch][q_len][hidden] in the layer's x
 * dtype (device); input_ln and post_ln are bf16 [hidden] device vectors,
 * borrowed; out is bf16 [batch][q_len][hidden]; out_normed (may be NULL, then
 * post_ln may be NULL too) is bf16 of the same shape and must not alias out.
 * Cache, position, launch and error behaviour as gattn_layer_step.  The
 * post-norm runs inside the o_proj launch (its last CTA to finish normalizes
 * every row) when batch * q_len * hidden <= 16384 and out, out_normed and
 * post_ln are 16-byte aligned, else in one more launch.  The norm of the
 * input is rounded to bf16 for a bf16 layer (kept fp32 for an fp32 one)
 * before the projections.  GATTN_E_INVALID_ARG for a NULL input_ln,
 * out_normed without post_ln or aliasing out.
 */
gattn_status gattn_layer_step_block(gattn_layer *layer, const void *x, gattn_kv *kv,
                                    const int32_t *cache_pos, int32_t batch, int32_t q_len,
                                    const void *input_ln, const void *post_ln, void *out,
                                    void *out_normed, gattn_stream stream);

/* Per-step launch report of the layer's last step: number of kernel launches
 * it enqueued, all of them this library's own kernels: 4 (q|k|v projection,
 * attention, the merge of its chunk partials with the output gate, o_proj)
 * when the q|k|v kernel converts x itself, else 5 with the x prep launch, one
 * more for a decoder-block step whose post-norm takes its own launch. */
int32_t gattn_layer_launches_per_step(const gattn_layer *layer);

/* The kernels of the layer's last step, in launch order. */
enum {
    GATTN_KERNEL_XPREP = 1,     /* x -> tensor-core operand (+ input RMSNorm of the block) */
    GATTN_KERNEL_PROJ_QKV = 2,  /* q|k|v dequant projection + norm / rotary / KV append */
    GATTN_KERNEL_ATTN = 3,      /* causal GQA attention over key chunks (one-chunk segments:
                                   output gate -> o_proj operand) */
    GATTN_KERNEL_MERGE = 4,     /* merge of the attention chunk partials, output gate -> o_proj
                                   operand */
    GATTN_KERNEL_PROJ_O = 5,    /* o_proj (+ residual and fused post-norm of the block) */
    GATTN_KERNEL_POSTNORM = 6   /* post-attention RMSNorm of the block, own launch */
};
/* Writes up to `cap` GATTN_KERNEL_* values (host array) and returns the launch
 * count of the last step (0 before any step), or -1 for bad arguments. */
int32_t gattn_layer_step_kernels(const gattn_layer *layer, int32_t *kinds, int32_t cap);

/* Instrumentation: with n >= 2 cudaEvent_t handles, each following step
 * records events[i] on its stream right before its i-th kernel launch (for
 * i < n - 1) and events[n-1] after its last launch, so per-kernel durations
 * can be read with cudaEventElapsedTime (use n = launches_per_step + 1).
 * n == 0 (or events == NULL) turns it off.  The events are borrowed.
 * Recording between kernels serializes them (no programmatic overlap), so use
 * it for per-kernel timing passes only. */
gattn_status gattn_layer_set_events(gattn_layer *layer, void *const *events, int32_t n);

/* Failure-detection test hook for the bounded device waits.
 *
 * Every wait of the projection kernels (a weight stage landing in shared
 * memory, a stage slot being released, partial sums arriving from the other
 * CTAs of a cluster) gives up after a time limit; the kernel then skips the
 * remaining work of that CTA, still reaches every barrier, and returns; the
 * layer's status word gets the timeout bit, so the next
 * gattn_layer_poll_status() returns GATTN_E_DEVICE_TIMEOUT and the context
 * stays usable.
 *
 * wait_limit_ns: the limit of those waits for the following steps, in ns;
 *   0 restores the default (2 s).  Negative: GATTN_E_INVALID_ARG.
 * withhold_stage: nonzero makes CTA 0 of every following q|k|v projection
 *   launch skip the copy of its last weight stage, so that the wait for it
 *   runs out after wait_limit_ns (the outputs of such a step are garbage);
 *   0 turns that off.
 *
 * Meant for tests of the timeout path; a layer that never calls it keeps the
 * default limit and withholds nothing. */
gattn_status gattn_layer_set_test_wait(gattn_layer *layer, int64_t wait_limit_ns,
                                       int32_t withhold_stage);

#ifdef __cplusplus
}
#endif

#endif /* GATTN_H */
