// kernels.cuh -- parameter blocks, layout constants and launchers shared by the
// library's translation units (internal; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "turbo.cuh"

struct gattn_layer;

namespace gattn {

// Launch kernel f and return the status of this launch alone.  (The
// `<<<...>>>` form followed by cudaGetLastError() would also report, and
// clear, an error left by an earlier unrelated asynchronous launch.)  A sticky
// error of the context is reported as it is.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_plain(void (*f)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, f, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------- projection layout
//
// A projection matrix W [N][K] (q|k|v concatenated for the fused launch) is
// repacked into "units" of 32 rows x 128 k.  A row block is kWR units stacked
// along N (one per consumer warp); the device buffer is ordered
// [row block][k unit][warp][unit bytes], so one pipeline stage (all warps'
// units of one k unit) is a single contiguous bulk copy.
//
// Unit bytes: codes 512*bits (per lane 16*bits bytes, 16-byte chunk i of lane
// t at (i*32 + t)*16), then scale/bias pairs 128*(128/group) bytes: for group
// gi of the unit, lane-quad g, row slot rs (rows g, g+8, g+16, g+24) one
// uint32 (bf16 scale low half, bf16 bias high half) at ((gi*8 + g)*4 + rs)*4.
//
// Lane t = 4g + c holds the tensor-core A fragments of both 16-row m-tiles
// for all 8 k16-steps: fragment value v (0..7) of MMA mi = 2*kstep + mt is
// row mt*16 + g + 8*((v>>1)&1), k kstep*16 + 2c + 8*(v>>2) + (v&1), stored as
// code number mi*8 + v of the lane's bitstream (4-bit codes use the nibble
// order 0,4,1,5,2,6,3,7 inside each word so that one mask extracts a pair).
constexpr int kWR = 4;            // consumer warps per CTA = 32-row tiles per row block
constexpr int kRBR = 32 * kWR;    // rows per row block
constexpr int kKU = 128;          // k per unit

// Threads of a projection CTA: kWR consumer warps and one producer warp.
__host__ __device__ constexpr int proj_threads(int NT) { return NT > 0 ? (kWR + 1) * 32 : 0; }

__host__ __device__ inline int unit_code_bytes(int bits) { return 512 * bits; }
__host__ __device__ inline int unit_sb_bytes(int group) { return 128 * (128 / group); }
__host__ __device__ inline int unit_bytes(int bits, int group)
{
    return unit_code_bytes(bits) + unit_sb_bytes(group);
}

// x operand in tensor-core B-fragment order, fp16, for MP = 8*NT columns:
// element (m, k) at half offset (((ku*NT + m/8)*8 + kstep)*32 + lane)*4 + hi*2 + e
// with ku = k/128, kstep = (k%128)/16, q = k%16, hi = q/8, lane = (m%8)*4 + (q%8)/2,
// e = q%2.  Group sums of the same fp16 values: xsum[(ku*(128/group) + gi)*MP + m].
__host__ __device__ inline long long x16_offset(int m, int k, int NT)
{
    int ku = k >> 7, kk = k & 127, kstep = kk >> 4, q = kk & 15;
    int lane = ((m & 7) << 2) | ((q & 7) >> 1);
    return ((((long long)ku * NT + (m >> 3)) * 8 + kstep) * 32 + lane) * 4 + ((q >> 3) << 1) +
           (q & 1);
}

// One cluster computes one block of rows (whole heads for the q|k|v
// projection) over all of K: its rbc row blocks times ks k-splits are the
// cluster's CTAs (rank = row block * ks + split).  Partial sums are reduced
// through distributed shared memory, so no global scratch is used.
struct ProjArgs {
    const uint8_t *w;     // repacked weights
    const __half *x16;    // B-fragment-ordered x
    const float *xsum;    // group sums of x16
    int nrb, nku;         // row blocks, k units
    int N;                // valid rows
    int M;                // valid x rows (columns of the product)
    int group;
    int unit_bytes, step_bytes, stage_bytes, stages;
    int rbc;              // row blocks per cluster
    int ks;               // k splits per row block (cluster size = rbc * ks)
    int eb_rows;          // rows per cluster = rbc * kRBR
    int xsplit;           // > 0: column m + xsplit holds the low fp16 part of column m
    int recv_cap;         // floats of the split-K receive area (proj_recv_cap)
    // > 0 (q|k|v only): the CTA converts the layer input x itself into a table
    // of this many bytes of shared memory (its k units' fp16 fragments and group
    // sums), and the stages carry weights only; 0: x16 / xsum come prepared
    int xtab_bytes;
    const void *xraw;     // x [M][K] for the table
    int x_f32;            // x dtype: fp32 (1) or bf16 (0)
    unsigned long long wait_ns;   // bound of every wait on a stage
    // failure test hook (q|k|v): nonzero makes CTA 0 withhold its last weight
    // stage, so that stage's wait runs out
    int withhold;
    unsigned *status;
};

#ifdef __CUDACC__
__device__ __forceinline__ unsigned arg_fold(const ProjArgs &a)
{
    return arg_fold(a.w, a.x16, a.xsum, a.nrb, a.nku, a.N, a.M, a.group, a.unit_bytes, a.step_bytes,
                    a.stage_bytes, a.stages, a.rbc, a.ks, a.eb_rows, a.xsplit, a.recv_cap,
                    a.xtab_bytes, a.xraw, a.x_f32, a.wait_ns, a.withhold, a.status);
}
#endif

// qkv epilogue: per head block, RMSNorm + RoPE + bf16 append / q and gate outputs
struct EpiQKV {
    int R;                         // q_len; column m is sequence m / R, row m % R
    int H, Hk, d, rd;
    int Nq, Nkv;
    const int *cache_pos;
    int cap;
    __nv_bfloat16 *kc, *vc;        // cache bases
    long long st_tok, st_head, st_batch;
    const uint16_t *q_norm, *k_norm;
    float eps;
    const float2 *inv_freq2;       // [rd/2] inv_freq as float pairs: hi = fp32(f), lo = fp32(f - hi)
    __nv_bfloat16 *qn;             // [B][R][H][d]
    float *gate;                   // [M][H*d]
    float *tap_y;                  // [M][Nq + 2 Nkv] or null
    // Bf16KTurbo4V cache: the new V rows are quantized (turbo.cuh), not stored
    // as bf16 (null: bf16 V)
    uint8_t *vq_codes, *vq_scales;
    long long cq_head, cq_batch, sq_head, sq_batch;   // byte strides
    // symmetric Turbo4 cache: the new K rows quantized the same way (null: bf16 K)
    uint8_t *kq_codes, *kq_scales;
    long long kcq_head, kcq_batch, ksq_head, ksq_batch;
    TurboTables tq;
};

#ifdef __CUDACC__
__device__ __forceinline__ unsigned arg_fold(const EpiQKV &e)
{
    unsigned h = arg_fold(e.R, e.H, e.Hk, e.d, e.rd, e.Nq, e.Nkv, e.cache_pos, e.cap, e.kc, e.vc,
                          e.st_tok, e.st_head, e.st_batch, e.q_norm, e.k_norm, e.eps, e.inv_freq2,
                          e.qn, e.gate, e.tap_y, e.vq_codes, e.vq_scales, e.cq_head, e.cq_batch,
                          e.sq_head, e.sq_batch, e.kq_codes, e.kq_scales, e.kcq_head, e.kcq_batch,
                          e.ksq_head, e.ksq_batch, e.tq.inv_sqrt_d);
#pragma unroll
    for (int i = 0; i < 16; i += 4)
        h ^= arg_fold(e.tq.lv[i], e.tq.th[i < 15 ? i : 14]);
    return h;
}
#endif

struct EpiO {
    int R;
    const int *cache_pos;
    int cap;
    __nv_bfloat16 *out;            // [M][N]
    const void *resid;             // decoder block: out = bf16(resid + o_proj), or null
    int resid_f32;                 // resid dtype: fp32 (1) or bf16 (0)
    // decoder block, post-attention RMSNorm in the o_proj launch (null: none):
    // out_n = bf16(RMSNorm(out) * post_w), finished by the last CTA to arrive
    const uint16_t *post_w;        // [N] bf16 bits
    __nv_bfloat16 *out_n;          // [M][N]
    float eps;
    float *ss_part;                // [grid][M] each CTA's sums of squares of its stored rows
    unsigned *ticket;              // CTAs arrived; zero between launches
};

#ifdef __CUDACC__
__device__ __forceinline__ unsigned arg_fold(const EpiO &e)
{
    return arg_fold(e.R, e.cache_pos, e.cap, e.out, e.resid, e.resid_f32, e.post_w, e.out_n, e.eps,
                    e.ss_part, e.ticket);
}
#endif

// the post-norm rides in the o_proj launch up to this many output elements
// (one CTA normalizes every row); larger steps launch postnorm_kernel
constexpr int kPostFuseMaxElems = 16384;

enum { kModeQKV = 0, kModeO = 1 };

// Floats of the receive area a projection CTA reserves for the partial sums
// the cluster's CTAs push to it (proj.cuh): at most MP = 8 NT operand columns.
// q|k|v: ceil(M / csize) columns (x2 with the fp32 low planes) of ks x eb_rows
// values, at most (MP + 15) * 128 for clusters of <= 8 CTAs;
// o_proj: ks * M * ceil(128 / csize) <= MP * 143 for clusters of <= 16 CTAs.
__host__ __device__ inline int proj_recv_cap(int mode, int NT)
{
    return mode == kModeQKV ? (8 * NT + 15) * 128 : 8 * NT * 143;
}

// launchers (return cudaGetLastError() of the launch)
cudaError_t launch_proj(int bits, int NT, int mode, const ProjArgs &a, const EpiQKV &eq,
                        const EpiO &eo, int grid, bool pdl, cudaStream_t s);
int proj_smem_bytes(const ProjArgs &a);
// shared memory past the projection's stage ring: barriers, flags, epilogue
// statics; the q|k|v epilogue stages up to kWR head rows of d <= 256 values
constexpr int kValsFloats = kWR * 256;
__host__ __device__ inline int proj_tail_bytes(int eb_rows)
{
    (void)eb_rows;
    return 256 + kValsFloats * 4 + 2 * 256 * 4 + 128 * 8 + 32 * 4;
}
cudaError_t proj_set_smem_limits(int bits, int NT, int mode, int bytes);
cudaError_t proj_occupancy(int bits, int NT, int mode, int group, int smem, int *blocks_per_sm);
// clusters of csize CTAs that can be resident at once (0: that size cannot launch)
cudaError_t proj_max_clusters(int bits, int NT, int mode, int group, int smem, int csize, int *n);

// fp32 x is split exactly into hi = fp16(x) (column m) and lo = fp16(x - hi)
// (column M + m); bf16 x converts to fp16 exactly (finite, |x| < 65504).
// in_w (bf16 [K], or null): decoder-block input, the operand is RMSNorm(x) * in_w.
cudaError_t launch_xprep(const void *x, int x_dtype, int M, int K, int group, int NT, __half *x16,
                         float *xsum, const uint16_t *in_w, float eps, bool pdl, cudaStream_t s);
// out_n[m] = bf16(RMSNorm(r[m]) * w) for the M bf16 rows of r (N columns each).
cudaError_t launch_postnorm(const __nv_bfloat16 *r, const uint16_t *w, float eps, int M, int N,
                            __nv_bfloat16 *out_n, bool pdl, cudaStream_t s);

struct RepackSrc {
    const uint32_t *packed[3];
    const uint16_t *scales[3];
    const uint16_t *biases[3];
    int rows[3];                   // rows of each source, concatenated in order
    int nsrc;
};
cudaError_t launch_repack(const RepackSrc &src, int K, int bits, int group, int nrb, uint8_t *dst,
                          cudaStream_t s);
cudaError_t launch_dequant_tiles(const uint8_t *w, int N, int K, int bits, int group, int nrb,
                                 float *out, cudaStream_t s);
cudaError_t launch_unpack_codes(const uint32_t *packed, long long N, long long K, int bits,
                                uint8_t *codes, cudaStream_t s);

// Where one projection of a layer lives in its repacked tile layout (for
// entry points outside api.cu): row blocks [rb0, rb1) of buffer w hold the
// projection's rows row0 .. row0 + rows - 1 (counted from the buffer's row 0).
struct ProjTiles {
    const uint8_t *w;      // the buffer's first row block
    int nku, bits, group, step_bytes;
    int row0, rows, K;
};
bool layer_proj_tiles(const ::gattn_layer *layer, int proj, ProjTiles *out);

// ------------------------------------------------------------- attention

constexpr int kAttnWarps = 8;          // consumer warps
constexpr int kAttnThreads = (kAttnWarps + 1) * 32;
constexpr int kAttnUnit = 16;          // tokens per stream-K unit
constexpr int kAttnTile = 64;         // tokens per pipeline stage (<= 64: the P tile width)
constexpr int kAttnStages = 4;        // pipeline stages, at most (fewer when shared memory is short)
constexpr int kMaxRowBlocks = 64;
// query rows an attention row block holds, at most (more when one head has more
// rows): one 16-row MMA tile, so a tile's products stay short and a KV group's
// rows spread over more CTAs
constexpr int kRowBlockRows = 16;
constexpr int kAttnMaxRows = 64;       // query rows per segment

// floats per attention partial slot: m[64], l[64], O[64][d]
__host__ __device__ inline int attn_slot_floats(int d) { return 2 * kAttnMaxRows + kAttnMaxRows * d; }

struct AttnArgs {
    const __nv_bfloat16 *qn;     // [B][R][H][d]
    const float *gate;           // [M][H*d]
    const int *cache_pos;
    int B, R, H, Hk, d, cap;
    int nrb;                     // row blocks per KV group
    int nrb_u;                   // row blocks per KV group of the unchunked partition
    int rb_h0[kMaxRowBlocks];    // first head of each row block (relative to the group)
    int rb_nh[kMaxRowBlocks];    // heads of each row block
    float scale_log2;            // log2(e) / sqrt(d)
    int min_units;               // minimum 16-token units per chunk
    int split;                   // chunks per CTA aimed at (balance against per-chunk work)
    int max_chunks;              // chunks per segment, at most (<= 32)
    int attn_grid;               // CTAs of the attention launch (the chunk plan depends on it)
    int merge_rows;              // rows a segment, at most: the merge launch's CTAs per segment
    float *ws;                   // chunk partials, attn_slot_floats(d) per item
    // o_proj operand
    __half *x16;
    float *xsum;
    int NT, group_o;
    float *tap_attn;             // [M][H*d] or null
    unsigned *status;
    // Bf16KTurbo4V cache (vq != 0): V code / scale rows, the byte -> fp16 level
    // pair table, and the inverse rotation applied in the merge
    int vq;                      // 1: Turbo4 V, 2: Turbo4 K and V
    const uint8_t *vq_codes, *vq_scales;
    long long cq_head, cq_batch, sq_head, sq_batch;   // byte strides
    const uint8_t *kq_codes, *kq_scales;               // vq == 2
    long long kcq_head, kcq_batch, ksq_head, ksq_batch;
    uint32_t vq_tl[2], vq_th[2]; // low / high bytes of the 8 positive fp16 levels (turbo.cuh)
    float inv_sqrt_d;
    // attention mask (null: causal): byte (b, head or 0, row r, position t),
    // nonzero = attend; replaces the causal rule; positions >= mask_len unread
    const uint8_t *mask;
    int mask_heads, mask_len;
    long long mask_row, mask_head, mask_batch;
    // the layer's count of attention CTAs started (each takes the next work slot)
    unsigned long long *slot_ctr;
};

#ifdef __CUDACC__
__device__ __forceinline__ unsigned arg_fold(const AttnArgs &a)
{
    unsigned h = arg_fold(a.qn, a.gate, a.cache_pos, a.B, a.R, a.H, a.Hk, a.d, a.cap, a.nrb, a.nrb_u,
                          a.scale_log2, a.min_units, a.split, a.max_chunks, a.attn_grid, a.merge_rows, a.ws,
                          a.x16, a.xsum, a.NT,
                          a.group_o, a.tap_attn, a.status, a.vq, a.vq_codes, a.vq_scales,
                          a.cq_head, a.cq_batch, a.sq_head, a.sq_batch, a.kq_codes, a.kq_scales,
                          a.kcq_head, a.kcq_batch, a.ksq_head, a.ksq_batch, a.vq_tl[0], a.vq_tl[1],
                          a.vq_th[0], a.vq_th[1], a.inv_sqrt_d, a.mask, a.mask_heads, a.mask_len,
                          a.mask_row, a.mask_head, a.mask_batch, a.slot_ctr);
#pragma unroll
    for (int i = 0; i < kMaxRowBlocks; i += 4)
        h ^= arg_fold(a.rb_h0[i], a.rb_nh[i]);
    return h;
}
#endif

cudaError_t launch_attn(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap,
                        const CUtensorMap &vmap, int grid, bool pdl, cudaStream_t s);
// the merge launch after every attention launch (segments = B * Hk * nrb);
// vq: the cache format of the attention instance (0, 1, 2)
cudaError_t launch_attn_merge(int DB, int vq, const AttnArgs &a, int segments, bool pdl,
                              cudaStream_t s);
// the Bf16KTurbo4V instances (attn_vq.cu); vmap is unused there
cudaError_t launch_attn_vq(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap, int grid,
                           bool pdl, cudaStream_t s);
int attn_vq_smem_bytes(int MT, int DB);
cudaError_t attn_vq_set_smem_limits();
// the symmetric Turbo4 instances (attn_vqk.cu); no tensor map is read there
cudaError_t launch_attn_vqk(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap, int grid,
                            bool pdl, cudaStream_t s);
cudaError_t attn_vqk_set_smem_limits();
// standalone Turbo4 quantizer: one warp per row of d bf16 values
cudaError_t launch_turbo4_quantize(const uint16_t *v, long long rows, int d, uint8_t *codes,
                                   uint8_t *scales, const TurboTables &t, cudaStream_t s);
int attn_smem_bytes(int MT, int DB);
cudaError_t attn_set_smem_limits();

}  // namespace gattn

// records the thread-local message returned by gattn_last_error()
void gattn_set_error(const char *msg);
