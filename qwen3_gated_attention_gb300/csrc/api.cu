// api.cu -- host side of the C ABI declared in include/gattn.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "gattn.h"
#include "common.cuh"
#include "kernels.cuh"

using namespace gattn;

namespace {

thread_local std::string g_err;

gattn_status fail(gattn_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
gattn_status fail(gattn_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

#define CUDA_TRY(expr)                                                                             \
    do {                                                                                           \
        cudaError_t e_ = (expr);                                                                   \
        if (e_ != cudaSuccess)                                                                     \
            return fail(GATTN_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));             \
    } while (0)

constexpr int kMaxHidden = 16384;   // hidden and num_heads*head_dim

bool bits_ok(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }
bool group_ok(int g) { return g == 32 || g == 64 || g == 128; }

int proj_bits(const gattn_cfg &c, int p) { return c.proj_bits[p] ? c.proj_bits[p] : c.bits; }
int proj_group(const gattn_cfg &c, int p) { return c.proj_group[p] ? c.proj_group[p] : c.group_size; }

int rotary_dims(const gattn_cfg &c)
{
    return (int)((double)c.head_dim * (double)c.partial_rotary_factor);
}

gattn_status validate(const gattn_cfg *c)
{
    if (!c)
        return fail(GATTN_E_INVALID_ARG, "cfg is NULL");
    if (c->hidden <= 0 || c->num_heads <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
        return fail(GATTN_E_INVALID_ARG, "hidden, num_heads, num_kv_heads, head_dim must be > 0");
    if (c->num_heads % c->num_kv_heads)
        return fail(GATTN_E_INVALID_ARG, "num_heads %% num_kv_heads != 0");
    if (!(c->partial_rotary_factor > 0.f && c->partial_rotary_factor <= 1.f))
        return fail(GATTN_E_INVALID_ARG, "partial_rotary_factor must be in (0, 1]");
    const int rd = rotary_dims(*c);
    if (rd < 2 || (rd & 1))
        return fail(GATTN_E_INVALID_ARG, "rotary dims %d must be even and >= 2", rd);
    if (!(c->rope_theta > 0.f) || !(c->rms_eps >= 0.f))
        return fail(GATTN_E_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");
    if (c->x_dtype != GATTN_DTYPE_F32 && c->x_dtype != GATTN_DTYPE_BF16)
        return fail(GATTN_E_INVALID_ARG, "x_dtype must be GATTN_DTYPE_F32 or GATTN_DTYPE_BF16");
    for (int p = 0; p < 4; ++p) {
        if (c->proj_bits[p] < 0 || c->proj_group[p] < 0)
            return fail(GATTN_E_INVALID_ARG, "proj_bits/proj_group must be >= 0");
        if (!bits_ok(proj_bits(*c, p)))
            return fail(GATTN_E_INVALID_ARG, "bits %d of projection %d not in {2,3,4,5,6,8}",
                        proj_bits(*c, p), p);
        if (!group_ok(proj_group(*c, p)))
            return fail(GATTN_E_INVALID_ARG, "group %d of projection %d not in {32,64,128}",
                        proj_group(*c, p), p);
    }
    if (c->max_batch <= 0 || c->max_q_len <= 0)
        return fail(GATTN_E_INVALID_ARG, "max_batch and max_q_len must be > 0");
    if (c->head_chunk != 0 && c->head_chunk != 1)
        return fail(GATTN_E_INVALID_ARG, "head_chunk must be 0 or 1");
    // shapes this library implements
    if (c->head_dim % 64 || c->head_dim > 256)
        return fail(GATTN_E_UNSUPPORTED, "head_dim %d: this library needs a multiple of 64 <= 256",
                    c->head_dim);
    if (c->hidden % 128)
        return fail(GATTN_E_UNSUPPORTED, "hidden %d must be a multiple of 128", c->hidden);
    // sizes whose weight tiles, scratch and row counts stay within the kernels'
    // 32-bit indexes (checked before any product of two fields is formed)
    if (c->hidden > kMaxHidden || c->num_heads > kMaxHidden / 64 ||
        c->num_heads * c->head_dim > kMaxHidden)
        return fail(GATTN_E_UNSUPPORTED, "hidden and num_heads*head_dim must be <= %d", kMaxHidden);
    if ((c->num_heads * c->head_dim) % 128)
        return fail(GATTN_E_UNSUPPORTED, "num_heads*head_dim must be a multiple of 128");
    if (proj_bits(*c, 0) != proj_bits(*c, 1) || proj_bits(*c, 0) != proj_bits(*c, 2) ||
        proj_group(*c, 0) != proj_group(*c, 1) || proj_group(*c, 0) != proj_group(*c, 2))
        return fail(GATTN_E_UNSUPPORTED, "q, k and v must share bits and group (one fused launch)");
    if (proj_group(*c, 3) > c->head_dim)
        return fail(GATTN_E_UNSUPPORTED, "o_proj group must not exceed head_dim");
    if (c->max_batch > 32 || c->max_q_len > 32 ||
        c->max_batch * c->max_q_len > (c->x_dtype == GATTN_DTYPE_F32 ? 16 : 32))
        return fail(GATTN_E_UNSUPPORTED,
                    "max_batch, max_q_len and their product must be <= 32 (product <= 16 for fp32 x, "
                    "which takes two fp16 planes)");
    const int gqa = c->num_heads / c->num_kv_heads;
    if (gqa > kRowBlockRows * kMaxRowBlocks)
        return fail(GATTN_E_UNSUPPORTED, "gqa too large");
    return GATTN_OK;
}

struct ProjPlan {
    int N = 0, K = 0, bits = 0, group = 0, nrb = 0, nku = 0, ubytes = 0, step_bytes = 0;
    int rbc = 1;                              // row blocks per cluster (whole heads for q|k|v)
    int stage_bytes[3] = {0, 0, 0}, stages[3] = {0, 0, 0};  // per NT index
    int ks[3] = {1, 1, 1}, grid[3] = {0, 0, 0};
    int xtab[3] = {0, 0, 0};                  // q|k|v: bytes of the converted-x table (0: none)
    uint8_t *w = nullptr;
};

int nt_index(int NT) { return NT == 1 ? 0 : (NT == 2 ? 1 : 2); }

// Attention row blocks of a KV group for q_len rows: the head chunks of the
// verify plan (enabled or not), each cut into blocks of whole heads of at most
// kRowBlockRows rows (one head when q_len is larger).  Writes up to kMaxRowBlocks (first head, heads) pairs when the
// arrays are given; returns the block count (-1 past kMaxRowBlocks) and the
// largest block's rows.
int attn_row_blocks(int q_len, int H, int Hk, int enabled, int *rb_h0, int *rb_nh, int *max_rows)
{
    int32_t first[kMaxRowBlocks * 64], len[kMaxRowBlocks * 64];
    const int nchunks = gattn_head_chunk_plan(q_len, H, Hk, enabled, first, len, kMaxRowBlocks * 64);
    const int per_group = nchunks / Hk;
    int nrb = 0, mr = 0;
    for (int j = 0; j < per_group; ++j) {
        const int hpb = std::max(1, kRowBlockRows / q_len);
        for (int h = 0; h < len[j]; h += hpb) {
            if (nrb >= kMaxRowBlocks)
                return -1;
            if (rb_h0) {
                rb_h0[nrb] = first[j] + h;
                rb_nh[nrb] = std::min(hpb, len[j] - h);
            }
            mr = std::max(mr, std::min(hpb, len[j] - h) * q_len);
            ++nrb;
        }
    }
    if (max_rows)
        *max_rows = mr;
    return nrb;
}

constexpr int kAttnMinUnits = 4;     // 16-token units per attention chunk, at least
constexpr int kAttnSplit = 8;        // attention chunks per CTA aimed at
constexpr int kChunkRowsBudget = 512; // attention chunks x segment rows, at most

// Upper bound of the attention items (segment chunks) of a step: the chunk
// length is at least the unchunked partition's units over split x grid, so the
// items are at most split * grid * nrb / nrb_u plus one partial chunk per
// segment; and a segment has at most kMaxChunks (32) chunks.
long long attn_items_bound(int grid, int split, int nrb, int nrb_u, int batch, int Hk)
{
    const long long segs = (long long)batch * Hk * nrb;
    return std::min(((long long)split * grid * nrb + nrb_u - 1) / nrb_u + segs, 32 * segs);
}

// shared memory a q|k|v CTA may spend on converting x itself (the table of its
// k units' fp16 fragments and group sums); a larger table keeps the x prep kernel
constexpr int kXTabMax = 24 * 1024;
constexpr int kMaxCluster = 8;       // portable cluster size

void plan_proj(ProjPlan &p, int N, int K, int bits, int group, int rbc, int mode)
{
    p.N = N;
    p.K = K;
    p.bits = bits;
    p.group = group;
    p.rbc = rbc;
    p.nrb = (N + kRBR - 1) / kRBR;
    p.nrb = (p.nrb + rbc - 1) / rbc * rbc;    // whole clusters (padding rows are zero)
    p.nku = K / kKU;
    p.ubytes = unit_bytes(bits, group);
    p.step_bytes = kWR * p.ubytes;
    for (int i = 0; i < 3; ++i) {
        const int NT = 1 << i;
        const int xb = 2048 * NT, sb = (kKU / group) * 32 * NT;
        int sbytes = p.step_bytes + xb + sb;
        sbytes = (sbytes + 127) & ~127;
        p.stage_bytes[i] = sbytes;
        // a small ring per CTA so that three or four CTAs (12-16 consumer warps)
        // share an SM: the stage loop is latency bound, not bandwidth bound.
        // o_proj at 32 operand columns takes a ring twice as deep (its CTAs
        // stream only a few stages each, measured faster at batched_9b)
        int st = ((mode == kModeO && NT >= 4 ? 96 : 48) * 1024) / sbytes;
        if (st < 2) st = 2;
        if (st > 8) st = 8;
        // the drained ring holds the CTA's partial sums [8*NT][kRBR] floats
        while (st * sbytes < 8 * NT * kRBR * 4 && st < 8)
            ++st;
        p.stages[i] = st;
    }
}

}  // namespace

struct gattn_layer {
    gattn_cfg cfg{};
    int rd = 0, gqa = 0, Nq = 0, Nkv = 0, Ko = 0;
    int device = 0, num_sms = 0;
    ProjPlan pqkv, po;
    int M_max = 0;
    // scratch
    __half *x16_a = nullptr, *x16_o = nullptr;
    float *xsum_a = nullptr, *xsum_o = nullptr;
    __nv_bfloat16 *qn = nullptr;
    float *gate = nullptr;
    float *ws_attn = nullptr;              // attention chunk partials
    long long items_cap = 0;
    unsigned *status = nullptr;
    double *inv_freq = nullptr;
    float2 *inv_freq2 = nullptr;           // the same frequencies as float (hi, lo) pairs
    uint16_t *q_norm = nullptr, *k_norm = nullptr;
    size_t ws_attn_floats = 0;
    int attn_grid = 0;
    int max_seg = 0;
    float *ss_part = nullptr;              // decoder-block post-norm: per-CTA sums of squares
    unsigned *post_ticket = nullptr;
    unsigned long long *slot_ctr = nullptr;   // attention CTAs started (work slots, attn.cuh)
    // gattn_layer_step_host: device copies of the step's x and cache_pos (two
    // slots, filled on copy_stream while the previous step runs) and of out
    void *x_stage[2] = {nullptr, nullptr}, *out_stage = nullptr;
    int32_t *pos_stage[2] = {nullptr, nullptr};
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t stage_in[2] = {nullptr, nullptr};     // a slot's copies have landed
    cudaEvent_t stage_free[2] = {nullptr, nullptr};   // the step that read a slot is done
    int stage_slot = 0;
    // Bf16KTurbo4V caches: decision tables (passed by value) and the bytes of
    // the 8 positive fp16 levels the attention dequantizes with
    TurboTables tq{};
    uint32_t tq_tl[2] = {0, 0}, tq_th[2] = {0, 0};
    gattn_taps taps{};
    gattn_mask mask{};                     // attention mask of the following steps (mask.mask null: causal)
    bool weights_set = false;
    int launches = 0;
    int32_t kinds[8] = {0};                // GATTN_KERNEL_* of the last step's launches
    bool pdl = true;
    std::vector<cudaEvent_t> events;
    unsigned long long wait_ns = kWaitLimitNs;   // bound of the projection kernels' waits
    int withhold = 0;                             // failure test hook (see gattn_layer_set_test_wait)
};

struct gattn_kv {
    gattn_layer *layer = nullptr;
    gattn_kv_desc desc{};          // K (and V for a bf16 cache); v is NULL for Turbo4 V
    bool turbo = false;            // Bf16KTurbo4V: V as codes + E4M3 scales
    gattn_kv_turbo4v_desc tdesc{};
    bool kturbo = false;           // symmetric Turbo4: K as codes + E4M3 scales too
    void *kq_codes = nullptr, *kq_scales = nullptr;
    CUtensorMap kmap;   // CUtensorMap is itself 64-byte aligned
    CUtensorMap vmap;
};

bool gattn::layer_proj_tiles(const gattn_layer *L, int proj, ProjTiles *out)
{
    if (!L || !out || proj < 0 || proj > 3 || !L->weights_set)
        return false;
    const ProjPlan &p = proj == 3 ? L->po : L->pqkv;
    out->w = p.w;
    out->nku = p.nku;
    out->bits = p.bits;
    out->group = p.group;
    out->step_bytes = p.step_bytes;
    out->K = p.K;
    out->row0 = proj == 0 ? 0 : (proj == 1 ? L->Nq : (proj == 2 ? L->Nq + L->Nkv : 0));
    out->rows = proj == 0 ? L->Nq : (proj == 3 ? L->po.N : L->Nkv);
    return true;
}

void gattn_set_error(const char *msg) { g_err = msg; }

extern "C" {

const char *gattn_last_error(void) { return g_err.c_str(); }

gattn_status gattn_cfg_validate(const gattn_cfg *cfg) { return validate(cfg); }

int32_t gattn_rotary_dims(const gattn_cfg *cfg) { return cfg ? rotary_dims(*cfg) : -1; }

int32_t gattn_head_chunk_plan(int32_t q_len, int32_t num_heads, int32_t num_kv_heads,
                              int32_t enabled, int32_t *first, int32_t *len, int32_t cap)
{
    if (q_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || cap < 0 ||
        (cap > 0 && (!first || !len)))
        return -1;
    const int gqa = num_heads / num_kv_heads;
    // eligible: more than 32 (row, head) pairs per KV group and at most 32 rows
    const bool eligible = enabled && q_len <= 32 && (long long)q_len * gqa > 32;
    int per = gqa;
    if (eligible) {
        per = 32 / q_len;
        per = per < gqa ? per : gqa;
        per = per > 1 ? per : 1;
    }
    const int per_group = (gqa + per - 1) / per;
    const int count = num_kv_heads * per_group;
    int n = 0;
    for (int g = 0; g < num_kv_heads; ++g)
        for (int j = 0; j < per_group; ++j, ++n)
            if (n < cap) {
                first[n] = g * gqa + j * per;
                len[n] = (j == per_group - 1) ? gqa - j * per : per;
            }
    return count;
}

gattn_status gattn_layer_create(const gattn_cfg *cfg, gattn_layer **out)
{
    if (!out)
        return fail(GATTN_E_INVALID_ARG, "out is NULL");
    *out = nullptr;
    gattn_status st = validate(cfg);
    if (st != GATTN_OK)
        return st;
    gattn_layer *L = new (std::nothrow) gattn_layer();
    if (!L)
        return fail(GATTN_E_CUDA, "out of host memory");
    L->cfg = *cfg;
    const gattn_cfg &c = L->cfg;
    L->rd = rotary_dims(c);
    L->gqa = c.num_heads / c.num_kv_heads;
    L->Nq = 2 * c.num_heads * c.head_dim;
    L->Nkv = c.num_kv_heads * c.head_dim;
    L->Ko = c.num_heads * c.head_dim;
    L->M_max = c.max_batch * c.max_q_len;
    auto cleanup = [&](gattn_status s) {
        gattn_layer_destroy(L);
        return s;
    };
#define TRY(expr)                                                                                  \
    do {                                                                                           \
        cudaError_t e_ = (expr);                                                                   \
        if (e_ != cudaSuccess)                                                                     \
            return cleanup(fail(GATTN_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)));   \
    } while (0)
    TRY(cudaGetDevice(&L->device));
    TRY(cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device));

    // a q|k|v cluster covers whole heads (RMSNorm needs every row of a head)
    plan_proj(L->pqkv, L->Nq + 2 * L->Nkv, c.hidden, proj_bits(c, 0), proj_group(c, 0),
              std::max(1, c.head_dim / kRBR), kModeQKV);
    plan_proj(L->po, c.hidden, L->Ko, proj_bits(c, 3), proj_group(c, 3), 1, kModeO);

    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        cudaError_t e = attn_set_smem_limits();
        for (int b : {2, 3, 4, 5, 6, 8})
            for (int NT : {1, 2, 4})
                for (int mode : {kModeQKV, kModeO})
                    if (e == cudaSuccess)
                        e = proj_set_smem_limits(b, NT, mode, 200 * 1024);
        attr_err = e;
    });
    TRY(attr_err);
    for (ProjPlan *p : {&L->pqkv, &L->po}) {
        const int mode = p == &L->pqkv ? kModeQKV : kModeO;
        for (int i = 0; i < 3; ++i) {
            const int NT = 1 << i;
            ProjArgs a{};
            a.stages = p->stages[i];
            a.stage_bytes = p->stage_bytes[i];
            a.eb_rows = p->rbc * kRBR;
            a.recv_cap = proj_recv_cap(mode, NT);
            const int smem = proj_smem_bytes(a);
            const int nclusters = p->nrb / p->rbc;
            // 16-CTA clusters (non-portable) when this kernel can run them
            // (the q|k|v projection, which attention waits on, keeps the portable
            // size: a cluster larger than 8 can wait several microseconds for a GPC
            // with room for all of its CTAs)
            int max_cluster = kMaxCluster, n16 = 0;
            if (p == &L->po &&
                proj_max_clusters(p->bits, NT, kModeO, p->group, smem, 16, &n16) == cudaSuccess &&
                n16 > 0)
                max_cluster = 16;
            cudaGetLastError();
            // q|k|v with at most 16 operand columns: each CTA converts the x of its
            // own k units when that table is small (no separate x prep launch)
            auto xtab_for = [&](int ks) -> int {
                if (mode != kModeQKV || NT > 2)
                    return 0;
                const int xe = 2048 * NT + (kKU / p->group) * 4 * 8 * NT;
                const int xt = (p->nku + ks - 1) / ks * xe;
                return xt <= kXTabMax ? xt : 0;
            };
            // the largest k split (any count up to the cluster limit) whose
            // clusters all fit on the GPU at once: one wave (a second, partial
            // wave of clusters costs more than the split saves)
            int ks = 1;
            for (int cand = std::min(max_cluster / p->rbc, p->nku); cand > 1; --cand) {
                const int csize = cand * p->rbc;
                const int sm_c = smem + xtab_for(cand);
                int occ = 0;
                TRY(proj_occupancy(p->bits, NT, mode, p->group, sm_c, &occ));
                if (occ < 1)
                    occ = 1;
                if ((long long)nclusters * csize > (long long)L->num_sms * occ)
                    continue;
                int nres = 0;
                if (proj_max_clusters(p->bits, NT, mode, p->group, sm_c, csize, &nres) !=
                    cudaSuccess) {
                    cudaGetLastError();
                    continue;
                }
                if (nres >= nclusters) {
                    ks = cand;
                    break;
                }
            }
            p->ks[i] = ks;
            p->xtab[i] = xtab_for(ks);
            p->grid[i] = nclusters * p->rbc * ks;
        }
    }
    // one attention CTA per SM; a segment's contributors (at most the grid)
    // fit the merge's factor table of 160
    L->attn_grid = std::min(L->num_sms, 159);

    const int MP = 32;  // columns of the widest (NT = 4) operand layout
    const size_t nku_a = c.hidden / kKU, nku_o = L->Ko / kKU;
    TRY(cudaMalloc(&L->pqkv.w, (size_t)L->pqkv.nrb * L->pqkv.nku * L->pqkv.step_bytes));
    TRY(cudaMalloc(&L->po.w, (size_t)L->po.nrb * L->po.nku * L->po.step_bytes));
    TRY(cudaMalloc(&L->x16_a, nku_a * 4 * 2048));
    TRY(cudaMalloc(&L->x16_o, nku_o * 4 * 2048));
    TRY(cudaMemset(L->x16_o, 0, nku_o * 4 * 2048));
    TRY(cudaMalloc(&L->xsum_a, nku_a * (kKU / L->pqkv.group) * MP * sizeof(float)));
    TRY(cudaMalloc(&L->xsum_o, nku_o * (kKU / L->po.group) * MP * sizeof(float)));
    TRY(cudaMemset(L->xsum_o, 0, nku_o * (kKU / L->po.group) * MP * sizeof(float)));
    TRY(cudaMalloc(&L->qn, (size_t)L->M_max * L->Ko * 2));
    for (int i = 0; i < 2; ++i) {
        TRY(cudaMalloc(&L->x_stage[i], (size_t)L->M_max * c.hidden *
                                           (c.x_dtype == GATTN_DTYPE_F32 ? 4 : 2)));
        TRY(cudaMalloc(&L->pos_stage[i], (size_t)c.max_batch * sizeof(int32_t)));
        TRY(cudaEventCreateWithFlags(&L->stage_in[i], cudaEventDisableTiming));
        TRY(cudaEventCreateWithFlags(&L->stage_free[i], cudaEventDisableTiming));
    }
    TRY(cudaMalloc(&L->out_stage, (size_t)L->M_max * c.hidden * 2));
    TRY(cudaStreamCreateWithFlags(&L->copy_stream, cudaStreamNonBlocking));
    TRY(cudaMalloc(&L->gate, (size_t)L->M_max * L->Ko * sizeof(float)));
    // attention segments: batch x KV heads x row blocks (at most gqa row blocks)
    // attention scratch: chunk partials and completion counters for the largest
    // step the configuration admits (every q_len, both head partitions)
    {
        int nrb_max = 1;
        for (int R = 1; R <= c.max_q_len; ++R) {
            const int nrb = attn_row_blocks(R, c.num_heads, c.num_kv_heads, c.head_chunk, nullptr,
                                            nullptr, nullptr);
            const int nrb_u = attn_row_blocks(R, c.num_heads, c.num_kv_heads, 0, nullptr, nullptr,
                                              nullptr);
            if (nrb < 0 || nrb_u < 0)
                return cleanup(fail(GATTN_E_UNSUPPORTED, "too many attention row blocks"));
            nrb_max = std::max(nrb_max, std::max(nrb, nrb_u));
            L->items_cap = std::max(L->items_cap, attn_items_bound(L->attn_grid, kAttnSplit, nrb, nrb_u,
                                                                   c.max_batch, c.num_kv_heads));
        }
        L->max_seg = c.max_batch * c.num_kv_heads * nrb_max;
    }
    L->ws_attn_floats = (size_t)L->items_cap * attn_slot_floats(c.head_dim);
    TRY(cudaMalloc(&L->ws_attn, L->ws_attn_floats * sizeof(float)));
    TRY(cudaMalloc(&L->status, sizeof(unsigned)));
    TRY(cudaMemset(L->status, 0, sizeof(unsigned)));
    {
        float lv[16], th[15];
        gattn_turbo4_codebook(lv, th);
        std::memcpy(L->tq.lv, lv, sizeof lv);
        std::memcpy(L->tq.th, th, sizeof th);
        L->tq.inv_sqrt_d = (float)(1.0 / std::sqrt((double)c.head_dim));
        for (int m = 0; m < 8; ++m) {
            const __half h = __float2half_rn(lv[8 + m]);
            uint16_t h16;
            std::memcpy(&h16, &h, 2);
            L->tq_tl[m >> 2] |= (uint32_t)(h16 & 0xFF) << (8 * (m & 3));
            L->tq_th[m >> 2] |= (uint32_t)(h16 >> 8) << (8 * (m & 3));
        }
    }
    {
        const int gmax = *std::max_element(L->po.grid, L->po.grid + 3);
        TRY(cudaMalloc(&L->ss_part, (size_t)gmax * L->M_max * sizeof(float)));
        TRY(cudaMalloc(&L->post_ticket, sizeof(unsigned)));
        TRY(cudaMemset(L->post_ticket, 0, sizeof(unsigned)));
        TRY(cudaMalloc(&L->slot_ctr, sizeof(unsigned long long)));
        TRY(cudaMemset(L->slot_ctr, 0, sizeof(unsigned long long)));
    }

    std::vector<double> inv(L->rd / 2);
    for (int i = 0; i < L->rd / 2; ++i)
        inv[i] = std::pow((double)c.rope_theta, -2.0 * (double)i / (double)L->rd);
    TRY(cudaMalloc(&L->inv_freq, inv.size() * sizeof(double)));
    TRY(cudaMemcpy(L->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice));
    {
        std::vector<float2> pairs(inv.size());
        for (size_t i = 0; i < inv.size(); ++i) {
            pairs[i].x = (float)inv[i];
            pairs[i].y = (float)(inv[i] - (double)pairs[i].x);
        }
        TRY(cudaMalloc(&L->inv_freq2, pairs.size() * sizeof(float2)));
        TRY(cudaMemcpy(L->inv_freq2, pairs.data(), pairs.size() * sizeof(float2),
                       cudaMemcpyHostToDevice));
    }
    TRY(cudaMalloc(&L->q_norm, c.head_dim * 2));
    TRY(cudaMalloc(&L->k_norm, c.head_dim * 2));
#undef TRY
    *out = L;
    return GATTN_OK;
}

void gattn_layer_destroy(gattn_layer *L)
{
    if (!L)
        return;
    void *ptrs[] = {L->pqkv.w, L->po.w,      L->x16_a,  L->x16_o,   L->xsum_a,  L->xsum_o,
                    L->qn,     L->gate,      L->ws_attn, L->status,  L->inv_freq, L->inv_freq2,
                    L->q_norm, L->k_norm,
                    L->ss_part, L->post_ticket, L->slot_ctr,
                    L->x_stage[0], L->x_stage[1], L->out_stage, L->pos_stage[0],
                    L->pos_stage[1]};
    for (void *p : ptrs)
        if (p)
            cudaFree(p);
    for (int i = 0; i < 2; ++i) {
        if (L->stage_in[i])
            cudaEventDestroy(L->stage_in[i]);
        if (L->stage_free[i])
            cudaEventDestroy(L->stage_free[i]);
    }
    if (L->copy_stream)
        cudaStreamDestroy(L->copy_stream);
    delete L;
}

gattn_status gattn_layer_set_weights(gattn_layer *L, const gattn_weights *w, gattn_stream stream)
{
    if (!L || !w)
        return fail(GATTN_E_INVALID_ARG, "layer or weights is NULL");
    for (int p = 0; p < 4; ++p)
        if (!w->proj[p].packed || !w->proj[p].scales || !w->proj[p].biases)
            return fail(GATTN_E_INVALID_ARG, "projection %d has a NULL buffer", p);
    if (!w->q_norm || !w->k_norm)
        return fail(GATTN_E_INVALID_ARG, "q_norm/k_norm is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    RepackSrc a{};
    a.nsrc = 3;
    const int rows[3] = {L->Nq, L->Nkv, L->Nkv};
    for (int i = 0; i < 3; ++i) {
        a.packed[i] = w->proj[i].packed;
        a.scales[i] = w->proj[i].scales;
        a.biases[i] = w->proj[i].biases;
        a.rows[i] = rows[i];
    }
    CUDA_TRY(launch_repack(a, L->pqkv.K, L->pqkv.bits, L->pqkv.group, L->pqkv.nrb, L->pqkv.w, s));
    RepackSrc o{};
    o.nsrc = 1;
    o.packed[0] = w->proj[3].packed;
    o.scales[0] = w->proj[3].scales;
    o.biases[0] = w->proj[3].biases;
    o.rows[0] = L->po.N;
    CUDA_TRY(launch_repack(o, L->po.K, L->po.bits, L->po.group, L->po.nrb, L->po.w, s));
    CUDA_TRY(cudaMemcpyAsync(L->q_norm, w->q_norm, L->cfg.head_dim * 2, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(L->k_norm, w->k_norm, L->cfg.head_dim * 2, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    L->weights_set = true;
    return GATTN_OK;
}

gattn_status gattn_kv_register(gattn_layer *L, const gattn_kv_desc *d, gattn_kv **out)
{
    if (!L || !d || !out)
        return fail(GATTN_E_INVALID_ARG, "NULL argument");
    *out = nullptr;
    if (!d->k || !d->v)
        return fail(GATTN_E_INVALID_ARG, "cache pointers are NULL");
    if ((reinterpret_cast<uintptr_t>(d->k) | reinterpret_cast<uintptr_t>(d->v)) & 15)
        return fail(GATTN_E_INVALID_ARG, "cache pointers must be 16-byte aligned");
    if (d->batch <= 0 || d->capacity < 16)
        return fail(GATTN_E_INVALID_ARG, "batch must be > 0 and capacity >= 16");
    if (d->stride_token <= 0 || d->stride_head <= 0 || d->stride_batch <= 0 ||
        (d->stride_token | d->stride_head | d->stride_batch) & 7)
        return fail(GATTN_E_INVALID_ARG, "strides must be positive multiples of 8 elements");
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        CUDA_TRY(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                  cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !fn)
            return fail(GATTN_E_CUDA, "cuTensorMapEncodeTiled is not available");
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    gattn_kv *kv = new (std::nothrow) gattn_kv();
    if (!kv)
        return fail(GATTN_E_CUDA, "out of host memory");
    kv->layer = L;
    kv->desc = *d;
    const cuuint64_t dims[4] = {(cuuint64_t)L->cfg.head_dim, (cuuint64_t)d->capacity,
                                (cuuint64_t)L->cfg.num_kv_heads, (cuuint64_t)d->batch};
    const cuuint64_t strides[3] = {(cuuint64_t)d->stride_token * 2, (cuuint64_t)d->stride_head * 2,
                                   (cuuint64_t)d->stride_batch * 2};
    const cuuint32_t box[4] = {64, kAttnUnit, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    for (int i = 0; i < 2; ++i) {
        CUresult r = encode(i == 0 ? &kv->kmap : &kv->vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                            i == 0 ? d->k : d->v, dims, strides, box, es,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            delete kv;
            return fail(GATTN_E_INVALID_ARG, "cuTensorMapEncodeTiled rejected the cache (code %d)",
                        (int)r);
        }
    }
    *out = kv;
    return GATTN_OK;
}

// Rules for the Turbo4 code / scale planes of a cache (V, and K for the
// symmetric format): pointers, capacity, strides.
static gattn_status check_turbo_planes(const gattn_layer *L, const char *which, const void *codes,
                                       const void *scales, int32_t capacity, int64_t cs_head,
                                       int64_t cs_batch, int64_t ss_head, int64_t ss_batch)
{
    const int hd = L->cfg.head_dim;
    if (hd != 64 && hd != 128 && hd != 256)
        return fail(GATTN_E_INVALID_ARG, "a Turbo4 cache needs head_dim 64, 128 or 256 (got %d)", hd);
    if (!codes || !scales)
        return fail(GATTN_E_INVALID_ARG, "%s code or scale pointer is NULL", which);
    if ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(scales)) & 15)
        return fail(GATTN_E_INVALID_ARG, "%s code and scale pointers must be 16-byte aligned", which);
    if (capacity < 16 || capacity % 16)
        return fail(GATTN_E_INVALID_ARG, "a Turbo4 cache needs capacity %% 16 == 0 (got %d)",
                    (int)capacity);
    const long long cap = capacity;
    if (cs_head <= 0 || cs_batch <= 0 || ss_head <= 0 || ss_batch <= 0 ||
        (cs_head | cs_batch | ss_head | ss_batch) & 15)
        return fail(GATTN_E_INVALID_ARG, "code and scale strides must be positive multiples of 16 bytes");
    if (cs_head < cap * (hd / 2) || ss_head < cap * (hd / 16))
        return fail(GATTN_E_INVALID_ARG, "a head's code or scale rows overlap the next head's");
    return GATTN_OK;
}

gattn_status gattn_kv_register_turbo4v(gattn_layer *L, const gattn_kv_turbo4v_desc *d,
                                       gattn_kv **out)
{
    if (!L || !d || !out)
        return fail(GATTN_E_INVALID_ARG, "NULL argument");
    *out = nullptr;
    const gattn_status pst = check_turbo_planes(L, "V", d->v_codes, d->v_scales, d->capacity,
                                                d->code_stride_head, d->code_stride_batch,
                                                d->scale_stride_head, d->scale_stride_batch);
    if (pst != GATTN_OK)
        return pst;
    gattn_kv_desc kd{};
    kd.k = d->k;
    kd.v = d->k;                // checked like a bf16 V pointer, never read as V
    kd.batch = d->batch;
    kd.capacity = d->capacity;
    kd.stride_token = d->k_stride_token;
    kd.stride_head = d->k_stride_head;
    kd.stride_batch = d->k_stride_batch;
    gattn_kv *kv = nullptr;
    const gattn_status st = gattn_kv_register(L, &kd, &kv);
    if (st != GATTN_OK)
        return st;
    kv->desc.v = nullptr;
    kv->turbo = true;
    kv->tdesc = *d;
    *out = kv;
    return GATTN_OK;
}

gattn_status gattn_kv_register_turbo4(gattn_layer *L, const gattn_kv_turbo4_desc *d,
                                      gattn_kv **out)
{
    if (!L || !d || !out)
        return fail(GATTN_E_INVALID_ARG, "NULL argument");
    *out = nullptr;
    if (d->batch <= 0)
        return fail(GATTN_E_INVALID_ARG, "batch must be > 0");
    for (int side = 0; side < 2; ++side) {
        const gattn_status st = check_turbo_planes(
            L, side ? "V" : "K", side ? d->v_codes : d->k_codes, side ? d->v_scales : d->k_scales,
            d->capacity, d->code_stride_head, d->code_stride_batch, d->scale_stride_head,
            d->scale_stride_batch);
        if (st != GATTN_OK)
            return st;
    }
    gattn_kv *kv = new (std::nothrow) gattn_kv();
    if (!kv)
        return fail(GATTN_E_CUDA, "out of host memory");
    kv->layer = L;
    kv->desc.batch = d->batch;           // no bf16 planes: no tensor maps either
    kv->desc.capacity = d->capacity;
    std::memset(&kv->kmap, 0, sizeof(kv->kmap));
    std::memset(&kv->vmap, 0, sizeof(kv->vmap));
    kv->turbo = true;
    kv->tdesc.v_codes = d->v_codes;
    kv->tdesc.v_scales = d->v_scales;
    kv->tdesc.batch = d->batch;
    kv->tdesc.capacity = d->capacity;
    kv->tdesc.code_stride_head = d->code_stride_head;
    kv->tdesc.code_stride_batch = d->code_stride_batch;
    kv->tdesc.scale_stride_head = d->scale_stride_head;
    kv->tdesc.scale_stride_batch = d->scale_stride_batch;
    kv->kturbo = true;
    kv->kq_codes = d->k_codes;
    kv->kq_scales = d->k_scales;
    *out = kv;
    return GATTN_OK;
}

gattn_status gattn_turbo4_quantize_device(const void *v, int64_t rows, int32_t d, void *codes,
                                          void *scales, gattn_stream stream)
{
    if (rows < 0 || (rows > 0 && (!v || !codes || !scales)))
        return fail(GATTN_E_INVALID_ARG, "bad rows or NULL pointer");
    if (d != 64 && d != 128 && d != 256)
        return fail(GATTN_E_INVALID_ARG, "d must be 64, 128 or 256 (got %d)", (int)d);
    TurboTables t{};
    float lv[16], th[15];
    gattn_turbo4_codebook(lv, th);
    std::memcpy(t.lv, lv, sizeof lv);
    std::memcpy(t.th, th, sizeof th);
    t.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
    CUDA_TRY(launch_turbo4_quantize(static_cast<const uint16_t *>(v), rows, d,
                                    static_cast<uint8_t *>(codes), static_cast<uint8_t *>(scales), t,
                                    reinterpret_cast<cudaStream_t>(stream)));
    return GATTN_OK;
}

void gattn_kv_destroy(gattn_kv *kv) { delete kv; }

gattn_status gattn_layer_set_taps(gattn_layer *L, const gattn_taps *t)
{
    if (!L)
        return fail(GATTN_E_INVALID_ARG, "layer is NULL");
    L->taps = t ? *t : gattn_taps{};
    return GATTN_OK;
}

gattn_status gattn_layer_set_mask(gattn_layer *L, const gattn_mask *m)
{
    if (!L)
        return fail(GATTN_E_INVALID_ARG, "layer is NULL");
    if (!m || !m->mask) {
        L->mask = gattn_mask{};
        return GATTN_OK;
    }
    if (m->heads != 1 && m->heads != L->cfg.num_heads)
        return fail(GATTN_E_INVALID_ARG, "mask heads must be 1 or num_heads (%d), got %d",
                    (int)L->cfg.num_heads, (int)m->heads);
    if (m->positions <= 0 || m->stride_row < m->positions || m->stride_head < 0 ||
        m->stride_batch < 0)
        return fail(GATTN_E_INVALID_ARG, "bad mask row length or strides");
    L->mask = *m;
    return GATTN_OK;
}

int32_t gattn_layer_launches_per_step(const gattn_layer *L) { return L ? L->launches : -1; }

int32_t gattn_layer_step_kernels(const gattn_layer *L, int32_t *kinds, int32_t cap)
{
    if (!L || cap < 0 || (cap > 0 && !kinds))
        return -1;
    for (int i = 0; i < L->launches && i < cap; ++i)
        kinds[i] = L->kinds[i];
    return L->launches;
}


gattn_status gattn_layer_set_events(gattn_layer *L, void *const *events, int32_t n)
{
    if (!L || n < 0 || (n > 0 && !events))
        return fail(GATTN_E_INVALID_ARG, "bad event arguments");
    if (n == 1)
        return fail(GATTN_E_INVALID_ARG, "need at least 2 events (before and after a step)");
    L->events.assign(reinterpret_cast<cudaEvent_t const *>(events),
                     reinterpret_cast<cudaEvent_t const *>(events) + n);
    return GATTN_OK;
}

gattn_status gattn_layer_set_test_wait(gattn_layer *L, int64_t wait_limit_ns,
                                       int32_t withhold_stage)
{
    if (!L || wait_limit_ns < 0)
        return fail(GATTN_E_INVALID_ARG, "bad wait limit arguments");
    L->wait_ns = wait_limit_ns ? (unsigned long long)wait_limit_ns : kWaitLimitNs;
    L->withhold = withhold_stage ? 1 : 0;
    return GATTN_OK;
}

namespace {

// The decoder block around the layer (gattn_layer_step_block); null: the layer alone.
struct BlockArgs {
    const uint16_t *input_ln, *post_ln;
    __nv_bfloat16 *out_normed;
};

// The argument checks of a step (everything but the data pointers).
gattn_status check_step(const gattn_layer *L, const gattn_kv *kv, int32_t batch, int32_t q_len)
{
    if (!L->weights_set)
        return fail(GATTN_E_STATE, "set_weights has not been called");
    if (kv->layer != L)
        return fail(GATTN_E_INVALID_ARG, "cache registered with another layer");
    const gattn_cfg &c = L->cfg;
    if (batch <= 0 || batch > c.max_batch || batch > kv->desc.batch)
        return fail(GATTN_E_INVALID_ARG, "batch %d outside [1, min(max_batch %d, cache batch %d)]",
                    batch, c.max_batch, kv->desc.batch);
    if (q_len <= 0 || q_len > c.max_q_len)
        return fail(GATTN_E_INVALID_ARG, "q_len %d outside [1, %d]", q_len, c.max_q_len);
    return GATTN_OK;
}

gattn_status step_impl(gattn_layer *L, const void *x, gattn_kv *kv, const int32_t *cache_pos,
                       int32_t batch, int32_t q_len, void *out, gattn_stream stream,
                       const BlockArgs *blk)
{
    if (!L || !x || !kv || !cache_pos || !out)
        return fail(GATTN_E_INVALID_ARG, "NULL argument");
    const gattn_status chk = check_step(L, kv, batch, q_len);
    if (chk != GATTN_OK)
        return chk;
    const gattn_cfg &c = L->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int M = batch * q_len;
    // the q|k|v operand has 2M columns for fp32 x (exact hi + lo fp16 planes)
    const int Ma = c.x_dtype == GATTN_DTYPE_F32 ? 2 * M : M;
    const int NTa = Ma <= 8 ? 1 : (Ma <= 16 ? 2 : 4);
    const int NT = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
    const int nia = nt_index(NTa), ni = nt_index(NT);
    const bool timing = !L->events.empty();
    const bool pdl = L->pdl && !timing;
    const int nev = (int)L->events.size();
    int launches = 0;
    // events[i] before the i-th launch (i < n - 1), events[n - 1] after the last
    auto mark = [&](int i) -> cudaError_t {
        return timing && i < nev - 1 ? cudaEventRecord(L->events[i], s) : cudaSuccess;
    };
    auto mark_end = [&]() -> cudaError_t {
        return timing ? cudaEventRecord(L->events[nev - 1], s) : cudaSuccess;
    };

    // attention segments: per KV group the head chunks of the verify plan, a
    // chunk of more than 64 rows cut into row blocks of whole heads
    AttnArgs t{};
    int max_rows = 0;
    const int nrb = attn_row_blocks(q_len, c.num_heads, c.num_kv_heads, c.head_chunk, t.rb_h0,
                                    t.rb_nh, &max_rows);
    const int nrb_u = attn_row_blocks(q_len, c.num_heads, c.num_kv_heads, 0, nullptr, nullptr,
                                      nullptr);
    if (nrb < 0 || nrb_u < 0)
        return fail(GATTN_E_UNSUPPORTED, "too many attention row blocks");
    if ((long long)batch * c.num_kv_heads * nrb > L->max_seg ||
        attn_items_bound(L->attn_grid, kAttnSplit, nrb, nrb_u, batch, c.num_kv_heads) > L->items_cap)
        return fail(GATTN_E_UNSUPPORTED, "attention items exceed the scratch sized at create");
    const int nchunks = gattn_head_chunk_plan(q_len, c.num_heads, c.num_kv_heads, c.head_chunk,
                                              nullptr, nullptr, 0);
    const int MT = (max_rows + 15) / 16;
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));

    // the head-chunked verify route hands the mask unchanged to each head chunk:
    // a broadcast mask fits every chunk, a mask over all heads does not
    if (L->mask.mask && L->mask.heads > 1 && nchunks > c.num_kv_heads)
        return fail(GATTN_E_UNSUPPORTED,
                    "a head-specific mask cannot take the head-chunked verify route "
                    "(q_len %d, %d query heads per KV head)", (int)q_len, (int)L->gqa);

    int32_t kinds[8] = {0};
    auto launched = [&](int32_t kind) { kinds[launches++] = kind; };

    // 1. x -> fp16 tensor-core operand + group sums: in the q|k|v kernel itself
    //    when its CTAs' tables fit (layer steps; x 16-byte aligned), else its
    //    own launch
    const bool xfold = !blk && L->pqkv.xtab[nia] > 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    if (!xfold) {
        CUDA_TRY(mark(launches));
        CUDA_TRY(launch_xprep(x, c.x_dtype, M, c.hidden, L->pqkv.group, NTa, L->x16_a, L->xsum_a,
                              blk ? blk->input_ln : nullptr, c.rms_eps, pdl, s));
        launched(GATTN_KERNEL_XPREP);
    }

    // 2. fused q|k|v projection with the norm / rotary / append epilogue
    ProjArgs a{};
    a.w = L->pqkv.w;
    a.x16 = L->x16_a;
    a.xsum = L->xsum_a;
    a.nrb = L->pqkv.nrb;
    a.nku = L->pqkv.nku;
    a.N = L->pqkv.N;
    a.M = M;
    a.group = L->pqkv.group;
    a.unit_bytes = L->pqkv.ubytes;
    a.step_bytes = L->pqkv.step_bytes;
    a.stage_bytes = L->pqkv.stage_bytes[nia];
    a.stages = L->pqkv.stages[nia];
    a.rbc = L->pqkv.rbc;
    a.ks = L->pqkv.ks[nia];
    a.eb_rows = a.rbc * kRBR;
    a.recv_cap = proj_recv_cap(kModeQKV, NTa);
    a.xtab_bytes = xfold ? L->pqkv.xtab[nia] : 0;
    a.xraw = x;
    a.x_f32 = c.x_dtype == GATTN_DTYPE_F32;
    a.xsplit = c.x_dtype == GATTN_DTYPE_F32 ? M : 0;
    a.status = L->status;
    a.wait_ns = L->wait_ns;
    a.withhold = L->withhold;
    EpiQKV eq{};
    eq.R = q_len;
    eq.H = c.num_heads;
    eq.Hk = c.num_kv_heads;
    eq.d = c.head_dim;
    eq.rd = L->rd;
    eq.Nq = L->Nq;
    eq.Nkv = L->Nkv;
    eq.cache_pos = cache_pos;
    eq.cap = kv->desc.capacity;
    eq.kc = static_cast<__nv_bfloat16 *>(kv->desc.k);
    eq.vc = static_cast<__nv_bfloat16 *>(kv->desc.v);
    eq.st_tok = kv->desc.stride_token;
    eq.st_head = kv->desc.stride_head;
    eq.st_batch = kv->desc.stride_batch;
    eq.q_norm = L->q_norm;
    eq.k_norm = L->k_norm;
    eq.eps = c.rms_eps;
    eq.inv_freq2 = L->inv_freq2;
    eq.qn = L->qn;
    eq.gate = L->gate;
    eq.tap_y = L->taps.y;
    if (kv->turbo) {
        eq.vq_codes = static_cast<uint8_t *>(kv->tdesc.v_codes);
        eq.vq_scales = static_cast<uint8_t *>(kv->tdesc.v_scales);
        eq.cq_head = kv->tdesc.code_stride_head;
        eq.cq_batch = kv->tdesc.code_stride_batch;
        eq.sq_head = kv->tdesc.scale_stride_head;
        eq.sq_batch = kv->tdesc.scale_stride_batch;
        eq.tq = L->tq;
        if (kv->kturbo) {
            eq.kq_codes = static_cast<uint8_t *>(kv->kq_codes);
            eq.kq_scales = static_cast<uint8_t *>(kv->kq_scales);
            eq.kcq_head = kv->tdesc.code_stride_head;
            eq.kcq_batch = kv->tdesc.code_stride_batch;
            eq.ksq_head = kv->tdesc.scale_stride_head;
            eq.ksq_batch = kv->tdesc.scale_stride_batch;
        }
    }
    EpiO eo{};
    CUDA_TRY(mark(launches));
    CUDA_TRY(launch_proj(L->pqkv.bits, NTa, kModeQKV, a, eq, eo, L->pqkv.grid[nia], pdl, s));
    launched(GATTN_KERNEL_PROJ_QKV);

    // 3. attention + merge + gate -> o_proj operand
    t.qn = L->qn;
    t.gate = L->gate;
    t.cache_pos = cache_pos;
    t.B = batch;
    t.R = q_len;
    t.H = c.num_heads;
    t.Hk = c.num_kv_heads;
    t.d = c.head_dim;
    t.cap = kv->desc.capacity;
    t.nrb = nrb;
    t.scale_log2 = scale_log2;
    t.nrb_u = nrb_u;
    t.ws = L->ws_attn;
    t.slot_ctr = L->slot_ctr;
    t.min_units = kAttnMinUnits;
    t.split = kAttnSplit;
    t.attn_grid = L->attn_grid;
    t.merge_rows = max_rows;
    // the partials a step stores and merges grow with rows x chunks: segments
    // of many rows are cut into fewer chunks (a route-independent bound: the
    // largest row block has the same rows in both head partitions)
    t.max_chunks = std::max(4, std::min(32, kChunkRowsBudget / std::max(1, max_rows)));
    t.x16 = L->x16_o;
    t.xsum = L->xsum_o;
    t.NT = NT;
    t.group_o = L->po.group;
    t.tap_attn = L->taps.attn;
    t.status = L->status;

    if (L->mask.mask) {
        t.mask = L->mask.mask;
        t.mask_heads = L->mask.heads;
        t.mask_len = L->mask.positions;
        t.mask_row = L->mask.stride_row;
        t.mask_head = L->mask.stride_head;
        t.mask_batch = L->mask.stride_batch;
    }
    if (kv->turbo) {
        t.vq = 1;
        t.vq_codes = static_cast<const uint8_t *>(kv->tdesc.v_codes);
        t.vq_scales = static_cast<const uint8_t *>(kv->tdesc.v_scales);
        t.cq_head = kv->tdesc.code_stride_head;
        t.cq_batch = kv->tdesc.code_stride_batch;
        t.sq_head = kv->tdesc.scale_stride_head;
        t.sq_batch = kv->tdesc.scale_stride_batch;
        t.vq_tl[0] = L->tq_tl[0];
        t.vq_tl[1] = L->tq_tl[1];
        t.vq_th[0] = L->tq_th[0];
        t.vq_th[1] = L->tq_th[1];
        t.inv_sqrt_d = L->tq.inv_sqrt_d;
        if (kv->kturbo) {
            t.vq = 2;
            t.kq_codes = static_cast<const uint8_t *>(kv->kq_codes);
            t.kq_scales = static_cast<const uint8_t *>(kv->kq_scales);
            t.kcq_head = kv->tdesc.code_stride_head;
            t.kcq_batch = kv->tdesc.code_stride_batch;
            t.ksq_head = kv->tdesc.scale_stride_head;
            t.ksq_batch = kv->tdesc.scale_stride_batch;
        }
    }
    CUDA_TRY(mark(launches));
    if (kv->kturbo)
        CUDA_TRY(launch_attn_vqk(MT, c.head_dim / 64, t, kv->kmap, L->attn_grid, pdl, s));
    else if (kv->turbo)
        CUDA_TRY(launch_attn_vq(MT, c.head_dim / 64, t, kv->kmap, L->attn_grid, pdl, s));
    else
        CUDA_TRY(launch_attn(MT, c.head_dim / 64, t, kv->kmap, kv->vmap, L->attn_grid, pdl, s));
    launched(GATTN_KERNEL_ATTN);
    CUDA_TRY(mark(launches));
    CUDA_TRY(launch_attn_merge(c.head_dim / 64, kv->kturbo ? 2 : kv->turbo ? 1 : 0, t,
                               batch * c.num_kv_heads * nrb, pdl, s));
    launched(GATTN_KERNEL_MERGE);
    CUDA_TRY(mark(launches));

    // 4. o_proj
    ProjArgs o = a;
    o.w = L->po.w;
    o.x16 = L->x16_o;
    o.xsum = L->xsum_o;
    o.nrb = L->po.nrb;
    o.nku = L->po.nku;
    o.N = L->po.N;
    o.group = L->po.group;
    o.unit_bytes = L->po.ubytes;
    o.step_bytes = L->po.step_bytes;
    o.stage_bytes = L->po.stage_bytes[ni];
    o.stages = L->po.stages[ni];
    o.rbc = 1;
    o.ks = L->po.ks[ni];
    o.eb_rows = kRBR;
    o.recv_cap = proj_recv_cap(kModeO, NT);
    o.xsplit = 0;
    o.withhold = 0;
    EpiO e2{};
    e2.R = q_len;
    e2.cache_pos = cache_pos;
    e2.cap = kv->desc.capacity;
    e2.out = static_cast<__nv_bfloat16 *>(out);
    e2.resid = blk ? x : nullptr;
    e2.resid_f32 = c.x_dtype == GATTN_DTYPE_F32;
    // decoder block: the post-norm rides in this launch when one CTA can do
    // it quickly and the rows allow 16-byte vectors
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool post_fused = blk && blk->out_normed && M * c.hidden <= kPostFuseMaxElems &&
                            a16(out) && a16(blk->out_normed) && a16(blk->post_ln);
    if (post_fused) {
        e2.post_w = blk->post_ln;
        e2.out_n = blk->out_normed;
        e2.eps = c.rms_eps;
        e2.ss_part = L->ss_part;
        e2.ticket = L->post_ticket;
    }
    CUDA_TRY(mark(launches));
    CUDA_TRY(launch_proj(L->po.bits, NT, kModeO, o, eq, e2, L->po.grid[ni], pdl, s));
    launched(GATTN_KERNEL_PROJ_O);

    // 5. decoder block: the post-attention RMSNorm of the residual stream,
    //    in its own launch when the o_proj did not take it
    if (blk && blk->out_normed && !post_fused) {
        CUDA_TRY(mark(launches));
        CUDA_TRY(launch_postnorm(static_cast<const __nv_bfloat16 *>(out), blk->post_ln, c.rms_eps, M,
                                 c.hidden, blk->out_normed, pdl, s));
        launched(GATTN_KERNEL_POSTNORM);
    }
    CUDA_TRY(mark_end());
    L->launches = launches;
    std::memcpy(L->kinds, kinds, sizeof kinds);
    return GATTN_OK;
}

}  // namespace

gattn_status gattn_layer_step(gattn_layer *L, const void *x, gattn_kv *kv, const int32_t *cache_pos,
                              int32_t batch, int32_t q_len, void *out, gattn_stream stream)
{
    return step_impl(L, x, kv, cache_pos, batch, q_len, out, stream, nullptr);
}

gattn_status gattn_layer_step_host(gattn_layer *L, const void *x_host, gattn_kv *kv,
                                   const int32_t *cache_pos_host, int32_t batch, int32_t q_len,
                                   void *out_host, gattn_stream stream)
{
    if (!L || !x_host || !kv || !cache_pos_host || !out_host)
        return fail(GATTN_E_INVALID_ARG, "NULL argument");
    const gattn_status chk = check_step(L, kv, batch, q_len);
    if (chk != GATTN_OK)
        return chk;
    const gattn_cfg &c = L->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t elems = (size_t)batch * q_len * c.hidden;
    // the inputs go to the slot the step before last read, on the layer's copy
    // stream once that step is done with it, so they land while the previous
    // step still runs; the step waits for them, out comes back on `stream`
    const int sl = L->stage_slot;
    CUDA_TRY(cudaStreamWaitEvent(L->copy_stream, L->stage_free[sl], 0));
    CUDA_TRY(cudaMemcpyAsync(L->x_stage[sl], x_host,
                             elems * (c.x_dtype == GATTN_DTYPE_F32 ? 4 : 2),
                             cudaMemcpyHostToDevice, L->copy_stream));
    CUDA_TRY(cudaMemcpyAsync(L->pos_stage[sl], cache_pos_host, (size_t)batch * sizeof(int32_t),
                             cudaMemcpyHostToDevice, L->copy_stream));
    CUDA_TRY(cudaEventRecord(L->stage_in[sl], L->copy_stream));
    CUDA_TRY(cudaStreamWaitEvent(s, L->stage_in[sl], 0));
    const gattn_status st = step_impl(L, L->x_stage[sl], kv, L->pos_stage[sl], batch, q_len,
                                      L->out_stage, stream, nullptr);
    if (st != GATTN_OK)
        return st;
    CUDA_TRY(cudaEventRecord(L->stage_free[sl], s));
    CUDA_TRY(cudaMemcpyAsync(out_host, L->out_stage, elems * 2, cudaMemcpyDeviceToHost, s));
    L->stage_slot = sl ^ 1;
    return GATTN_OK;
}

gattn_status gattn_layer_step_block(gattn_layer *L, const void *x, gattn_kv *kv,
                                    const int32_t *cache_pos, int32_t batch, int32_t q_len,
                                    const void *input_ln, const void *post_ln, void *out,
                                    void *out_normed, gattn_stream stream)
{
    if (!input_ln)
        return fail(GATTN_E_INVALID_ARG, "input_ln is NULL");
    if (out_normed && !post_ln)
        return fail(GATTN_E_INVALID_ARG, "out_normed needs post_ln");
    if (out_normed && out_normed == out)
        return fail(GATTN_E_INVALID_ARG, "out_normed must not alias out");
    BlockArgs blk{static_cast<const uint16_t *>(input_ln), static_cast<const uint16_t *>(post_ln),
                  static_cast<__nv_bfloat16 *>(out_normed)};
    return step_impl(L, x, kv, cache_pos, batch, q_len, out, stream, &blk);
}

gattn_status gattn_layer_poll_status(gattn_layer *L, gattn_stream stream)
{
    if (!L)
        return fail(GATTN_E_INVALID_ARG, "layer is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned v = 0;
    CUDA_TRY(cudaStreamSynchronize(s));
    CUDA_TRY(cudaMemcpy(&v, L->status, sizeof v, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemset(L->status, 0, sizeof v));
    if (v & kStatusTimeout)
        return fail(GATTN_E_DEVICE_TIMEOUT, "a bounded device wait gave up");
    if (v & kStatusRange)
        return fail(GATTN_E_DEVICE_RANGE, "cache_pos + q_len exceeded the cache capacity");
    return GATTN_OK;
}

gattn_status gattn_unpack_codes_device(const uint32_t *packed, int64_t N, int64_t K, int32_t bits,
                                       uint8_t *codes, gattn_stream stream)
{
    if (!packed || !codes || N < 0 || K < 0 || bits < 1 || bits > 8 || (K * bits) % 32)
        return fail(GATTN_E_INVALID_ARG, "bad unpack arguments");
    CUDA_TRY(launch_unpack_codes(packed, N, K, bits, codes, reinterpret_cast<cudaStream_t>(stream)));
    return GATTN_OK;
}

gattn_status gattn_layer_dequant_device(gattn_layer *L, int32_t proj, float *w, gattn_stream stream)
{
    if (!L || !w || proj < 0 || proj > 3)
        return fail(GATTN_E_INVALID_ARG, "bad dequant arguments");
    if (!L->weights_set)
        return fail(GATTN_E_STATE, "set_weights has not been called");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const ProjPlan &p = proj == 3 ? L->po : L->pqkv;
    float *tmp = nullptr;
    CUDA_TRY(cudaMalloc(&tmp, (size_t)p.nrb * kRBR * p.K * sizeof(float)));
    cudaError_t e = launch_dequant_tiles(p.w, p.nrb * kRBR, p.K, p.bits, p.group, p.nrb, tmp, s);
    const int row0 = proj == 0 ? 0 : (proj == 1 ? L->Nq : (proj == 2 ? L->Nq + L->Nkv : 0));
    const int rows = proj == 0 ? L->Nq : (proj == 3 ? L->po.N : L->Nkv);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(w, tmp + (size_t)row0 * p.K, (size_t)rows * p.K * sizeof(float),
                            cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    cudaFree(tmp);
    if (e != cudaSuccess)
        return fail(GATTN_E_CUDA, "dequant failed: %s", cudaGetErrorString(e));
    return GATTN_OK;
}

}  // extern "C"
