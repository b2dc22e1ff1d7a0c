// attn.cuh -- the attention kernel template, instantiated for bf16 V caches
// in attn.cu and for Bf16KTurbo4V caches in attn_vq.cu.
#pragma once
#include "common.cuh"
#include "kernels.cuh"

namespace gattn {

// bytes of one 64-wide head_dim box of a tile (kAttnTile tokens x 128 bytes);
// a multiple of 1024 so every box starts on a 128-byte-swizzle atom
constexpr int kDBox = kAttnTile * 128;
static_assert(kDBox % 1024 == 0, "tile boxes must stay swizzle-atom aligned");

template <int MT, int DB, int VQ>
struct AttnSmem {
    static constexpr int kTileBytes = DB * kDBox;             // kAttnTile tokens x d bf16
    // K and V of a stage: the bf16 tile, or (Turbo4) the tile's code rows (d/2
    // bytes per token) followed by its scale rows (d/16 bytes per token); V is
    // Turbo4 for VQ >= 1, K too for VQ == 2 (the symmetric format)
    static constexpr int kVCodeBytes = kAttnTile * DB * 32;
    static constexpr int kQuantBytes = (kVCodeBytes + kAttnTile * DB * 4 + 1023) & ~1023;
    static constexpr int kKBytes = VQ == 2 ? kQuantBytes : kTileBytes;
    static constexpr int kVBytes = VQ ? kQuantBytes : kTileBytes;
    static constexpr int kStageBytes = kKBytes + kVBytes;     // K + V
    static constexpr int kDqBytes = VQ ? kTileBytes : 0;      // Turbo4: dequantized fp16 V tile
    static constexpr int kDqKBytes = VQ == 2 ? kTileBytes : 0;    // and K tile
    static constexpr int kQBytes = MT * 16 * DB * 64 * 2;
    static constexpr int kPBytes = MT * 16 * 128;             // rows x 64 tokens bf16
    // as many K/V stages (2 .. kAttnStages) as fit beside the rest in 227 KB
    static constexpr int kFixed = kDqBytes + kDqKBytes + kQBytes + kPBytes +
                                  2 * kAttnWarps * 64 * 4 + 80 * 8 + 2 * kAttnStages * 8 + 512 + 1024;
    static constexpr int kFit = (227 * 1024 - kFixed) / kStageBytes;
    static constexpr int kNStages = kFit < 2 ? 2 : (kFit > kAttnStages ? kAttnStages : kFit);
    static constexpr int kStages = kNStages * kStageBytes;
    static constexpr int kDq = kStages;
    static constexpr int kDqK = kDq + kDqBytes;
    static constexpr int kQ = kDqK + kDqKBytes;
    static constexpr int kP = kQ + kQBytes;
    static constexpr int kRedMax = kP + kPBytes;              // [8][64] floats
    static constexpr int kRedL = kRedMax + kAttnWarps * 64 * 4;
    static constexpr int kPrefix = kRedL + kAttnWarps * 64 * 4;   // 2 x [33] long long
    static constexpr int kBars = kPrefix + 80 * 8;
    static constexpr int kFlags = kBars + 2 * kNStages * 8;
    static constexpr int kTotal = kFlags + 512 + 1024;        // + alignment slack
    static_assert(kTotal <= 227 * 1024, "attention shared memory exceeds 227 KB");
};

// One Turbo4 dequantization item: 32 columns (c) of token tl of a tile, from
// its 16 code bytes and 2 E4M3 scales into the fp16 tile (the bf16 tile's
// swizzled layout).  Split into its loads and its conversion so that a thread
// issues the loads of all its items before converting any: the shared-memory
// accesses are ordered asm statements, so only this order lets the items'
// arithmetic overlap.
struct TurboItem {
    uint4 cb;
    uint32_t sb;
};

// Shared-memory addresses: cst / sst the code / scale rows.
template <int DB>
__device__ __forceinline__ TurboItem turbo_item_load(uint32_t cst, uint32_t sst, int tl, int c,
                                                     bool live)
{
    TurboItem it{make_uint4(0, 0, 0, 0), 0u};
    if (live) {
        it.cb = lds_v4(cst + tl * (DB * 32) + c * 16);
        it.sb = lds_u16(sst + tl * (DB * 4) + c * 2);
    }
    return it;
}

// A 16-byte store is served eight lanes at a time; those lanes share a token
// and take its 32-column pieces c, so each lane writes its four 8-column
// chunks in an order rotated by c: at every step the eight lanes hit eight
// different bank groups.  A not-live item (zero scales) writes zeros.
template <int DB>
__device__ __forceinline__ void turbo_item_store(uint32_t dst, const TurboItem &it, int tl, int c,
                                                 const uint32_t (&lvl_lo)[2],
                                                 const uint32_t (&lvl_hi)[2])
{
    constexpr int kRotShift = DB == 4 ? 1 : 0;
    const int rot = (c >> kRotShift) & 3;
    const __half2 s0 = __half2half2(e4m3_to_half((uint8_t)(it.sb & 0xFF)));
    const __half2 s1 = __half2half2(e4m3_to_half((uint8_t)(it.sb >> 8)));
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const int q = (st + rot) & 3;            // bytes 4q .. 4q + 3
        const uint32_t wq = q == 0 ? it.cb.x : (q == 1 ? it.cb.y : (q == 2 ? it.cb.z : it.cb.w));
        const __half2 sc = q < 2 ? s0 : s1;      // groups 2c, 2c + 1
        uint32_t o[4];
        turbo4_levels8(wq, lvl_lo, lvl_hi, o);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
            const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&o[k2]), sc);
            o[k2] = *reinterpret_cast<const uint32_t *>(&v);
        }
        const int ch = 4 * c + q;                // 8-column chunk of the row
        sts_v4(dst + (ch >> 3) * kDBox + tl * 128 + (((ch & 7) ^ (tl & 7)) << 4), o[0], o[1], o[2],
               o[3]);
    }
}

// Chunks per segment, at most: the chunk length grows for longer segments so
// that one merge combines every partial of a segment (lane j holds chunk j).
constexpr int kMaxChunks = 32;

// The chunk plan of a step, the same in every CTA: sequence b's segments (one
// per KV head and row block) are cut into nc[b] <= kMaxChunks chunks of cu
// 16-token units.  cu depends only on the lengths and on the row-block count of
// the unchunked head partition (nrb_u), so the head-chunk route and the plain
// route cut every segment at the same tokens, and each row sees the same chunks
// in both.
struct ChunkPlan {
    int cu;                        // units per chunk
    const int *ub, *nc;            // units / chunks of each sequence's segments
    const long long *pi;           // first item of each sequence [B + 1]
};

struct Item {
    int b, kh, rb, chunk;
    long long seg, first;          // segment id, the segment's first item
    int u0, u1;                    // units [u0, u1) of the segment
};

__device__ __forceinline__ Item item_of(const ChunkPlan &cp, int B, int Hk, int nrb, long long i)
{
    Item it;
    int b = 0;
    while (b + 1 < B && cp.pi[b + 1] <= i)
        ++b;
    const int n = cp.nc[b];
    const long long loc = i - cp.pi[b];
    const long long sl = loc / n;
    it.b = b;
    it.chunk = (int)(loc - sl * n);
    it.kh = (int)(sl / nrb);
    it.rb = (int)(sl % nrb);
    it.seg = ((long long)b * Hk + it.kh) * nrb + it.rb;
    it.first = cp.pi[b] + sl * n;
    it.u0 = it.chunk * cp.cu;
    it.u1 = min(cp.ub[b], (it.chunk + 1) * cp.cu);
    return it;
}

// The chunk plan of a step for an attention launch of `grid` CTAs (every CTA
// of that launch and of the merge launch computes the same one): per sequence
// the units ub, the chunks per segment nc, the first item pi and the first
// item's unit offset uo (pi[B], uo[B]: totals), in shared memory; returns cu.
// cu units per chunk: the unchunked partition's unit count over split x the
// grid, at least min_units and at least the longest segment's units over
// max_chunks (<= kMaxChunks).  Called by every thread of the block (two barriers).
__device__ __forceinline__ int chunk_plan(const AttnArgs &a, int grid, int *ub, int *nc,
                                          long long *pi, long long *uo, int *cu_slot)
{
    const int tid = threadIdx.x;
    if (tid < a.B) {
        const int p0 = a.cache_pos[tid];
        const bool valid = p0 >= 0 && p0 + a.R <= a.cap;
        ub[tid] = valid ? (p0 + a.R + kAttnUnit - 1) / kAttnUnit : 0;
    }
    __syncthreads();
    if (tid == 0) {
        long long uu = 0;
        int umax = 0;
        for (int b = 0; b < a.B; ++b) {
            uu += (long long)ub[b] * a.Hk * a.nrb_u;
            umax = max(umax, ub[b]);
        }
        const long long parts = (long long)a.split * grid;
        const long long per = (uu + parts - 1) / parts;
        int cu = (int)(per > a.min_units ? per : a.min_units);
        cu = max(cu, (umax + a.max_chunks - 1) / a.max_chunks);
        long long ai = 0, au = 0;
        for (int b = 0; b < a.B; ++b) {
            const int n = (ub[b] + cu - 1) / cu;
            nc[b] = n;
            pi[b] = ai;
            uo[b] = au;
            ai += (long long)n * a.Hk * a.nrb;
            au += (long long)ub[b] * a.Hk * a.nrb;
        }
        pi[a.B] = ai;
        uo[a.B] = au;
        *cu_slot = cu;
    }
    __syncthreads();
    return *cu_slot;
}

// The first item (in item order) that starts at unit offset x or later; uo[b]
// is the unit offset of sequence b's first item (uo[B]: all units).
__device__ __forceinline__ long long first_item_at(const ChunkPlan &cp, const long long *uo, int B,
                                                   long long x)
{
    if (x >= uo[B])
        return cp.pi[B];
    int b = 0;
    while (b + 1 < B && uo[b + 1] <= x)
        ++b;
    const long long loc = x - uo[b];
    const int ubb = cp.ub[b];              // > 0: an empty sequence spans no offsets
    const long long sl = loc / ubb;
    const long long r = loc - sl * ubb;
    return cp.pi[b] + sl * cp.nc[b] + (r + cp.cu - 1) / cp.cu;
}

template <int MT, int DB, int VQ>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap)
{
    using L = AttnSmem<MT, DB, VQ>;
    constexpr int D = DB * 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + L::kQ;
    uint8_t *dq = smem + L::kDq;                                // Turbo4 only
    uint8_t *dqk = smem + L::kDqK;                              // symmetric Turbo4 only
    uint8_t *ps = smem + L::kP;
    float *red_max = reinterpret_cast<float *>(smem + L::kRedMax);
    float *red_l = reinterpret_cast<float *>(smem + L::kRedL);
    long long *pi = reinterpret_cast<long long *>(smem + L::kPrefix);     // [33] first item
    long long *uo = pi + 40;                // [33] unit offset of each sequence's first item
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *empty = full + L::kNStages;
    int *flags = reinterpret_cast<int *>(smem + L::kFlags);   // [0] abort [2] work slot [4] cu
    int *ub = flags + 8;                                        // units per segment of b [32]
    int *nc = ub + 32;                                          // chunks per segment of b [32]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gqa = a.H / a.Hk;

    // Dependents (the o_proj) may launch at once.  Before waiting for the q|k|v
    // projection this kernel only reads cache_pos and cache rows older than the
    // step: the projection starts its dependents after its own wait, so every
    // earlier kernel (which wrote those rows) has completed by then.
    pdl_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < L::kNStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kAttnWarps);
        }
        flags[0] = 0;
        // this CTA's work slot, in the order the CTAs start: every launch adds
        // exactly gridDim.x to the layer's counter, so the slots of a launch
        // are 0 .. gridDim.x - 1 whatever the counter held before
        flags[2] = (int)(atomicAdd(a.slot_ctr, 1ull) % gridDim.x);
        fence_mbar_init();
    }
    const int cu = chunk_plan(a, gridDim.x, ub, nc, pi, uo, &flags[4]);
    const ChunkPlan cp{cu, ub, nc, pi};

    // the items of slot c: with no more items than CTAs, item c (the CTAs that
    // start last, while the previous kernel still holds their SMs, are left
    // without work); else contiguous item ranges balanced by units: slot c
    // takes the items that start in its share of the units (consecutive
    // chunks of a segment in one CTA share its q rows)
    const long long U = uo[a.B], c = flags[2], items = pi[a.B];
    const bool one_each = items <= (long long)gridDim.x;
    const long long beg = one_each ? min(c, items) : first_item_at(cp, uo, a.B, U * c / gridDim.x);
    const long long end = one_each ? min(c + 1, items)
                                   : first_item_at(cp, uo, a.B, U * (c + 1) / gridDim.x);
    volatile int *abort = flags;

    if (warp == kAttnWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && beg < end) {
            if constexpr (VQ != 2)
                prefetch_tensormap(&kmap);
            if constexpr (!VQ)
                prefetch_tensormap(&vmap);
            const uint64_t pol = l2_evict_first_policy();
            long long it = 0;
            bool stop = false, waited = false;
            for (long long item = beg; item < end && !stop; ++item) {
                const Item p = item_of(cp, a.B, a.Hk, a.nrb, item);
                const int p0 = a.cache_pos[p.b];
                for (int u = p.u0; u < p.u1; u += kAttnTile / kAttnUnit, ++it) {
                    const int nun = min(kAttnTile / kAttnUnit, p.u1 - u);
                    // tiles that hold this step's new rows load after the projection
                    if (!waited && (it >= L::kNStages || (u + nun) * kAttnUnit > p0)) {
                        pdl_wait();
                        waited = true;
                    }
                    const int slot = (int)(it % L::kNStages);
                    const uint32_t ph = (uint32_t)((it / L::kNStages) & 1);
                    if (!mbar_wait(&empty[slot], ph ^ 1u, abort, a.status)) {
                        stop = true;
                        break;
                    }
                    uint8_t *kst = smem + slot * L::kStageBytes;
                    uint8_t *vst = kst + L::kKBytes;
                    // Turbo4 planes: the tile's code and scale rows are contiguous (the
                    // capacity is a multiple of the 16-token unit, so they end in range)
                    const uint32_t vq_code = VQ ? (uint32_t)(nun * kAttnUnit * DB * 32) : 0u;
                    const uint32_t vq_scale = VQ ? (uint32_t)(nun * kAttnUnit * DB * 4) : 0u;
                    const uint32_t tile_bytes = (uint32_t)(nun * DB * 2048);
                    mbar_arrive_expect_tx(&full[slot], (VQ == 2 ? vq_code + vq_scale : tile_bytes) +
                                                           (VQ ? vq_code + vq_scale : tile_bytes));
                    if constexpr (VQ != 2) {
                        for (int ui = 0; ui < nun; ++ui) {
                            const int t = (u + ui) * kAttnUnit;
#pragma unroll
                            for (int db = 0; db < DB; ++db) {
                                tensor4d_g2s(kst + db * kDBox + ui * 2048, &kmap, db * 64, t, p.kh,
                                             p.b, &full[slot], pol);
                                if constexpr (!VQ)
                                    tensor4d_g2s(vst + db * kDBox + ui * 2048, &vmap, db * 64, t,
                                                 p.kh, p.b, &full[slot], pol);
                            }
                        }
                    } else {
                        const long long t = (long long)u * kAttnUnit;
                        bulk_g2s(kst, a.kq_codes + p.b * a.kcq_batch + p.kh * a.kcq_head + t * (DB * 32),
                                 vq_code, &full[slot], pol);
                        bulk_g2s(kst + L::kVCodeBytes,
                                 a.kq_scales + p.b * a.ksq_batch + p.kh * a.ksq_head + t * (DB * 4),
                                 vq_scale, &full[slot], pol);
                    }
                    if constexpr (VQ) {
                        const long long t = (long long)u * kAttnUnit;
                        bulk_g2s(vst, a.vq_codes + p.b * a.cq_batch + p.kh * a.cq_head + t * (DB * 32),
                                 vq_code, &full[slot], pol);
                        bulk_g2s(vst + L::kVCodeBytes,
                                 a.vq_scales + p.b * a.sq_batch + p.kh * a.sq_head + t * (DB * 4),
                                 vq_scale, &full[slot], pol);
                    }
                }
            }
            if (!waited)
                pdl_wait();
            const long long first = it > L::kNStages ? it - L::kNStages : 0;
            for (long long i = first; i < it; ++i) {
                unsigned long long t0 = global_ns();
                while (!mbar_try(&full[i % L::kNStages], (uint32_t)((i / L::kNStages) & 1)) &&
                       global_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // --------------------------------------------------------------- consumers
    // the arguments read after the wait are brought into the constant cache
    // while waiting
    if (tid == 0)
        reinterpret_cast<volatile unsigned *>(flags)[5] = arg_fold(a);
    pdl_wait();                 // q rows come from the q|k|v projection
    const int g = lane >> 2, cq = lane & 3;
    long long it = 0, qseg = -1;
    for (long long item = beg; item < end; ++item) {
        const Item p = item_of(cp, a.B, a.Hk, a.nrb, item);
        const int nh = a.rb_nh[p.rb];
        const int h0 = p.kh * gqa + a.rb_h0[p.rb];
        const int nrows = nh * a.R;
        const int p0 = a.cache_pos[p.b];
        const int Lb = p0 + a.R;

        // ---- q rows of this segment into shared memory (swizzled 16-byte chunks),
        //      once per run of items of one segment
        constexpr int CH = D / 8;   // chunks per row
        const bool load_q = p.seg != qseg;
        qseg = p.seg;
        if (!load_q) {
        } else if constexpr (VQ == 2) {
            // symmetric Turbo4: the keys live in the rotated basis, so the rows
            // are rotated once (q' = H q / sqrt(d): q . k = q' . H k / sqrt(d))
            // and kept in fp16 for the fp16 products with the dequantized keys
            for (int i = warp; i < MT * 16; i += kAttnWarps) {
                float xr[8];
                const int hl = i / a.R, r = i % a.R;
                const __nv_bfloat16 *src =
                    a.qn + (((long long)p.b * a.R + r) * a.H + h0 + hl) * D;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    xr[k] = (i < nrows && k < D / 32) ? __bfloat162float(src[lane + 32 * k]) : 0.f;
                wht_warp(xr, D / 32, lane);
#pragma unroll
                for (int k = 0; k < D / 32; ++k) {
                    const int j = lane + 32 * k;
                    *reinterpret_cast<__half *>(qs + i * (D * 2) + (((j >> 3) ^ (i & 7)) << 4) +
                                                (j & 7) * 2) = __float2half_rn(xr[k] * a.inv_sqrt_d);
                }
            }
        } else {
            // every load first (one round trip), then the stores
            constexpr int NQ = (MT * 16 * CH + kAttnWarps * 32 - 1) / (kAttnWarps * 32);
            uint4 qv[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int idx = tid + q * kAttnWarps * 32, i = idx / CH, cc = idx % CH;
                qv[q] = make_uint4(0, 0, 0, 0);
                if (i < nrows) {
                    const int hl = i / a.R, r = i % a.R;
                    qv[q] = *reinterpret_cast<const uint4 *>(
                        a.qn + (((long long)p.b * a.R + r) * a.H + h0 + hl) * D + cc * 8);
                }
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int idx = tid + q * kAttnWarps * 32, i = idx / CH, cc = idx % CH;
                if (idx < MT * 16 * CH)
                    *reinterpret_cast<uint4 *>(qs + i * (D * 2) + ((cc ^ (i & 7)) << 4)) = qv[q];
            }
        }
        named_bar_sync(1, kAttnWarps * 32);

        float m_run[MT][2], l_run[MT][2], O[MT][DB][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            m_run[mt][0] = m_run[mt][1] = -INFINITY;
            l_run[mt][0] = l_run[mt][1] = 0.f;
#pragma unroll
            for (int j = 0; j < DB; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    O[mt][j][e] = 0.f;
        }

        for (int u = p.u0; u < p.u1; u += kAttnTile / kAttnUnit, ++it) {
            const int nun = min(kAttnTile / kAttnUnit, p.u1 - u);
            const int ntok = nun * kAttnUnit;
            const int t0 = u * kAttnUnit;
            const int slot = (int)(it % L::kNStages);
            const uint32_t ph = (uint32_t)((it / L::kNStages) & 1);
            const bool ok = mbar_wait(&full[slot], ph, abort, a.status);
            uint8_t *kst = smem + slot * L::kStageBytes;
            uint8_t *vst = kst + L::kKBytes;

            // symmetric Turbo4: each warp dequantizes the key rows of its own 8
            // tokens (the only ones its q K^T reads) into the fp16 key tile
            if constexpr (VQ == 2) {
                if (ok && warp * 8 < ntok) {
                    const uint32_t lvl_lo[2] = {a.vq_tl[0], a.vq_tl[1]};
                    const uint32_t lvl_hi[2] = {a.vq_th[0], a.vq_th[1]};
                    constexpr int kKItems = (8 * DB * 2 + 31) / 32;
                    TurboItem ki[kKItems];
#pragma unroll
                    for (int k = 0; k < kKItems; ++k) {
                        const int it2 = lane + 32 * k;
                        const int tl = warp * 8 + it2 / (DB * 2), c = it2 % (DB * 2);
                        ki[k] = turbo_item_load<DB>(smem_u32(kst), smem_u32(kst) + L::kVCodeBytes,
                                                    tl, c, it2 < 8 * DB * 2 && tl < ntok && t0 + tl < Lb);
                    }
#pragma unroll
                    for (int k = 0; k < kKItems; ++k) {
                        const int it2 = lane + 32 * k;
                        const int tl = warp * 8 + it2 / (DB * 2), c = it2 % (DB * 2);
                        if (it2 < 8 * DB * 2)
                            turbo_item_store<DB>(smem_u32(dqk), ki[k], tl, c, lvl_lo, lvl_hi);
                    }
                    __syncwarp();
                }
            }

            // positions past the sequence end hold stale memory: zero those V rows
            // (Turbo4: the dequantization writes zeros there instead)
            if (!VQ && ok && t0 + ntok > Lb) {
                const int first = Lb - t0 > 0 ? Lb - t0 : 0;
                for (int idx = tid; idx < (ntok - first) * DB * 8; idx += kAttnWarps * 32) {
                    const int row = first + idx / (DB * 8), rest = idx % (DB * 8);
                    const int db = rest >> 3, cc = rest & 7;
                    *reinterpret_cast<uint4 *>(vst + db * kDBox + row * 128 + cc * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }

            // ---- S = q K^T for this warp's 8 tokens; the head_dim contraction is
            //      spread over SPLIT independent accumulator chains (MMA latency)
            // (two chains whatever the row count, so a row's sums do not depend on
            // how many rows its segment has: the head-chunk route and the plain
            // route add every score in the same order)
            constexpr int SPLIT = 2;
            float sc[MT][4];
            float scs[SPLIT][MT][4];
            const bool has_tok = ok && (warp * 8 < ntok);
            // attention mask: this lane's score bytes (bit mt * 4 + e), loaded before
            // the q K^T loop so that their latency hides behind it
            uint32_t mkeep = 0;
            if (a.mask && has_tok) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = mt * 16 + g + ((e & 2) ? 8 : 0);
                        const int t = t0 + warp * 8 + 2 * cq + (e & 1);
                        if (i < nrows && t < Lb && t < a.mask_len) {
                            const int hh = h0 + i / a.R, rr = i % a.R;
                            const uint8_t *mp = a.mask + p.b * a.mask_batch +
                                                (a.mask_heads > 1 ? hh : 0) * a.mask_head +
                                                rr * a.mask_row + t;
                            if (__ldg(mp))
                                mkeep |= 1u << (mt * 4 + e);
                        }
                    }
            }
#pragma unroll
            for (int q = 0; q < SPLIT; ++q)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        scs[q][mt][e] = 0.f;
            if (has_tok) {
                const int tok = warp * 8 + (lane & 7);
#pragma unroll
                for (int k2 = 0; k2 < 2 * DB; ++k2) {
                    const int chunk = k2 * 4 + (lane >> 3);
                    uint32_t kb[4];
                    ldsm_x4(kb, smem_u32((VQ == 2 ? dqk : kst) + (chunk >> 3) * kDBox + tok * 128 +
                                         (((chunk & 7) ^ (tok & 7)) << 4)));
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int ks = 2 * k2 + h;
                            const int qrow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                            const int qch = 2 * ks + (lane >> 4);
                            uint32_t qa[4];
                            ldsm_x4(qa, smem_u32(qs + qrow * (D * 2) + ((qch ^ (qrow & 7)) << 4)));
                            if constexpr (VQ == 2)
                                mma_f16(scs[ks % SPLIT][mt], qa, kb[2 * h], kb[2 * h + 1],
                                        scs[ks % SPLIT][mt]);
                            else
                                mma_bf16(scs[ks % SPLIT][mt], qa, kb[2 * h], kb[2 * h + 1],
                                         scs[ks % SPLIT][mt]);
                        }
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float t = scs[0][mt][e];
#pragma unroll
                    for (int q = 1; q < SPLIT; ++q)
                        t += scs[q][mt][e];
                    sc[mt][e] = t;
                }
            // ---- mask (causal per verify row), scale, warp row max
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = mt * 16 + g + ((e & 2) ? 8 : 0);
                    const int t = t0 + warp * 8 + 2 * cq + (e & 1);
                    const bool vis = has_tok && i < nrows &&
                                     (a.mask ? ((mkeep >> (mt * 4 + e)) & 1u) != 0u
                                             : t <= p0 + (i % a.R));
                    sc[mt][e] = vis ? sc[mt][e] * a.scale_log2 : -INFINITY;
                }
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float mx = fmaxf(sc[mt][2 * hr], sc[mt][2 * hr + 1]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    if (cq == 0)
                        red_max[warp * 64 + mt * 16 + g + 8 * hr] = mx;
                }
            }
            named_bar_sync(1, kAttnWarps * 32);
            // ---- Turbo4 V: dequantize the tile into the fp16 tile (same layout as the
            //      bf16 V tile); every warp has finished the previous tile's P V
            if constexpr (VQ) {
                if (ok) {
                    const uint32_t cst = smem_u32(vst), sst = cst + L::kVCodeBytes;
                    const uint32_t dq_a = smem_u32(dq);
                    const uint32_t lvl_lo[2] = {a.vq_tl[0], a.vq_tl[1]}, lvl_hi[2] = {a.vq_th[0], a.vq_th[1]};
                    // every item's loads first, then their conversions (see TurboItem)
                    constexpr int kItems = (kAttnTile * DB * 2 + kAttnWarps * 32 - 1) /
                                           (kAttnWarps * 32);
                    TurboItem vi[kItems];
#pragma unroll
                    for (int k = 0; k < kItems; ++k) {
                        const int idx = tid + k * kAttnWarps * 32;
                        const int tl = idx / (DB * 2), c = idx % (DB * 2);   // token, 32 columns
                        vi[k] = turbo_item_load<DB>(cst, sst, tl, c,
                                                    idx < kAttnTile * DB * 2 && tl < ntok &&
                                                        t0 + tl < Lb);
                    }
#pragma unroll
                    for (int k = 0; k < kItems; ++k) {
                        const int idx = tid + k * kAttnWarps * 32;
                        const int tl = idx / (DB * 2), c = idx % (DB * 2);
                        if (idx < kAttnTile * DB * 2)
                            turbo_item_store<DB>(dq_a, vi[k], tl, c, lvl_lo, lvl_hi);
                    }
                }
            }
            // ---- online softmax update, P to shared memory
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = mt * 16 + g + 8 * hr;
                    float tmax = -INFINITY;
#pragma unroll
                    for (int w2 = 0; w2 < kAttnWarps; ++w2)
                        tmax = fmaxf(tmax, red_max[w2 * 64 + i]);
                    const float m_new = fmaxf(m_run[mt][hr], tmax);
                    const float base = (m_new == -INFINITY) ? 0.f : m_new;
                    const float alpha = exp2f(m_run[mt][hr] - base);
                    m_run[mt][hr] = m_new;
                    const float p0f = exp2f(sc[mt][2 * hr] - base);
                    const float p1f = exp2f(sc[mt][2 * hr + 1] - base);
                    // P in the V tile's type (bf16, or fp16 for the Turbo4 tile); l sums the
                    // rounded values the MMA multiplies
                    float pr0, pr1;
                    uint32_t pk;
                    if constexpr (VQ) {
                        const __half2 hp = __floats2half2_rn(p0f, p1f);
                        pk = *reinterpret_cast<const uint32_t *>(&hp);
                        pr0 = __low2float(hp);
                        pr1 = __high2float(hp);
                    } else {
                        pk = pack_bf16x2(p0f, p1f);
                        pr0 = bf16_lo(pk);
                        pr1 = bf16_hi(pk);
                    }
                    l_run[mt][hr] = l_run[mt][hr] * alpha + (pr0 + pr1);
#pragma unroll
                    for (int j = 0; j < DB; ++j) {
                        O[mt][j][2 * hr] *= alpha;
                        O[mt][j][2 * hr + 1] *= alpha;
                    }
                    if (has_tok)
                        *reinterpret_cast<uint32_t *>(ps + i * 128 + ((warp ^ (i & 7)) << 4) +
                                                      cq * 4) = pk;
                }
            }
            named_bar_sync(1, kAttnWarps * 32);
            // ---- O += P V for this warp's head_dim slice
            const uint8_t *vt = VQ ? dq : vst;
            if (ok) {
#pragma unroll
                for (int kt = 0; kt < kAttnTile / 16; ++kt) {
                    if (kt * 16 < ntok) {
                        const int tok = kt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                        uint32_t vb[DB][2];
#pragma unroll
                        for (int j = 0; j < DB; j += 2) {
                            const int nd = warp * DB + j;
                            if (j + 1 < DB) {
                                const int chunk = nd + (lane >> 4);
                                uint32_t r[4];
                                ldsm_x4_trans(r, smem_u32(vt + (chunk >> 3) * kDBox + tok * 128 +
                                                          (((chunk & 7) ^ (tok & 7)) << 4)));
                                vb[j][0] = r[0];
                                vb[j][1] = r[1];
                                vb[j + 1][0] = r[2];
                                vb[j + 1][1] = r[3];
                            } else {
                                const int chunk = nd;
                                ldsm_x2_trans(vb[j][0], vb[j][1],
                                              smem_u32(vt + (chunk >> 3) * kDBox + tok * 128 +
                                                       (((chunk & 7) ^ (tok & 7)) << 4)));
                            }
                        }
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int prow = mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                            const int pch = 2 * kt + (lane >> 4);
                            uint32_t pa[4];
                            ldsm_x4(pa, smem_u32(ps + prow * 128 + ((pch ^ (prow & 7)) << 4)));
#pragma unroll
                            for (int j = 0; j < DB; ++j) {
                                if constexpr (VQ)
                                    mma_f16(O[mt][j], pa, vb[j][0], vb[j][1], O[mt][j]);
                                else
                                    mma_bf16(O[mt][j], pa, vb[j][0], vb[j][1], O[mt][j]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }

        // the row sums of l: per warp (its tokens), then over the warps in order
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float l = l_run[mt][hr];
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                if (cq == 0)
                    red_l[warp * 64 + mt * 16 + g + 8 * hr] = l;
            }
        const int n = cp.nc[p.b];
        if (VQ == 0 && n == 1) {
            // ---- the segment's only chunk: normalize, gate and write the o_proj
            //      operand from the accumulators (the same products as a one-slot
            //      merge: o * (1 / l)); the gate is requested before the barrier
            const long long Ktot = (long long)a.H * D;
            float2 gv[MT][DB][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = mt * 16 + g + 8 * hr;
                    const long long base = ((long long)p.b * a.R + r % a.R) * Ktot +
                                           (long long)(h0 + r / a.R) * D;
#pragma unroll
                    for (int j = 0; j < DB; ++j)
                        gv[mt][j][hr] = r < nrows ? __ldcg(reinterpret_cast<const float2 *>(
                                                        a.gate + base + (warp * DB + j) * 8 + 2 * cq))
                                                  : make_float2(0.f, 0.f);
                }
            named_bar_sync(1, kAttnWarps * 32);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = mt * 16 + g + 8 * hr;
                    float l = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kAttnWarps; ++w2)
                        l += red_l[w2 * 64 + r];
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    const int m = p.b * a.R + r % a.R, h = h0 + r / a.R;
                    float rs = 0.f;
#pragma unroll
                    for (int j = 0; j < DB; ++j) {
                        const int c = h * D + (warp * DB + j) * 8 + 2 * cq;
                        const float o0 = O[mt][j][2 * hr] * inv, o1 = O[mt][j][2 * hr + 1] * inv;
                        const __half q0 = __float2half_rn(o0 * (1.f / (1.f + __expf(-gv[mt][j][hr].x))));
                        const __half q1 = __float2half_rn(o1 * (1.f / (1.f + __expf(-gv[mt][j][hr].y))));
                        if (r < nrows) {
                            *reinterpret_cast<__half2 *>(a.x16 + x16_offset(m, c, a.NT)) =
                                __halves2half2(q0, q1);
                            if (a.tap_attn)
                                *reinterpret_cast<float2 *>(a.tap_attn + (long long)m * Ktot + c) =
                                    make_float2(o0, o1);
                        }
                        rs += __half2float(q0) + __half2float(q1);
                    }
                    rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                    rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                    if (cq == 0)
                        red_max[warp * 64 + r] = rs;     // this warp's columns of row r
                }
            named_bar_sync(1, kAttnWarps * 32);
            // group sums of the fp16 operand: a group of gs columns is the column
            // slices of gs / (8 DB) consecutive warps, added in warp order
            const int gs = a.group_o, ng = D / gs, wpg = gs / (8 * DB), MP = 8 * a.NT;
            for (int idx = tid; idx < nrows * ng; idx += kAttnWarps * 32) {
                const int r = idx / ng, gi = idx % ng;
                float t = 0.f;
                for (int w2 = gi * wpg; w2 < (gi + 1) * wpg; ++w2)
                    t += red_max[w2 * 64 + r];
                const int m = p.b * a.R + r % a.R, c0 = (h0 + r / a.R) * D + gi * gs;
                a.xsum[((long long)(c0 >> 7) * (kKU / gs) + ((c0 & 127) / gs)) * MP + m] = t;
            }
        } else {
            // ---- partial (m, l, O) of this chunk into its slot (valid rows only)
            const long long sf = attn_slot_floats(D);
            float *part = a.ws + item * sf;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int j = 0; j < DB; ++j) {
                    const int col = (warp * DB + j) * 8 + 2 * cq;
                    const int r0 = mt * 16 + g;
                    if (r0 < nrows)
                        *reinterpret_cast<float2 *>(part + 2 * kAttnMaxRows + (long long)r0 * D + col) =
                            make_float2(O[mt][j][0], O[mt][j][1]);
                    if (r0 + 8 < nrows)
                        *reinterpret_cast<float2 *>(part + 2 * kAttnMaxRows + (long long)(r0 + 8) * D +
                                                    col) = make_float2(O[mt][j][2], O[mt][j][3]);
                }
            named_bar_sync(1, kAttnWarps * 32);
            if (warp == 0 && cq == 0) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int i = mt * 16 + g + 8 * hr;
                        float l = 0.f;
#pragma unroll
                        for (int w2 = 0; w2 < kAttnWarps; ++w2)
                            l += red_l[w2 * 64 + i];
                        part[i] = m_run[mt][hr];
                        part[kAttnMaxRows + i] = l;
                    }
            }
        }
        // red_l and red_max are rewritten by the next item
        named_bar_sync(1, kAttnWarps * 32);
    }
}


template <int MT, int DB, int VQ>
static cudaError_t launch_attn_t(const AttnArgs &a, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, int grid, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = AttnSmem<MT, DB, VQ>::kTotal;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<MT, DB, VQ>, a, kmap, vmap);
}

// the (MT, DB) instances: MT = 16-row tiles of a segment's rows, DB = d / 64
// The merge launch that follows every attention launch: CTA (segment, row i)
// merges row i of the segment's n chunk partials (segments of one chunk were
// finished by the attention kernel, except for the Turbo4 V formats, whose
// rows are rotated back here).  Warp w
// owns the row's columns 32 w .. 32 w + 31 (lane = column); every lane loads
// its column of all n <= 32 slots at once together with the chunks' (m, l)
// and its gate value, so the merge costs one round of loads.  The slots are
// added in slot order.  Turbo4 V rows are rotated back through shared memory
// by one warp.  Writes the attention tap, the fp16 o_proj operand and its
// group sums (warp sums added in warp order).
template <int DB, int VQ>
__global__ void __launch_bounds__(DB * 64) attn_merge_kernel(const AttnArgs a)
{
    constexpr int D = DB * 64, NW = D / 32;
    __shared__ int ub[32], nc[32], cu_slot;
    __shared__ long long pi[33], uo[33];
    __shared__ float row[D], wsum[NW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the o_proj launch may start streaming its weights at once
    pdl_launch_dependents();
    chunk_plan(a, a.attn_grid, ub, nc, pi, uo, &cu_slot);
    const long long seg = blockIdx.x / a.merge_rows;
    const int i = blockIdx.x % a.merge_rows;
    const int rb = (int)(seg % a.nrb), kh = (int)((seg / a.nrb) % a.Hk);
    const int b = (int)(seg / ((long long)a.nrb * a.Hk));
    const int n = nc[b], nrows = a.rb_nh[rb] * a.R;
    if (n == 0 || (VQ == 0 && n == 1) || i >= nrows)
        return;
    const int gqa = a.H / a.Hk;
    const int h = kh * gqa + a.rb_h0[rb] + i / a.R, m = b * a.R + i % a.R;
    const long long Ktot = (long long)a.H * D, sf = attn_slot_floats(D);
    const long long kb = (long long)m * Ktot + (long long)h * D + warp * 32 + lane;
    const float *slots = a.ws + (pi[b] + ((long long)kh * a.nrb + rb) * n) * sf;
    const float *col = slots + 2 * kAttnMaxRows + (long long)i * D + warp * 32 + lane;
    pdl_wait();                 // the chunk partials come from the attention launch
    const float mj = lane < n ? __ldcg(slots + lane * sf + i) : -INFINITY;
    const float lj = lane < n ? __ldcg(slots + lane * sf + kAttnMaxRows + i) : 0.f;
    const float gt = __ldcg(a.gate + kb);
    float v[kMaxChunks];
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j)
        v[j] = j < n ? __ldcg(col + j * sf) : 0.f;
    float M = mj;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = mj == -INFINITY ? 0.f : exp2f(mj - M);
    float L = f * lj;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j) {
        const float fj = __shfl_sync(0xffffffffu, f, j);
        if (j < n)
            acc = fmaf(fj, v[j], acc);
    }
    float o = acc * (L > 0.f ? 1.f / L : 0.f);
    if constexpr (VQ != 0) {
        // the values were attended in their Walsh-Hadamard basis: H o / sqrt(d)
        row[warp * 32 + lane] = o;
        __syncthreads();
        if (warp == 0) {
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                x[k] = k < NW ? row[lane + 32 * k] : 0.f;
            wht_warp(x, NW, lane);
#pragma unroll
            for (int k = 0; k < NW; ++k)
                row[lane + 32 * k] = x[k] * a.inv_sqrt_d;
        }
        __syncthreads();
        o = row[warp * 32 + lane];
    }
    const int c = h * D + warp * 32 + lane;
    const __half q = __float2half_rn(o * (1.f / (1.f + __expf(-gt))));
    a.x16[x16_offset(m, c, a.NT)] = q;
    if (a.tap_attn)
        a.tap_attn[kb] = o;
    // group sums of the fp16 operand: groups of gs (32, 64 or 128) columns,
    // gs / 32 consecutive warps
    float t = __half2float(q);
#pragma unroll
    for (int off = 16; off; off >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0)
        wsum[warp] = t;
    __syncthreads();
    const int gs = a.group_o, wpg = gs / 32, MP = 8 * a.NT;
    if (threadIdx.x < D / gs) {
        float g = 0.f;
        for (int w = 0; w < wpg; ++w)
            g += wsum[threadIdx.x * wpg + w];
        const int c0 = h * D + threadIdx.x * gs;
        a.xsum[((long long)(c0 >> 7) * (kKU / gs) + ((c0 & 127) / gs)) * MP + m] = g;
    }
}

// The merge for a bf16 V cache when the o_proj groups are at most 64 columns:
// CTA (segment, row i, slice sl) merges columns 64 sl .. 64 sl + 63 of row i,
// whole groups, so its group sums need no other CTA.  Column by column the
// arithmetic of attn_merge_kernel (the same results bit for bit), on d / 64
// times as many CTAs, each loading that fraction of the row's partials.
template <int DB>
__global__ void __launch_bounds__(64) attn_merge_slice_kernel(const AttnArgs a)
{
    constexpr int D = DB * 64;
    __shared__ int ub[32], nc[32], cu_slot;
    __shared__ long long pi[33], uo[33];
    __shared__ float wsum[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the o_proj launch may start streaming its weights at once
    pdl_launch_dependents();
    chunk_plan(a, a.attn_grid, ub, nc, pi, uo, &cu_slot);
    const int sl = (int)(blockIdx.x % DB);
    const long long rowid = blockIdx.x / DB;
    const long long seg = rowid / a.merge_rows;
    const int i = (int)(rowid % a.merge_rows);
    const int rb = (int)(seg % a.nrb), kh = (int)((seg / a.nrb) % a.Hk);
    const int b = (int)(seg / ((long long)a.nrb * a.Hk));
    const int n = nc[b], nrows = a.rb_nh[rb] * a.R;
    if (n <= 1 || i >= nrows)
        return;
    const int gqa = a.H / a.Hk;
    const int h = kh * gqa + a.rb_h0[rb] + i / a.R, m = b * a.R + i % a.R;
    const int col0 = sl * 64 + warp * 32 + lane;           // column within the head
    const long long Ktot = (long long)a.H * D, sf = attn_slot_floats(D);
    const long long kb = (long long)m * Ktot + (long long)h * D + col0;
    const float *slots = a.ws + (pi[b] + ((long long)kh * a.nrb + rb) * n) * sf;
    const float *col = slots + 2 * kAttnMaxRows + (long long)i * D + col0;
    pdl_wait();                 // the chunk partials come from the attention launch
    const float mj = lane < n ? __ldcg(slots + lane * sf + i) : -INFINITY;
    const float lj = lane < n ? __ldcg(slots + lane * sf + kAttnMaxRows + i) : 0.f;
    const float gt = __ldcg(a.gate + kb);
    float v[kMaxChunks];
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j)
        v[j] = j < n ? __ldcg(col + j * sf) : 0.f;
    float M = mj;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = mj == -INFINITY ? 0.f : exp2f(mj - M);
    float L = f * lj;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j) {
        const float fj = __shfl_sync(0xffffffffu, f, j);
        if (j < n)
            acc = fmaf(fj, v[j], acc);
    }
    const float o = acc * (L > 0.f ? 1.f / L : 0.f);
    const int c = h * D + col0;
    const __half q = __float2half_rn(o * (1.f / (1.f + __expf(-gt))));
    a.x16[x16_offset(m, c, a.NT)] = q;
    if (a.tap_attn)
        a.tap_attn[kb] = o;
    // group sums of the fp16 operand: groups of gs (32 or 64) columns, the
    // slice's warps added in warp order
    float t = __half2float(q);
#pragma unroll
    for (int off = 16; off; off >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0)
        wsum[warp] = t;
    __syncthreads();
    const int gs = a.group_o, wpg = gs / 32, MP = 8 * a.NT;
    if (threadIdx.x < 64 / gs) {
        float g = 0.f;
        for (int w = 0; w < wpg; ++w)
            g += wsum[threadIdx.x * wpg + w];
        const int c0 = h * D + sl * 64 + threadIdx.x * gs;
        a.xsum[((long long)(c0 >> 7) * (kKU / gs) + ((c0 & 127) / gs)) * MP + m] = g;
    }
}

template <int DB>
static cudaError_t launch_attn_merge_slice_t(const AttnArgs &a, int segments, bool pdl,
                                             cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(segments * a.merge_rows * DB);
    cfg.blockDim = dim3(64);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_slice_kernel<DB>, a);
}

template <int DB, int VQ>
static cudaError_t launch_attn_merge_t(const AttnArgs &a, int segments, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(segments * a.merge_rows);
    cfg.blockDim = dim3(DB * 64);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel<DB, VQ>, a);
}

#define GATTN_ATTN_INSTANCES(X)                                                                    \
    X(1, 1) X(2, 1) X(1, 2) X(2, 2) X(1, 4) X(2, 4)

}  // namespace gattn
