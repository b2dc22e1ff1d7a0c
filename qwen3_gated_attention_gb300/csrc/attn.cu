// attn.cu -- causal GQA decode / verify attention over a bf16 KV cache.
//
// For every (sequence b, KV head kh, row block rb) segment the rows are the
// R new rows of the row block's query heads (one KV group, or one chunk of it
// when the verify head-chunk plan is on), and the keys are cache positions
// [0, cache_pos[b] + R).  Segments are cut into 16-token units and all units
// of all segments are split stream-K over the grid, so variable lengths
// balance across SMs.  One producer warp streams K/V tiles (up to 64 tokens x
// head_dim) with 4-D TMA tensor copies (128-byte swizzle) into a two-stage
// ring; one tile read serves every query row of the segment.  Eight consumer
// warps compute S = q K^T and O += P V with bf16 mma.sync (fp32 accumulate)
// and an online softmax in the log2 domain.
//
// Each CTA writes a partial (m, l, O) per segment piece; the last CTA to
// arrive on a segment (counter, no waiting) merges the partials in a fixed
// order, applies the output gate attn * sigmoid(gate), and writes the o_proj
// operand directly in tensor-core fragment order (fp16) with its group sums.
#include "common.cuh"
#include "kernels.cuh"

namespace gattn {

// bytes of one 64-wide head_dim box of a tile (kAttnTile tokens x 128 bytes);
// a multiple of 1024 so every box starts on a 128-byte-swizzle atom
constexpr int kDBox = kAttnTile * 128;
static_assert(kDBox % 1024 == 0, "tile boxes must stay swizzle-atom aligned");

template <int MT, int DB>
struct AttnSmem {
    static constexpr int kTileBytes = DB * kDBox;             // kAttnTile tokens x d bf16
    static constexpr int kStageBytes = 2 * kTileBytes;        // K + V
    static constexpr int kQBytes = MT * 16 * DB * 64 * 2;
    static constexpr int kPBytes = MT * 16 * 128;             // rows x 64 tokens bf16
    // as many K/V stages (2 .. kAttnStages) as fit beside the rest in 227 KB
    static constexpr int kFixed = kQBytes + kPBytes + 2 * kAttnWarps * 64 * 4 + 40 * 8 +
                                  2 * kAttnStages * 8 + 256 + 1024;
    static constexpr int kFit = (227 * 1024 - kFixed) / kStageBytes;
    static constexpr int kNStages = kFit < 2 ? 2 : (kFit > kAttnStages ? kAttnStages : kFit);
    static constexpr int kStages = kNStages * kStageBytes;
    static constexpr int kQ = kStages;
    static constexpr int kP = kQ + kQBytes;
    static constexpr int kRedMax = kP + kPBytes;              // [8][64] floats
    static constexpr int kRedL = kRedMax + kAttnWarps * 64 * 4;
    static constexpr int kPrefix = kRedL + kAttnWarps * 64 * 4;   // [33] long long
    static constexpr int kBars = kPrefix + 40 * 8;
    static constexpr int kFlags = kBars + 2 * kNStages * 8;
    static constexpr int kTotal = kFlags + 256 + 1024;        // + alignment slack
};

template <int MT, int DB>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap)
{
    using L = AttnSmem<MT, DB>;
    constexpr int D = DB * 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qs = smem + L::kQ;
    uint8_t *ps = smem + L::kP;
    float *red_max = reinterpret_cast<float *>(smem + L::kRedMax);
    float *red_l = reinterpret_cast<float *>(smem + L::kRedL);
    long long *prefix = reinterpret_cast<long long *>(smem + L::kPrefix);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *empty = full + L::kNStages;
    int *flags = reinterpret_cast<int *>(smem + L::kFlags);   // [0] abort [1] last [2..] ub
    int *ub = flags + 4;                                        // units per segment of b [32]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gqa = a.H / a.Hk;

    // Dependents (the merge) may launch at once.  Before waiting for the q|k|v
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
        flags[1] = 0;
        fence_mbar_init();
    }
    if (tid < a.B) {
        const int p0 = a.cache_pos[tid];
        const bool valid = p0 >= 0 && p0 + a.R <= a.cap;
        ub[tid] = valid ? (p0 + a.R + kAttnUnit - 1) / kAttnUnit : 0;
    }
    __syncthreads();
    if (tid == 0) {
        long long acc = 0;
        for (int b = 0; b < a.B; ++b) {
            prefix[b] = acc;
            acc += (long long)ub[b] * a.Hk * a.nrb;
        }
        prefix[a.B] = acc;
    }
    __syncthreads();

    // Ranges are cut over attn_ranges(T) CTAs, each owning at least min_units
    // units (the merge kernel counts contributors by range); the remaining CTAs
    // have nothing to do.
    const long long T = prefix[a.B], c = blockIdx.x;
    const long long G = attn_ranges(T, gridDim.x, a.min_units);
    const long long beg = c < G ? sk_start(c, T, G) : T, end = c < G ? sk_start(c + 1, T, G) : T;
    volatile int *abort = flags;

    if (warp == kAttnWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && beg < end) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const uint64_t pol = l2_evict_first_policy();
            long long it = 0;
            bool stop = false, waited = false;
            for (long long pos = beg; pos < end && !stop;) {
                const Piece p = find_piece(prefix, ub, a.B, a.Hk, a.nrb, pos, end);
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
                    uint8_t *vst = kst + L::kTileBytes;
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(nun * DB * 2048 * 2));
                    for (int ui = 0; ui < nun; ++ui) {
                        const int t = (u + ui) * kAttnUnit;
#pragma unroll
                        for (int db = 0; db < DB; ++db) {
                            tensor4d_g2s(kst + db * kDBox + ui * 2048, &kmap, db * 64, t, p.kh, p.b,
                                         &full[slot], pol);
                            tensor4d_g2s(vst + db * kDBox + ui * 2048, &vmap, db * 64, t, p.kh, p.b,
                                         &full[slot], pol);
                        }
                    }
                }
                pos = p.seg_start + p.u1;
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
    pdl_wait();                 // q rows come from the q|k|v projection
    const int g = lane >> 2, cq = lane & 3;
    const int NT = a.NT, MP = 8 * NT;
    const int Ktot = a.H * D;
    long long it = 0;
    for (long long pos = beg; pos < end;) {
        const Piece p = find_piece(prefix, ub, a.B, a.Hk, a.nrb, pos, end);
        const int nh = a.rb_nh[p.rb];
        const int h0 = p.kh * gqa + a.rb_h0[p.rb];
        const int nrows = nh * a.R;
        const int p0 = a.cache_pos[p.b];
        const int Lb = p0 + a.R;

        // ---- q rows of this segment into shared memory (swizzled 16-byte chunks)
        constexpr int CH = D / 8;   // chunks per row
        for (int idx = tid; idx < MT * 16 * CH; idx += kAttnWarps * 32) {
            const int i = idx / CH, cc = idx % CH;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (i < nrows) {
                const int hl = i / a.R, r = i % a.R;
                const __nv_bfloat16 *src =
                    a.qn + (((long long)p.b * a.R + r) * a.H + h0 + hl) * D + cc * 8;
                v = *reinterpret_cast<const uint4 *>(src);
            }
            *reinterpret_cast<uint4 *>(qs + i * (D * 2) + ((cc ^ (i & 7)) << 4)) = v;
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
            uint8_t *vst = kst + L::kTileBytes;

            // positions past the sequence end hold stale memory: zero those V rows
            if (ok && t0 + ntok > Lb) {
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
            constexpr int SPLIT = MT >= 4 ? 1 : (MT >= 2 ? 2 : 4);
            float sc[MT][4];
            float scs[SPLIT][MT][4];
            const bool has_tok = ok && (warp * 8 < ntok);
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
                    ldsm_x4(kb, smem_u32(kst + (chunk >> 3) * kDBox + tok * 128 +
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
                    const bool vis = has_tok && i < nrows && t <= p0 + (i % a.R);
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
                    const uint32_t pk = pack_bf16x2(p0f, p1f);
                    l_run[mt][hr] = l_run[mt][hr] * alpha + (bf16_lo(pk) + bf16_hi(pk));
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
                                ldsm_x4_trans(r, smem_u32(vst + (chunk >> 3) * kDBox + tok * 128 +
                                                          (((chunk & 7) ^ (tok & 7)) << 4)));
                                vb[j][0] = r[0];
                                vb[j][1] = r[1];
                                vb[j + 1][0] = r[2];
                                vb[j + 1][1] = r[3];
                            } else {
                                const int chunk = nd;
                                ldsm_x2_trans(vb[j][0], vb[j][1],
                                              smem_u32(vst + (chunk >> 3) * kDBox + tok * 128 +
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
                            for (int j = 0; j < DB; ++j)
                                mma_bf16(O[mt][j], pa, vb[j][0], vb[j][1], O[mt][j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }

        // ---- partial (m, l, O) of this piece into slot seg + c (valid rows only);
        //      a separate merge kernel combines the slots of each segment
        float *part = a.ws + (p.seg + c) * (long long)attn_slot_floats(D);
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
        // red_l is reused by the next piece: keep warp 0's reads before new writes
        named_bar_sync(1, kAttnWarps * 32);
        pos = p.seg_start + p.u1;
    }
}

template <int MT, int DB>
static cudaError_t launch_attn_t(const AttnArgs &a, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, int grid, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = AttnSmem<MT, DB>::kTotal;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<MT, DB>, a, kmap, vmap);
}

int attn_smem_bytes(int MT, int DB)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return AttnSmem<mt, db>::kTotal;
    GATTN_CASE(1, 1) GATTN_CASE(2, 1) GATTN_CASE(3, 1) GATTN_CASE(4, 1)
    GATTN_CASE(1, 2) GATTN_CASE(2, 2) GATTN_CASE(3, 2) GATTN_CASE(4, 2)
    GATTN_CASE(1, 4) GATTN_CASE(2, 4) GATTN_CASE(3, 4) GATTN_CASE(4, 4)
#undef GATTN_CASE
    return -1;
}

cudaError_t attn_set_smem_limits()
{
    cudaError_t e = cudaSuccess;
#define GATTN_SET(mt, db)                                                                          \
    if (e == cudaSuccess)                                                                          \
        e = cudaFuncSetAttribute(attn_kernel<mt, db>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 AttnSmem<mt, db>::kTotal);
    GATTN_SET(1, 1) GATTN_SET(2, 1) GATTN_SET(3, 1) GATTN_SET(4, 1)
    GATTN_SET(1, 2) GATTN_SET(2, 2) GATTN_SET(3, 2) GATTN_SET(4, 2)
    GATTN_SET(1, 4) GATTN_SET(2, 4) GATTN_SET(3, 4) GATTN_SET(4, 4)
#undef GATTN_SET
    return e;
}

cudaError_t launch_attn(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap,
                        const CUtensorMap &vmap, int grid, bool pdl, cudaStream_t s)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return launch_attn_t<mt, db>(a, kmap, vmap, grid, pdl, s);
    GATTN_CASE(1, 1) GATTN_CASE(2, 1) GATTN_CASE(3, 1) GATTN_CASE(4, 1)
    GATTN_CASE(1, 2) GATTN_CASE(2, 2) GATTN_CASE(3, 2) GATTN_CASE(4, 2)
    GATTN_CASE(1, 4) GATTN_CASE(2, 4) GATTN_CASE(3, 4) GATTN_CASE(4, 4)
#undef GATTN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gattn
