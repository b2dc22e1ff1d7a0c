// fused.cu -- the whole gated-attention layer step as one persistent kernel.
//
// At decode and speculative-verify batch sizes every step of the layer moves
// megabytes but computes little, and a chain of separate launches spends most
// of its time in launch gaps and pipeline fill.  This kernel runs the step with
// one CTA per SM (cooperative launch: every CTA is resident, so CTAs may wait
// for flags that other CTAs set) and keeps HBM busy from its first cycle:
//
//   producer warp   one thread streams, in order, everything the CTA will read
//                   into one shared-memory byte ring: its q|k|v weight stages,
//                   its K/V tiles (4-D TMA), its o_proj weight stages.  Copies
//                   whose source this step writes first (K/V tiles holding the
//                   new rows, the o_proj operand) are armed in the ring at once
//                   and issued when the flag of their source is set.
//   8 consumer warps
//     A  q|k|v dequant-GEMV over a stream-K range of (row block, k unit)
//        items; each warp owns 16 rows of a 32-row unit.  Partials go to global
//        slots; the last CTA to finish an epilogue group (whole heads) sums them
//        in a fixed order, applies RMSNorm + partial RoPE, writes q (bf16), the
//        gate and the new bf16 cache rows, and sets the group's ready flag.
//     B  causal GQA attention over a stream-K range of 16-token units of all
//        (sequence, KV head, head chunk) segments, after the ready flags of the
//        segment's heads; partial (m, l, O) per piece, then a segment counter.
//     C  merge: CTA j combines the partials of o_proj k unit j (128 columns of
//        heads x head_dim) once its segments are complete, applies
//        attn * sigmoid(gate), writes the operand in fragment order with its
//        group sums and sets the unit's flag.
//     D  o_proj dequant-GEMV like A; the last CTA of a row block writes bf16 out.
//
// Every wait is bounded (kWaitLimitNs): on expiry the status word gets the
// timeout bit, a global abort flag stops the other CTAs' waits, and every CTA
// still runs to its exit.  The last CTA to exit clears the counters and flags
// for the next step.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "unpack.cuh"

namespace gattn {
namespace {

// ------------------------------------------------------------ memory order

// polling load: no ordering, no L1 (pair with fence_acq_rel_gpu once satisfied)
__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// gpu-scope release/acquire fence (cumulative: after a CTA barrier it covers
// the other threads' writes that the barrier ordered before it)
__device__ __forceinline__ void fence_acq_rel_gpu()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// orders this thread's generic-proxy global accesses with its async-proxy
// (bulk / tensor copy) accesses
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Next entry of `size` bytes in a ring of `rb` bytes, `h` being where the
// previous entry ended: entries never wrap, a tail too short for the entry is
// skipped.  Returns the entry's offset; `held` gets the bytes the entry holds
// until it is freed (its size plus any skipped tail).
__device__ __forceinline__ int ring_next(int &h, int size, int rb, int &held)
{
    int off = h;
    held = size;
    if (off + size > rb) {
        held += rb - off;
        off = 0;
    }
    h = off + size;
    if (h == rb)
        h = 0;
    return off;
}

__host__ __device__ __forceinline__ int round1k(int b) { return (b + 1023) & ~1023; }

// Bytes of one o_proj ring entry: weights, x fragments, x group sums.
__host__ __device__ __forceinline__ int o_entry_bytes(int step_o, int group_o)
{
    return round1k(step_o + 2048 + (kKU / group_o) * 32);
}

// Bytes of one K/V tile entry of nun 16-token units (K boxes, then V boxes).
__host__ __device__ __forceinline__ int kv_entry_bytes(int DB, int nun) { return 2 * DB * nun * 2048; }

// Global-memory wait (flag >= want), bounded like mbar_wait: relaxed polling
// with back-off, one acquire fence once the flag is seen.
__device__ __forceinline__ bool flag_wait(const unsigned *flag, unsigned want, unsigned *sync_abort,
                                          volatile int *abort, unsigned *status)
{
    if (ld_relaxed(flag) >= want) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        return true;
    }
    const unsigned long long t0 = global_ns();
    while (true) {
        __nanosleep(100);
        if (ld_relaxed(flag) >= want) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if (*abort || *reinterpret_cast<volatile unsigned *>(sync_abort)) {
            *abort = 1;
            return false;
        }
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
            atomicExch(sync_abort, 1u);
            return false;
        }
    }
}

// ----------------------------------------------------- projection unit rows
//
// Rows mt*16 .. mt*16+15 of one 32-row x 128-k unit against the one-tile
// (8-column) x operand: exact fp16 codes times x on the tensor cores, and per
// group y += scale * D + bias * sum(x).  The unit layout is the device tile
// layout of the projection kernel: lane t's code stream, MMA mi = 2*kstep + mt.
template <int BITS, int GROUP>
__device__ __forceinline__ void unit_rows(const uint8_t *unit, const uint2 *xf, const float *xs,
                                          int mt, int lane, float (&Y)[4])
{
    const uint8_t *sb = unit + unit_code_bytes(BITS);
    constexpr int kpg = GROUP / 16;     // k16-steps per group
    const int g = lane >> 2, c = lane & 3;
    uint32_t cw[4 * BITS];
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(unit + (i * 32 + lane) * 16);
        cw[4 * i] = v.x;
        cw[4 * i + 1] = v.y;
        cw[4 * i + 2] = v.z;
        cw[4 * i + 3] = v.w;
    }
    // two independent accumulator chains per group when the group allows it
    constexpr int SPLIT = kpg >= 2 ? 2 : 1;
    float D[SPLIT][4];
#pragma unroll
    for (int sp = 0; sp < SPLIT; ++sp)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            D[sp][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int sp = ks % SPLIT;
        uint32_t A[4];
        unpack_a<BITS>(cw, 2 * ks + mt, A);
        const uint2 b = xf[ks * 32 + lane];
        mma_f16(D[sp], A, b.x, b.y, D[sp]);
        if ((ks % kpg) == kpg - 1) {
            const int gi = ks / kpg;
            // scale/bias words of rows g + 16 mt and g + 8 + 16 mt
            const uint2 e = *reinterpret_cast<const uint2 *>(sb + (gi * 8 + g) * 16 + mt * 8);
            const float s0 = bf16_lo(e.x), b0 = bf16_hi(e.x);
            const float s1 = bf16_lo(e.y), b1 = bf16_hi(e.y);
            const float2 xv = *reinterpret_cast<const float2 *>(xs + gi * 8 + 2 * c);
            float dd[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dd[i] = D[0][i];
#pragma unroll
                for (int q = 1; q < SPLIT; ++q)
                    dd[i] += D[q][i];
#pragma unroll
                for (int q = 0; q < SPLIT; ++q)
                    D[q][i] = 0.f;
            }
            Y[0] = fmaf(s0, dd[0], fmaf(b0, xv.x, Y[0]));
            Y[1] = fmaf(s0, dd[1], fmaf(b0, xv.y, Y[1]));
            Y[2] = fmaf(s1, dd[2], fmaf(b1, xv.x, Y[2]));
            Y[3] = fmaf(s1, dd[3], fmaf(b1, xv.y, Y[3]));
        }
    }
}


// ------------------------------------------------------------ CTA state

// Shared-memory regions of one CTA (layout planned on the host by fused_plan).
struct Smem {
    uint8_t *ring;            // the byte ring
    uint8_t *xa;              // q|k|v operand slots: fragments [256] uint2 + group sums
    uint8_t *u;               // phase scratch: q / P tiles, epilogue values, merge factors
    float *red_max, *red_l;   // attention cross-warp reductions [kFW][64]
    uint64_t *full, *empty;   // [kFEntries] each
    int *flags;               // [0] abort (this CTA), [1] broadcast word
    long long *prefix;        // [kFMaxB + 1] first attention unit of each sequence
    int *ub, *cpos;           // [kFMaxB] 16-token units, cache_pos
    float *nq, *nk;           // q_norm / k_norm as fp32 [d]
    double *invf;             // RoPE inverse frequencies [rd / 2]
};

constexpr int kMiscBytes = 3840;
constexpr int kRedBytes = 2 * kFW * 64 * 4;
// merge scratch inside the phase scratch
constexpr int kMergePairs = 16;
constexpr int kMergeFct = 0;                                        // [16][kFMaxContrib] floats
constexpr int kMergeStage = kMergeFct + kMergePairs * kFMaxContrib * 4;   // [8][128] halves
constexpr int kMergeComb = kMergeStage + 8 * 128 * 2;               // [256] floats
constexpr int kMergeInfo = kMergeComb + 256 * 4;                    // [16] x 4 ints
constexpr int kMergeBytes = kMergeInfo + kMergePairs * 16;
constexpr int kXSlotBytes = 2048 + 128;

// This CTA's share of the three stream-K work lists.
struct Plan {
    int c, P;
    // every list is cut over at most as many CTAs as it has items, so each
    // participating CTA owns at least one and a row block's contributors are
    // consecutive CTAs
    long long Ta, Ga, ia0, ia1; // q|k|v items: (row block, k unit), row block major
    long long Tb, G, ub0, ub1;  // attention units, cut over G <= P CTAs
    long long To, Go, io0, io1; // o_proj items
};

// Consumer-side position in the ring: where the last entry ended, entries
// consumed.  Passed by value so that it lives in registers.
struct CRing {
    int h, e;
};

// Bytes of the raw x entry: this CTA's k units of every x row.
__host__ __device__ __forceinline__ int x_entry_bytes(int M, int ns, int esize)
{
    return round1k(M * ns * kKU * esize);
}

// ----------------------------------------------------------------- producer

// A copy armed in the ring but issued only once this step's kernel has written
// its source: K/V tiles holding the step's new rows, the o_proj operand.
struct Deferred {
    int kind;                 // 0: K/V tile, 1: o_proj operand of k unit ku
    int slot;                 // barrier pair
    uint32_t off;             // entry offset in the ring
    int b, kh, u, nun, ku;
};

__device__ __noinline__ void producer(const FusedArgs &a, const CUtensorMap *kmap,
                                      const CUtensorMap *vmap, const Smem &sm, const Plan &pl)
{
    constexpr int E = kFEntries;
    // loop invariants in registers (the asm statements below clobber memory)
    const int RB = a.ring_bytes, DB = a.d / 64;
    uint8_t *const ring = sm.ring;
    uint64_t *const full = sm.full, *const empty = sm.empty;
    volatile int *const abort = sm.flags;
    unsigned *const gabort = a.sync + 1, *const status = a.status;
    const unsigned *const rdy_a = a.sync + a.s_rdy_a, *const xo_rdy = a.sync + a.s_xo;
    const uint8_t *const wa = a.wa, *const wo = a.wo;
    const int step_a = a.step_a, step_o = a.step_o, nku_a = a.nku_a, nku_o = a.nku_o;
    const int Nq = a.Nq, Nkv = a.Nkv, d = a.d, GR = a.GR;
    const __half *const x16o = a.x16o;
    const float *const xsumo = a.xsumo;
    const int ng_o = kKU / a.group_o;
    const uint64_t pol = l2_evict_first_policy();
    int h = 0, in_use = 0, e = 0, nfree = 0;
    int held[E] = {};
    Deferred dq[E];
    int dh = 0, dt = 0;                   // deferred copies [dh, dt), in entry order
    bool dead = false;
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);

    auto aborted = [&]() -> bool {
        if (*abort || *reinterpret_cast<volatile unsigned *>(gabort)) {
            *abort = 1;
            return true;
        }
        return false;
    };
    auto give_up = [&]() {
        *abort = 1;
        atomicOr(status, kStatusTimeout);
        atomicExch(gabort, 1u);
    };
    // relaxed polls; service() fences once a source is seen ready
    auto ready = [&](const Deferred &q) -> bool {
        if (q.kind == 0)
            return ld_relaxed(rdy_a + (Nq + q.kh * d) / GR) != 0 &&
                   ld_relaxed(rdy_a + (Nq + Nkv + q.kh * d) / GR) != 0;
        return ld_relaxed(xo_rdy + q.ku) != 0;
    };
    auto issue = [&](const Deferred &q) {
        uint64_t *bar = &full[q.slot];
        uint8_t *dst = ring + q.off;
        if (q.kind == 0) {
            const int bs = q.nun * 2048;              // bytes per 64-wide box of this tile
            for (int ui = 0; ui < q.nun; ++ui) {
                const int t = (q.u + ui) * kAttnUnit;
                for (int db = 0; db < DB; ++db) {
                    tensor4d_g2s(dst + db * bs + ui * 2048, kmap, db * 64, t, q.kh, q.b, bar, pol);
                    tensor4d_g2s(dst + (DB + db) * bs + ui * 2048, vmap, db * 64, t, q.kh, q.b, bar,
                                 pol);
                }
            }
        } else {
            bulk_g2s(dst + step_o, x16o + q.ku * 1024, 2048, bar, pol);
            bulk_g2s(dst + step_o + 2048, xsumo + q.ku * ng_o * 8, ng_o * 32, bar, pol);
        }
    };
    // issue the oldest deferred copy once its source is ready (or at once when forced)
    auto service = [&](bool force) -> bool {
        if (dh == dt)
            return false;
        const Deferred &q = dq[dh & (E - 1)];
        if (!force && !ready(q))
            return false;
        fence_acq_rel_gpu();
        fence_proxy_async_global();
        issue(q);
        ++dh;
        return true;
    };
    // free the oldest entry once every consumer warp is done with it
    auto reclaim = [&]() -> bool {
        if (nfree < e && mbar_try(&empty[nfree & (E - 1)], (uint32_t)((nfree >> 5) & 1))) {
            in_use -= held[nfree & (E - 1)];
            ++nfree;
            return true;
        }
        return false;
    };
    // room for an entry holding `bytes`, and a free barrier pair
    auto make_room = [&](int bytes) -> bool {
        unsigned long long t0 = 0;
        while (in_use + bytes > RB || e - nfree >= E) {
            if (service(false) || reclaim()) {
                t0 = 0;
                continue;
            }
            if (aborted())
                return false;
            __nanosleep(32);
            const unsigned long long now = global_ns();
            if (!t0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                give_up();
                return false;
            }
        }
        return true;
    };
    // next entry: offset in the ring, or -1 when the CTA gave up
    auto take = [&](int size, uint32_t tx) -> int {
        int hb;
        const int off = ring_next(h, size, RB, hb);
        if (!make_room(hb))
            return -1;
        in_use += hb;
        held[e & (E - 1)] = hb;
        mbar_arrive_expect_tx(&full[e & (E - 1)], tx);
        return off;
    };

    const int ia0 = (int)pl.ia0, ia1 = (int)pl.ia1;
    if (ia1 > ia0) {
        // x: this CTA's k units of every row, in slot order (at most two runs)
        const int esize = a.x_f32 ? 4 : 2, K = nku_a * kKU;
        const int ns = min(ia1 - ia0, nku_a), ku0 = ia0 % nku_a;
        const int run0 = min(ns, nku_a - ku0), rowb = ns * kKU * esize;
        const int off = take(x_entry_bytes(a.M, ns, esize), (uint32_t)(a.M * rowb));
        if (off < 0) {
            dead = true;
        } else {
            const uint8_t *x = static_cast<const uint8_t *>(a.x);
            for (int m = 0; m < a.M; ++m) {
                uint8_t *dst = ring + off + m * rowb;
                const uint8_t *src = x + ((size_t)m * K) * esize;
                bulk_g2s(dst, src + (size_t)ku0 * kKU * esize, run0 * kKU * esize,
                         &full[e & (E - 1)], pol);
                if (run0 < ns)
                    bulk_g2s(dst + run0 * kKU * esize, src, (ns - run0) * kKU * esize,
                             &full[e & (E - 1)], pol);
            }
            ++e;
        }
        // A: q|k|v weight stages (item i = row block * nku + k unit = stage index)
        const int ea = round1k(step_a);
        for (int i = ia0; i < ia1 && !dead; ++i) {
            const int off2 = take(ea, (uint32_t)step_a);
            if (off2 < 0) {
                dead = true;
                break;
            }
            bulk_g2s(ring + off2, wa + (size_t)i * step_a, (uint32_t)step_a, &full[e & (E - 1)], pol);
            ++e;
        }
    }
    // B: K/V tiles of up to three 16-token units; tiles reaching this step's
    // new rows wait for the epilogue groups of their KV head
    for (long long pos = pl.ub0; pos < pl.ub1 && !dead;) {
        const Piece p = find_piece(sm.prefix, sm.ub, a.B, a.Hk, a.nrb, pos, pl.ub1);
        const int p0 = sm.cpos[p.b];
        for (int u = p.u0; u < p.u1; u += 3) {
            const int nun = min(3, p.u1 - u);
            const int bytes = kv_entry_bytes(DB, nun);
            const int off = take(bytes, (uint32_t)bytes);
            if (off < 0) {
                dead = true;
                break;
            }
            Deferred q;
            q.kind = 0;
            q.slot = e & (E - 1);
            q.off = (uint32_t)off;
            q.b = p.b;
            q.kh = p.kh;
            q.u = u;
            q.nun = nun;
            q.ku = 0;
            if ((u + nun) * kAttnUnit > p0) {
                dq[dt & (E - 1)] = q;
                ++dt;
            } else {
                issue(q);
            }
            ++e;
        }
        pos = p.seg_start + p.u1;
    }
    // D: o_proj weight stages now; their operand once the merge has written it
    const int eo = o_entry_bytes(step_o, a.group_o);
    const uint32_t otx = (uint32_t)(step_o + 2048 + ng_o * 32);
    const int io0 = (int)pl.io0, io1 = (int)pl.io1;
    for (int i = io0; i < io1 && !dead; ++i) {
        const int off = take(eo, otx);
        if (off < 0) {
            dead = true;
            break;
        }
        bulk_g2s(ring + off, wo + (size_t)i * step_o, (uint32_t)step_o, &full[e & (E - 1)], pol);
        Deferred q;
        q.kind = 1;
        q.slot = e & (E - 1);
        q.off = (uint32_t)off;
        q.b = q.kh = q.u = q.nun = 0;
        q.ku = i % nku_o;
        dq[dt & (E - 1)] = q;
        ++dt;
        ++e;
    }
    // the remaining deferred copies; after an abort they are issued regardless
    // (their sources are valid memory) so that every armed entry completes
    unsigned long long t0 = global_ns();
    while (dh < dt) {
        if (aborted()) {
            service(true);
            continue;
        }
        if (service(false) || reclaim()) {
            t0 = global_ns();
            continue;
        }
        if (global_ns() - t0 > kWaitLimitNs)
            give_up();
        __nanosleep(100);
    }
    // every copy into this CTA's shared memory lands before the CTA may exit
    // (one time limit for all of them)
    t0 = global_ns();
    for (int j = nfree; j < e; ++j)
        while (!mbar_try(&full[j & (E - 1)], (uint32_t)((j >> 5) & 1)) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
}

// -------------------------------------------------- q|k|v operand slots

// The operand fragments and group sums of every k unit of this CTA's q|k|v
// items (slot s holds k unit (ku0 + s) mod nku), from the raw x rows that the
// producer put in the ring's first entry.  fp32 x splits exactly into an fp16
// high part (column m) and low part (column M + m); bf16 x converts exactly.
__device__ __noinline__ CRing build_x_slots(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                            CRing rg)
{
    const int n = (int)(pl.ia1 - pl.ia0);
    if (n <= 0)
        return rg;
    const int ns = min(n, a.nku_a), M = a.M, Mx = a.Mx, x_f32 = a.x_f32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int esize = x_f32 ? 4 : 2, rowe = ns * kKU;     // elements per staged row
    uint8_t *const xa = sm.xa;
    int held;
    const int off = ring_next(rg.h, x_entry_bytes(M, ns, esize), a.ring_bytes, held);
    const int slot = rg.e & (kFEntries - 1);
    const bool ok = mbar_wait(&sm.full[slot], (uint32_t)((rg.e >> 5) & 1), sm.flags, a.status);
    ++rg.e;
    const uint8_t *raw = sm.ring + off;
    auto pair = [&](int col, int kl) -> uint32_t {       // fp16 values at kl, kl + 1
        __half h0 = __ushort_as_half(0), h1 = __ushort_as_half(0);
        if (ok && x_f32 && col < 2 * M) {
            const int m = col < M ? col : col - M;
            const float2 v = *reinterpret_cast<const float2 *>(raw + ((size_t)m * rowe + kl) * 4);
            h0 = __float2half_rn(v.x);
            h1 = __float2half_rn(v.y);
            if (col >= M) {
                h0 = __float2half_rn(v.x - __half2float(h0));
                h1 = __float2half_rn(v.y - __half2float(h1));
            }
        } else if (ok && !x_f32 && col < M) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(raw + ((size_t)col * rowe + kl) * 2);
            h0 = __float2half_rn(__uint_as_float(v << 16));
            h1 = __float2half_rn(__uint_as_float(v & 0xFFFF0000u));
        }
        return (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    };
    for (int idx = tid; idx < ns * 256; idx += kFW * 32) {
        const int sl = idx >> 8, t = idx & 255;
        const int kstep = t >> 5, col = (t & 31) >> 2, cq = t & 3;
        const int kl = sl * kKU + kstep * 16 + 2 * cq;
        uint2 v = make_uint2(0u, 0u);
        if (col < Mx) {
            v.x = pair(col, kl);
            v.y = pair(col, kl + 8);
        }
        *reinterpret_cast<uint2 *>(xa + (size_t)sl * kXSlotBytes + t * 8) = v;
    }
    named_bar_sync(1, kFW * 32);
    if (lane == 0)
        mbar_arrive(&sm.empty[slot]);
    // group sums: a warp per (slot, column); lane = (k16-step, quad lane) holds
    // four values, the lanes of one group are consecutive
    const int ng = kKU / a.group_a, lpg = a.group_a / 4;
    for (int q = warp; q < ns * 8; q += kFW) {
        const int sl = q >> 3, col = q & 7;
        float sum = 0.f;
        if (col < Mx) {
            const int kstep = lane >> 2, cq = lane & 3;
            const uint2 v = *reinterpret_cast<const uint2 *>(
                xa + (size_t)sl * kXSlotBytes + ((kstep * 32 + col * 4 + cq) * 8));
            const __half2 p0 = *reinterpret_cast<const __half2 *>(&v.x);
            const __half2 p1 = *reinterpret_cast<const __half2 *>(&v.y);
            sum = (__low2float(p0) + __high2float(p0)) + (__low2float(p1) + __high2float(p1));
        }
        for (int o = 1; o < lpg && o < 32; o <<= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane % lpg == 0 && lane / lpg < ng)
            reinterpret_cast<float *>(xa + (size_t)sl * kXSlotBytes + 2048)[(lane / lpg) * 8 + col] =
                sum;
    }
    return rg;
}

// ------------------------------------------------------------ epilogues

// Pieces (CTAs) that contribute to row block rb of a projection with nku k
// units, T items cut stream-K over G <= T CTAs (none of them empty).
__device__ __forceinline__ int rb_pieces(int rb, int nku, long long T, long long G, long long *cf)
{
    const long long f = sk_owner((long long)rb * nku, T, G);
    const long long l = sk_owner((long long)rb * nku + nku - 1, T, G);
    *cf = f;
    return (int)(l - f + 1);
}

// q|k|v epilogue group grp (GR rows = whole heads): final sums of the partial
// slots in CTA order, then per head: the query gets RMSNorm + partial RoPE and
// is written as bf16; the gate is written as fp32; k gets RMSNorm + partial
// RoPE and v nothing, and both are appended to the cache as bf16 rows.
__device__ __noinline__ void epilogue_a(const FusedArgs &a, const Smem &sm, const Plan &pl, int grp)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *vals = reinterpret_cast<float *>(sm.u);
    const int d = a.d, per = d >> 5, half = a.rd >> 1, heads = a.GR / d;
    const int n0g = grp * a.GR;
    for (int m = 0; m < a.M; ++m) {
        for (int r = tid; r < a.GR; r += kFW * 32) {
            const int n = n0g + r, rb = n >> 7, rr = n & 127;
            long long cf;
            const int np = rb_pieces(rb, a.nku_a, pl.Ta, pl.Ga, &cf);
            float v = 0.f;
            for (int j = 0; j < np; ++j) {
                const float *sp = a.part_a + (cf + j + rb) * 1024 + rr;
                v += __ldcg(sp + m * 128);
                if (a.x_f32)
                    v += __ldcg(sp + (m + a.M) * 128);
            }
            vals[r] = v;
            if (a.tap_y)
                a.tap_y[(long long)m * a.Na + n] = v;
        }
        named_bar_sync(1, kFW * 32);
        const int b = m / a.R, r = m % a.R;
        const int p0 = sm.cpos[b];
        const bool valid = p0 >= 0 && p0 + a.R <= a.cap;
        for (int hb = warp; hb < heads; hb += kFW) {
            const int n0 = n0g + hb * d;
            const float *hv = vals + hb * d;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = i < per ? hv[lane + 32 * i] : 0.f;
            int kind, head;    // 0 query, 1 gate, 2 k, 3 v
            if (n0 < a.Nq) {
                head = n0 / (2 * d);
                kind = ((n0 % (2 * d)) >= d) ? 1 : 0;
            } else if (n0 < a.Nq + a.Nkv) {
                head = (n0 - a.Nq) / d;
                kind = 2;
            } else {
                head = (n0 - a.Nq - a.Nkv) / d;
                kind = 3;
            }
            if (kind == 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < per)
                        a.gate[(long long)m * a.H * d + head * d + lane + 32 * i] = v[i];
                continue;
            }
            if (kind == 0 || kind == 2) {
                // RMSNorm over the head: x / sqrt(mean(x^2) + eps) * w
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    ss = fmaf(v[i], v[i], ss);
#pragma unroll
                for (int o = 16; o; o >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float inv = rsqrtf(ss / (float)d + a.eps);
                const float *nw = kind == 0 ? sm.nq : sm.nk;
                // partial rotary on dims [0, rd): pairs (j, j + rd/2) at position p0 + r
                const double pos = (double)(p0 + r);
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = lane + 32 * i;
                    o[i] = i < per ? v[i] * inv * nw[j] : 0.f;
                    if (i < per && j < a.rd) {
                        const int fi = j < half ? j : j - half;
                        const int jp = j < half ? j + half : j - half;
                        const float partner = hv[jp] * inv * nw[jp];
                        const double ang = pos * sm.invf[fi];
                        const double turns = rint(ang * 0.15915494309189535);
                        const float red = (float)fma(-turns, 6.283185307179586, ang);
                        float sn, cs;
                        __sincosf(red, &sn, &cs);   // |red| <= pi: hardware path
                        o[i] = j < half ? o[i] * cs - partner * sn : o[i] * cs + partner * sn;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = o[i];
            }
            if (kind == 0) {
                __nv_bfloat16 *q = a.qn + (((long long)b * a.R + r) * a.H + head) * d;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < per)
                        q[lane + 32 * i] = __float2bfloat16_rn(v[i]);
                continue;
            }
            if (!valid) {
                if (lane == 0)
                    atomicOr(a.status, kStatusRange);
                continue;
            }
            __nv_bfloat16 *dst = (kind == 2 ? a.kc : a.vc) + (long long)b * a.st_batch +
                                 (long long)head * a.st_head + (long long)(p0 + r) * a.st_tok;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < per)
                    dst[lane + 32 * i] = __float2bfloat16_rn(v[i]);
        }
        named_bar_sync(1, kFW * 32);
    }
    // publish: the cache rows are read next by tensor copies (async proxy)
    fence_proxy_async_global();
    named_bar_sync(1, kFW * 32);
    if (tid == 0)
        st_release(a.sync + a.s_rdy_a + grp, 1u);
}

// o_proj epilogue of row block rb: sums of the partial slots in CTA order, bf16
// out (zero rows for sequences whose position is out of the cache's range).
__device__ __noinline__ void epilogue_o(const FusedArgs &a, const Smem &sm, const Plan &pl, int rb)
{
    long long cf;
    const int np = rb_pieces(rb, a.nku_o, pl.To, pl.Go, &cf);
    for (int idx = threadIdx.x; idx < a.M * kRBR; idx += kFW * 32) {
        const int m = idx >> 7, rr = idx & 127;
        const int b = m / a.R;
        const int pb = sm.cpos[b];
        const bool valid = pb >= 0 && pb + a.R <= a.cap;
        float v = 0.f;
        if (valid)
            for (int j = 0; j < np; ++j)
                v += __ldcg(a.part_o + (cf + j + rb) * 1024 + m * 128 + rr);
        a.out[(long long)m * a.No + rb * kRBR + rr] = __float2bfloat16_rn(v);
    }
}

// End of a projection piece (this CTA's items of one row block): the warps'
// rows go to partial slot (c + rb); the last of the row block's (q|k|v: the
// epilogue group's) pieces to arrive runs the epilogue.
__device__ __noinline__ void flush_piece(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                         int mode, int rb, float y0, float y1, float y2, float y3)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, cq = lane & 3;
    const bool qkv = mode == 0;
    float *sp = (qkv ? a.part_a : a.part_o) + (long long)(pl.c + rb) * 1024;
    const int row = (warp >> 1) * 32 + (warp & 1) * 16 + g, col = 2 * cq;
    sp[col * 128 + row] = y0;
    sp[(col + 1) * 128 + row] = y1;
    sp[col * 128 + row + 8] = y2;
    sp[(col + 1) * 128 + row + 8] = y3;
    named_bar_sync(1, kFW * 32);
    if (tid == 0) {
        int grp, expected = 0;
        long long cf;
        if (qkv) {
            grp = rb * kRBR / a.GR;
            for (int q = grp * a.GR / kRBR; q < (grp + 1) * a.GR / kRBR; ++q)
                expected += rb_pieces(q, a.nku_a, pl.Ta, pl.Ga, &cf);
        } else {
            grp = rb;
            expected = rb_pieces(rb, a.nku_o, pl.To, pl.Go, &cf);
        }
        // acq_rel: releases this CTA's partials, acquires the earlier pieces'
        const unsigned old = atom_add_acq_rel(a.sync + (qkv ? a.s_cnt_a : a.s_cnt_o) + grp, 1u);
        sm.flags[1] = (old + 1 == (unsigned)expected) ? grp + 1 : 0;
    }
    named_bar_sync(1, kFW * 32);
    const int last = sm.flags[1];
    if (last) {
        if (qkv)
            epilogue_a(a, sm, pl, last - 1);
        else
            epilogue_o(a, sm, pl, last - 1);
    }
}

// A (mode 0, q|k|v) or D (mode 1, o_proj): this CTA's items in order.
template <int BITS, int GROUP>
__device__ __noinline__ CRing proj_phase(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                         CRing rg, int mode)
{
    constexpr int E = kFEntries;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = warp & 1, uw = warp >> 1;
    // loop invariants in registers (the barrier asm below clobbers memory)
    uint8_t *const ring = sm.ring;
    const uint8_t *const xa = sm.xa;
    uint64_t *const full = sm.full, *const empty = sm.empty;
    volatile int *const abort = sm.flags;
    unsigned *const status = a.status;
    const int RB = a.ring_bytes;
    const bool qkv = mode == 0;
    const int i0 = (int)(qkv ? pl.ia0 : pl.io0), i1 = (int)(qkv ? pl.ia1 : pl.io1);
    const int nku = qkv ? a.nku_a : a.nku_o;
    const int ubytes = qkv ? a.ubytes_a : a.ubytes_o;
    const int step = qkv ? a.step_a : a.step_o;
    const int eb = qkv ? round1k(a.step_a) : o_entry_bytes(a.step_o, a.group_o);
    int rb = i0 / nku, ku = i0 % nku, xslot = 0;
    float Y[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = i0; i < i1; ++i) {
        const int slot = rg.e & (E - 1);
        const uint32_t par = (uint32_t)((rg.e >> 5) & 1);
        int held;
        const int off = ring_next(rg.h, eb, RB, held);
        ++rg.e;
        const uint8_t *ent = ring + off;
        const uint8_t *xsl = qkv ? xa + xslot * kXSlotBytes : ent + step;
        if (mbar_wait(&full[slot], par, abort, status))
            unit_rows<BITS, GROUP>(ent + uw * ubytes, reinterpret_cast<const uint2 *>(xsl),
                                   reinterpret_cast<const float *>(xsl + 2048), mt, lane, Y);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
        if (++xslot == nku)
            xslot = 0;
        if (++ku == nku || i + 1 == i1) {
            flush_piece(a, sm, pl, mode, rb, Y[0], Y[1], Y[2], Y[3]);
            Y[0] = Y[1] = Y[2] = Y[3] = 0.f;
        }
        if (ku == nku) {
            ku = 0;
            ++rb;
        }
    }
    return rg;
}

__device__ CRing proj_phase_any(const FusedArgs &a, const Smem &sm, const Plan &pl, CRing rg,
                                int mode)
{
    const int bits = mode == 0 ? a.bits_a : a.bits_o, group = mode == 0 ? a.group_a : a.group_o;
#define GATTN_PHASE(B_, G_)                                                                        \
    case (B_) * 256 + (G_):                                                                        \
        return proj_phase<B_, G_>(a, sm, pl, rg, mode);
    switch (bits * 256 + group) {
        GATTN_PHASE(2, 32) GATTN_PHASE(2, 64) GATTN_PHASE(2, 128)
        GATTN_PHASE(3, 32) GATTN_PHASE(3, 64) GATTN_PHASE(3, 128)
        GATTN_PHASE(4, 32) GATTN_PHASE(4, 64) GATTN_PHASE(4, 128)
        GATTN_PHASE(5, 32) GATTN_PHASE(5, 64) GATTN_PHASE(5, 128)
        GATTN_PHASE(6, 32) GATTN_PHASE(6, 64) GATTN_PHASE(6, 128)
        GATTN_PHASE(8, 32) GATTN_PHASE(8, 64) GATTN_PHASE(8, 128)
    default:
        return rg;
    }
#undef GATTN_PHASE
}

// ---------------------------------------------------------------- attention

// B: this CTA's pieces of the attention segments.  Per piece the query rows
// (nh heads x R rows of one KV group) are read once their epilogue groups are
// ready; per K/V tile S = q K^T and O += P V run on bf16 mma.sync with an
// online softmax in the log2 domain; the piece's partial (m, l, O) goes to
// slot (segment + c) and the segment's counter is raised.
template <int MT, int DB>
__device__ __noinline__ CRing attn_phase(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                         CRing rg)
{
    constexpr int D = DB * 64;
    constexpr int E = kFEntries;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, cq = lane & 3;
    // loop invariants in registers (the barrier asm below clobbers memory)
    volatile int *const abort = sm.flags;
    unsigned *const status = a.status;
    uint8_t *const ring = sm.ring;
    uint64_t *const full = sm.full, *const empty = sm.empty;
    uint8_t *const qs = sm.u;
    uint8_t *const ps = sm.u + MT * 16 * D * 2;
    float *const red_max = sm.red_max, *const red_l = sm.red_l;
    const long long *const prefix = sm.prefix;
    const int *const ubp = sm.ub, *const cpos = sm.cpos;
    const int R = a.R, H = a.H, B = a.B, Hk = a.Hk, nrb = a.nrb, gqa = a.gqa, RB = a.ring_bytes;
    const int d2 = 2 * a.d, GR = a.GR;
    const float scale_log2 = a.scale_log2;
    const __nv_bfloat16 *const qn = a.qn;
    float *const ws = a.ws;
    unsigned *const rdy_a = a.sync + a.s_rdy_a, *const seg_cnt = a.sync + a.s_seg;
    unsigned *const gabort = a.sync + 1;
    const long long c = pl.c, ub1 = pl.ub1;
    for (long long pos = pl.ub0; pos < ub1;) {
        const Piece p = find_piece(prefix, ubp, B, Hk, nrb, pos, ub1);
        const int nh = a.rb_nh[p.rb];
        const int h0 = p.kh * gqa + a.rb_h0[p.rb];
        const int nrows = nh * R;
        const int p0 = cpos[p.b];
        const int Lb = p0 + R;

        // ---- the segment's query rows, once their epilogue groups are done
        if (tid == 0)
            for (int h = h0; h < h0 + nh; ++h)
                if (!flag_wait(rdy_a + (h * d2) / GR, 1u, gabort, abort, status))
                    break;
        named_bar_sync(1, kFW * 32);
        constexpr int CH = D / 8;   // 16-byte chunks per row
        for (int idx = tid; idx < MT * 16 * CH; idx += kFW * 32) {
            const int i = idx / CH, cc = idx % CH;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (i < nrows) {
                const int hl = i / R, r = i % R;
                const __nv_bfloat16 *src = qn + (((long long)p.b * R + r) * H + h0 + hl) * D + cc * 8;
                v = __ldcg(reinterpret_cast<const uint4 *>(src));
            }
            *reinterpret_cast<uint4 *>(qs + i * (D * 2) + ((cc ^ (i & 7)) << 4)) = v;
        }
        named_bar_sync(1, kFW * 32);

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

        for (int u = p.u0; u < p.u1; u += 3) {
            const int nun = min(3, p.u1 - u);
            const int ntok = nun * kAttnUnit;
            const int t0 = u * kAttnUnit;
            const int slot = rg.e & (E - 1);
            const uint32_t ph = (uint32_t)((rg.e >> 5) & 1);
            int held;
            const int off = ring_next(rg.h, kv_entry_bytes(DB, nun), RB, held);
            ++rg.e;
            const bool ok = mbar_wait(&full[slot], ph, abort, status);
            const int bs = nun * 2048;          // bytes per 64-wide box of this tile
            uint8_t *kst = ring + off;
            uint8_t *vst = kst + DB * bs;

            // positions past the sequence end hold stale memory: zero those V rows
            if (ok && t0 + ntok > Lb) {
                const int first = Lb - t0 > 0 ? Lb - t0 : 0;
                for (int idx = tid; idx < (ntok - first) * DB * 8; idx += kFW * 32) {
                    const int row = first + idx / (DB * 8), rest = idx % (DB * 8);
                    const int db = rest >> 3, cc = rest & 7;
                    *reinterpret_cast<uint4 *>(vst + db * bs + row * 128 + cc * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                // the slot is refilled by tensor copies later: order these writes first
                fence_proxy_async_smem();
            }

            // ---- S = q K^T for this warp's 8 tokens, SPLIT independent chains
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
                    ldsm_x4(kb, smem_u32(kst + (chunk >> 3) * bs + tok * 128 +
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
                    const bool vis = has_tok && i < nrows && t <= p0 + (i % R);
                    sc[mt][e] = vis ? sc[mt][e] * scale_log2 : -INFINITY;
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
            named_bar_sync(1, kFW * 32);
            // ---- online softmax update, P to shared memory
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = mt * 16 + g + 8 * hr;
                    float tmax = -INFINITY;
#pragma unroll
                    for (int w2 = 0; w2 < kFW; ++w2)
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
            named_bar_sync(1, kFW * 32);
            // ---- O += P V for this warp's head_dim slice
            if (ok) {
#pragma unroll
                for (int kt = 0; kt < 3; ++kt) {
                    if (kt * 16 < ntok) {
                        const int tok = kt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                        uint32_t vb[DB][2];
#pragma unroll
                        for (int j = 0; j < DB; j += 2) {
                            const int nd = warp * DB + j;
                            if (j + 1 < DB) {
                                const int chunk = nd + (lane >> 4);
                                uint32_t r4[4];
                                ldsm_x4_trans(r4, smem_u32(vst + (chunk >> 3) * bs + tok * 128 +
                                                           (((chunk & 7) ^ (tok & 7)) << 4)));
                                vb[j][0] = r4[0];
                                vb[j][1] = r4[1];
                                vb[j + 1][0] = r4[2];
                                vb[j + 1][1] = r4[3];
                            } else {
                                const int chunk = nd;
                                ldsm_x2_trans(vb[j][0], vb[j][1],
                                              smem_u32(vst + (chunk >> 3) * bs + tok * 128 +
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

        // ---- partial (m, l, O) of this piece into slot segment + c (valid rows)
        float *part = ws + (p.seg + c) * (long long)attn_slot_floats(D);
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
        named_bar_sync(1, kFW * 32);
        if (warp == 0 && cq == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = mt * 16 + g + 8 * hr;
                    float l = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kFW; ++w2)
                        l += red_l[w2 * 64 + i];
                    part[i] = m_run[mt][hr];
                    part[kAttnMaxRows + i] = l;
                }
        }
        named_bar_sync(1, kFW * 32);
        if (tid == 0)
            atom_add_acq_rel(seg_cnt + p.seg, 1u);
        pos = p.seg_start + p.u1;
    }
    return rg;
}

__device__ CRing attn_phase_any(const FusedArgs &a, const Smem &sm, const Plan &pl, CRing rg)
{
    const int DB = a.d / 64;
#define GATTN_ATT(MT_, DB_)                                                                        \
    case (MT_) * 8 + (DB_):                                                                        \
        return attn_phase<MT_, DB_>(a, sm, pl, rg);
    switch (a.MT * 8 + DB) {
        GATTN_ATT(1, 1) GATTN_ATT(2, 1) GATTN_ATT(3, 1) GATTN_ATT(4, 1)
        GATTN_ATT(1, 2) GATTN_ATT(2, 2) GATTN_ATT(3, 2) GATTN_ATT(4, 2)
        GATTN_ATT(1, 4) GATTN_ATT(2, 4) GATTN_ATT(3, 4) GATTN_ATT(4, 4)
    default:
        return rg;
    }
#undef GATTN_ATT
}

// ------------------------------------------------------------------- merge

// C: o_proj k unit j = operand columns [128 j, 128 j + 128) of heads x head_dim.
// Per (row m, head h) pair the contributors of h's segment left m_c, l_c and
// O_c; with M = max m_c, attn = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
// The factors 2^(m_c - M) / L are formed once per pair (a warp over the
// contributors), then threads own columns so each partial row is one coalesced
// read.  a = attn * sigmoid(gate) goes to the operand in fragment order with
// its group sums, and the unit's flag is set.
__device__ __noinline__ void merge_unit(const FusedArgs &a, const Smem &sm, const Plan &pl, int j)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *fct = reinterpret_cast<float *>(sm.u + kMergeFct);
    __half *stage = reinterpret_cast<__half *>(sm.u + kMergeStage);
    float *comb = reinterpret_cast<float *>(sm.u + kMergeComb);
    int *info = reinterpret_cast<int *>(sm.u + kMergeInfo);   // [pair]: seg, row, first, count
    volatile int *abort = sm.flags;
    const int d = a.d, k0 = j * kKU;
    const int ha = k0 / d, hb = (k0 + kKU - 1) / d, nhu = hb - ha + 1;
    const int npairs = a.M * nhu;
    const int slotf = attn_slot_floats(d);
    if (tid < npairs) {
        const int m = tid / nhu, h = ha + tid % nhu;
        const int b = m / a.R, r = m % a.R;
        const int kh = h / a.gqa, hl = h % a.gqa;
        int rbi = 0;
        while (rbi + 1 < a.nrb && a.rb_h0[rbi + 1] <= hl)
            ++rbi;
        const long long seg = ((long long)b * a.Hk + kh) * a.nrb + rbi;
        const long long U = sm.ub[b];
        int cf = 0, n = 0;
        if (U > 0) {
            const long long s0 = sm.prefix[b] + (long long)(kh * a.nrb + rbi) * U;
            const long long f = sk_owner(s0, pl.Tb, pl.G), l = sk_owner(s0 + U - 1, pl.Tb, pl.G);
            cf = (int)f;
            n = (int)(l - f + 1);
        }
        info[tid * 4 + 0] = (int)seg;
        info[tid * 4 + 1] = (hl - a.rb_h0[rbi]) * a.R + r;
        info[tid * 4 + 2] = cf;
        info[tid * 4 + 3] = n;
    }
    named_bar_sync(1, kFW * 32);
    if (tid == 0) {
        bool ok = true;
        for (int q = 0; q < npairs && ok; ++q)
            ok = flag_wait(a.sync + a.s_seg + info[q * 4], (unsigned)info[q * 4 + 3], a.sync + 1,
                           abort, a.status);
        for (int h = ha; h <= hb && ok; ++h)      // the gate rows of the unit's heads
            ok = flag_wait(a.sync + a.s_rdy_a + (h * 2 * d + d) / a.GR, 1u, a.sync + 1, abort,
                           a.status);
    }
    named_bar_sync(1, kFW * 32);

    // ---- per pair: 2^(m_c - M) / L for every contributor
    constexpr int kPerLane = kFMaxContrib / 32;
    for (int q = warp; q < npairs; q += kFW) {
        const int seg = info[q * 4], i = info[q * 4 + 1], cf = info[q * 4 + 2], n = info[q * 4 + 3];
        const float *base = a.ws + ((long long)seg + cf) * slotf;
        float mv[kPerLane], lv[kPerLane];
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) {
            const int c = lane + 32 * u;
            mv[u] = c < n ? __ldcg(base + (long long)c * slotf + i) : -INFINITY;
            lv[u] = c < n ? __ldcg(base + (long long)c * slotf + kAttnMaxRows + i) : 0.f;
            mx = fmaxf(mx, mv[u]);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float L = 0.f;
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) {
            mv[u] = mv[u] == -INFINITY ? 0.f : exp2f(mv[u] - mx);
            L = fmaf(mv[u], lv[u], L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            L += __shfl_xor_sync(0xffffffffu, L, o);
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) {
            const int c = lane + 32 * u;
            if (c < n)
                fct[q * kFMaxContrib + c] = mv[u] * inv;
        }
    }
    named_bar_sync(1, kFW * 32);

    // ---- per column: sum of the weighted partial rows, gate, fp16 operand
    const int T = a.M * kKU;
    const int split = T >= kFW * 32 ? 1 : (kFW * 32) / T;
    auto finish = [&](int task, float o) {
        const int m = task >> 7, kk = task & 127, k = k0 + kk;
        const float gt = __ldcg(a.gate + (long long)m * a.H * d + k);
        const float gated = o * (1.f / (1.f + __expf(-gt)));
        stage[m * kKU + kk] = __float2half_rn(gated);
        if (a.tap_attn)
            a.tap_attn[(long long)m * a.H * d + k] = o;
    };
    for (int task = tid / split; task < T; task += (kFW * 32) / split) {
        const int part = tid % split;
        const int m = task >> 7, kk = task & 127, k = k0 + kk;
        const int h = k / d, dc = k - h * d;
        const int q = m * nhu + (h - ha);
        const int seg = info[q * 4], i = info[q * 4 + 1], cf = info[q * 4 + 2], n = info[q * 4 + 3];
        const float *base =
            a.ws + ((long long)seg + cf) * slotf + 2 * kAttnMaxRows + (long long)i * d + dc;
        const float *f = fct + q * kFMaxContrib;
        float acc = 0.f;
        int c = part;
        for (; c + 7 * split < n; c += 8 * split) {     // eight loads in flight
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = __ldcg(base + (long long)(c + u * split) * slotf);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                acc = fmaf(f[c + u * split], v[u], acc);
        }
        for (; c < n; c += split)
            acc = fmaf(f[c], __ldcg(base + (long long)c * slotf), acc);
        if (split == 1)
            finish(task, acc);
        else
            comb[tid] = acc;
    }
    if (split > 1) {
        named_bar_sync(1, kFW * 32);
        if (tid % split == 0 && tid / split < T) {
            float o = 0.f;
            for (int s2 = 0; s2 < split; ++s2)
                o += comb[tid + s2];
            finish(tid / split, o);
        }
    }
    named_bar_sync(1, kFW * 32);

    // ---- operand fragments (thread = (k16-step, lane)) and group sums
    {
        const int kstep = tid >> 5, col = lane >> 2, cq = lane & 3;
        const int kb = kstep * 16 + 2 * cq;
        uint2 v = make_uint2(0u, 0u);
        if (col < a.M) {
            const __half *sr = stage + col * kKU;
            v.x = (uint32_t)__half_as_ushort(sr[kb]) | ((uint32_t)__half_as_ushort(sr[kb + 1]) << 16);
            v.y = (uint32_t)__half_as_ushort(sr[kb + 8]) |
                  ((uint32_t)__half_as_ushort(sr[kb + 9]) << 16);
        }
        reinterpret_cast<uint2 *>(a.x16o + (long long)j * 1024)[tid] = v;
    }
    const int ng = kKU / a.group_o;
    for (int q = warp; q < ng * 8; q += kFW) {
        const int gi = q >> 3, col = q & 7;
        float s = 0.f;
        if (col < a.M)
            for (int k = lane; k < a.group_o; k += 32)
                s += __half2float(stage[col * kKU + gi * a.group_o + k]);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0)
            a.xsumo[((long long)j * ng + gi) * 8 + col] = s;
    }
    // publish: the operand is read next by bulk copies (async proxy)
    fence_proxy_async_global();
    named_bar_sync(1, kFW * 32);
    if (tid == 0)
        st_release(a.sync + a.s_xo + j, 1u);
}

}  // namespace

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kFThreads, 1)
    fused_kernel(const __grid_constant__ FusedArgs a, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem sm;
    sm.ring = base;
    sm.xa = base + a.off_x;
    sm.u = base + a.off_u;
    sm.red_max = reinterpret_cast<float *>(base + a.off_red);
    sm.red_l = sm.red_max + kFW * 64;
    uint8_t *misc = base + a.off_misc;
    sm.full = reinterpret_cast<uint64_t *>(misc);
    sm.empty = sm.full + kFEntries;
    sm.flags = reinterpret_cast<int *>(misc + 512);
    sm.prefix = reinterpret_cast<long long *>(misc + 576);
    sm.ub = reinterpret_cast<int *>(misc + 656);
    sm.cpos = reinterpret_cast<int *>(misc + 688);
    sm.nq = reinterpret_cast<float *>(misc + 768);
    sm.nk = reinterpret_cast<float *>(misc + 1792);
    sm.invf = reinterpret_cast<double *>(misc + 2816);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kFEntries; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kFW);
        }
        sm.flags[0] = sm.flags[1] = sm.flags[2] = 0;
        fence_mbar_init();
    }
    if (tid < a.B) {
        const int p0 = a.cache_pos[tid];
        const bool valid = p0 >= 0 && p0 + a.R <= a.cap;
        sm.cpos[tid] = p0;
        sm.ub[tid] = valid ? (p0 + a.R + kAttnUnit - 1) / kAttnUnit : 0;
    }
    for (int j = tid; j < a.d; j += kFThreads) {
        sm.nq[j] = __uint_as_float((uint32_t)a.q_norm[j] << 16);
        sm.nk[j] = __uint_as_float((uint32_t)a.k_norm[j] << 16);
    }
    for (int j = tid; j < a.rd / 2; j += kFThreads)
        sm.invf[j] = a.inv_freq[j];
    __syncthreads();
    if (tid == 0) {
        long long acc = 0;
        for (int b = 0; b < a.B; ++b) {
            sm.prefix[b] = acc;
            acc += (long long)sm.ub[b] * a.Hk * a.nrb;
        }
        sm.prefix[a.B] = acc;
    }
    __syncthreads();

    Plan pl;
    pl.c = blockIdx.x;
    pl.P = gridDim.x;
    pl.Ta = (long long)a.nrb_a * a.nku_a;
    pl.Ga = pl.Ta < pl.P ? pl.Ta : pl.P;
    pl.ia0 = pl.c < pl.Ga ? sk_start(pl.c, pl.Ta, pl.Ga) : pl.Ta;
    pl.ia1 = pl.c < pl.Ga ? sk_start(pl.c + 1, pl.Ta, pl.Ga) : pl.Ta;
    pl.Tb = sm.prefix[a.B];
    pl.G = attn_ranges(pl.Tb, pl.P, a.min_units);
    pl.ub0 = pl.c < pl.G ? sk_start(pl.c, pl.Tb, pl.G) : pl.Tb;
    pl.ub1 = pl.c < pl.G ? sk_start(pl.c + 1, pl.Tb, pl.G) : pl.Tb;
    pl.To = (long long)a.nrb_o * a.nku_o;
    pl.Go = pl.To < pl.P ? pl.To : pl.P;
    pl.io0 = pl.c < pl.Go ? sk_start(pl.c, pl.To, pl.Go) : pl.To;
    pl.io1 = pl.c < pl.Go ? sk_start(pl.c + 1, pl.To, pl.Go) : pl.To;

    if (warp == kFW) {
        if (lane == 0)
            producer(a, &kmap, &vmap, sm, pl);
        __syncwarp();
    } else {
        CRing rg{0, 0};
        rg = build_x_slots(a, sm, pl, rg);
        named_bar_sync(1, kFW * 32);
        rg = proj_phase_any(a, sm, pl, rg, 0);
        rg = attn_phase_any(a, sm, pl, rg);
        for (int j = pl.c; j < a.nku_o; j += pl.P)
            merge_unit(a, sm, pl, j);
        rg = proj_phase_any(a, sm, pl, rg, 1);
    }

    // the last CTA out clears the step's counters and flags
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atom_add_acq_rel(a.sync, 1u);
        sm.flags[2] = (old + 1 == gridDim.x) ? 1 : 0;
    }
    __syncthreads();
    if (sm.flags[2]) {
        for (int i = 1 + tid; i < a.nsync; i += kFThreads)
            a.sync[i] = 0u;
        __syncthreads();
        if (tid == 0) {
            fence_acq_rel_gpu();
            a.sync[0] = 0u;
        }
    }
}

// -------------------------------------------------------------------- host

bool fused_plan(FusedArgs &a, int num_sms, int max_smem)
{
    if (num_sms + 1 > kFMaxContrib || a.d % 64 || a.d > 256 || a.d == 192)
        return false;
    const long long Ta = (long long)a.nrb_a * a.nku_a;
    const long long per = (Ta + num_sms - 1) / num_sms;
    a.xslots = (int)std::min<long long>(a.nku_a, std::max<long long>(per, 1));
    a.xslot_bytes = kXSlotBytes;
    const int DB = a.d / 64;
    const int attn_u = a.MT * 16 * a.d * 2 + a.MT * 16 * 128;
    int u = std::max(std::max(attn_u, a.GR * 4), kMergeBytes);
    u = (u + 127) & ~127;
    const int xbytes = (a.xslots * kXSlotBytes + 127) & ~127;
    const int fixed = xbytes + u + kRedBytes + kMiscBytes + 1024;
    const int ring = (max_smem - fixed) & ~1023;
    const int need = std::max(std::max(round1k(a.step_a), kv_entry_bytes(DB, 3)),
                              std::max(o_entry_bytes(a.step_o, a.group_o),
                                       x_entry_bytes(a.M, a.xslots, a.x_f32 ? 4 : 2)));
    if (ring < 2 * need)
        return false;
    a.ring_bytes = ring;
    a.off_x = ring;
    a.off_u = ring + xbytes;
    a.off_red = a.off_u + u;
    a.off_misc = a.off_red + kRedBytes;
    a.smem_bytes = a.off_misc + kMiscBytes + 1024;
    return a.smem_bytes <= max_smem;
}

cudaError_t fused_set_smem_limits(int bytes)
{
    return cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t fused_occupancy(int smem, int *blocks_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fused_kernel, kFThreads,
                                                         smem);
}

cudaError_t launch_fused(const FusedArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         int grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = a.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_kernel, a, kmap, vmap);
}

}  // namespace gattn
