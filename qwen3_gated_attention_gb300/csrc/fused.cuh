// fused.cuh -- the whole gated-attention layer step as one persistent kernel.
//
// One CTA per SM (cooperative launch: every CTA is resident, so CTAs may wait
// on counters that other CTAs raise), every phase inlined into one kernel per
// configuration:
//
//   producer warp   one thread streams, in order, everything the CTA reads into
//                   one shared-memory byte ring: x, its q|k|v weight stages,
//                   its K/V tiles (4-D TMA), its o_proj weight stages.  Nothing
//                   it copies is written by the kernel, so nothing waits.
//   8 consumer warps
//     A  q|k|v dequant-GEMV over a stream-K range of (row block, k unit) items;
//        each warp owns 16 rows of a 32-row unit.  Partials go to global slots
//        and each epilogue group (whole heads) counts its pieces.
//     B  causal GQA attention over a stream-K range of 16-token units of all
//        (sequence, KV head, head chunk) segments.  Once the counts of its
//        heads are complete, a CTA sums the q partials of its query rows
//        itself (RMSNorm + partial RoPE into the q tile); the CTA holding the
//        new rows also forms the new K/V rows, patches them into its loaded
//        tile and appends them to the cache.  Partial (m, l, O) per piece, then
//        a segment counter.
//     C  merge: every CTA merges the attention partials of the o_proj k units
//        its items use (gate from the q|k|v partials), into its own x slots.
//     D  o_proj dequant-GEMV over (k unit, row block) items, one partial slot
//        each; the last item of a row block sums its k units and writes bf16.
//
// Every wait is bounded (kWaitLimitNs): on expiry the status word gets the
// timeout bit, a global abort flag stops the other CTAs' waits, and every CTA
// still runs to its exit.  The last CTA to exit clears the counters for the
// next step.
#pragma once

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

// Bytes of one o_proj ring entry (weights only: the operand is merged in place).
__host__ __device__ __forceinline__ int o_entry_bytes(int step_o) { return round1k(step_o); }

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
// group y += scale * D + bias * sum(x).  sum(x) comes from one more MMA per
// k16-step with an all-ones A fragment: every row of its result holds the
// column sums, so each lane gets exactly the sums of its own two columns.  The
// unit layout is the device tile layout of the projection kernel: lane t's
// code stream, MMA mi = 2*kstep + mt.
template <int BITS, int GROUP, int MTILE>
__device__ __forceinline__ void unit_rows(const uint8_t *unit, const uint2 *xf, int lane,
                                          float (&Y)[4])
{
    constexpr int mt = MTILE;   // compile time: every code-word index is static
    const uint8_t *sb = unit + unit_code_bytes(BITS);
    constexpr int kpg = GROUP / 16;     // k16-steps per group
    const int g = lane >> 2;
    const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
    uint32_t cw[4 * BITS];
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(unit + (i * 32 + lane) * 16);
        cw[4 * i] = v.x;
        cw[4 * i + 1] = v.y;
        cw[4 * i + 2] = v.z;
        cw[4 * i + 3] = v.w;
    }
    uint2 xb[8];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        xb[ks] = xf[ks * 32 + lane];
    // two independent accumulator chains per group (k16-steps alternate)
    constexpr int SPLIT = kpg >= 2 ? 2 : 1;
    float D[SPLIT][4], S[SPLIT][4];
#pragma unroll
    for (int q = 0; q < SPLIT; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            D[q][i] = S[q][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int q = ks % SPLIT;
        uint32_t A[4];
        unpack_a<BITS>(cw, 2 * ks + mt, A);
        mma_f16(D[q], A, xb[ks].x, xb[ks].y, D[q]);
        mma_f16(S[q], ones, xb[ks].x, xb[ks].y, S[q]);
        if ((ks % kpg) == kpg - 1) {
            const int gi = ks / kpg;
            // scale/bias words of rows g + 16 mt and g + 8 + 16 mt
            const uint2 e = *reinterpret_cast<const uint2 *>(sb + (gi * 8 + g) * 16 + mt * 8);
            const float s0 = bf16_lo(e.x), b0 = bf16_hi(e.x);
            const float s1 = bf16_lo(e.y), b1 = bf16_hi(e.y);
            float dd[4], ss[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dd[i] = D[0][i];
                ss[i] = S[0][i];
#pragma unroll
                for (int r = 1; r < SPLIT; ++r) {
                    dd[i] += D[r][i];
                    ss[i] += S[r][i];
                }
#pragma unroll
                for (int r = 0; r < SPLIT; ++r)
                    D[r][i] = S[r][i] = 0.f;
            }
            Y[0] = fmaf(s0, dd[0], fmaf(b0, ss[0], Y[0]));
            Y[1] = fmaf(s0, dd[1], fmaf(b0, ss[1], Y[1]));
            Y[2] = fmaf(s1, dd[2], fmaf(b1, ss[0], Y[2]));
            Y[3] = fmaf(s1, dd[3], fmaf(b1, ss[1], Y[3]));
        }
    }
}

// ------------------------------------------------------------ CTA state

// Shared-memory regions of one CTA (layout planned on the host by fused_plan).
struct Smem {
    uint8_t *ring;            // the byte ring
    uint8_t *xa;              // q|k|v operand slots: fragments [256] uint2 + group sums
    uint8_t *u;               // phase scratch: q / P tiles, merge factors
    float *red_max, *red_l;   // attention cross-warp reductions [kFW][64]
    float *stg;               // per-warp staging row [kFW][256] (norm / rotary partners)
    __nv_bfloat16 *kvn;       // this step's new K and V rows [2][kFMaxB][256]
    uint64_t *full, *empty;   // [kFEntries] each
    int *flags;               // [0] abort (this CTA), [1] broadcast word
    long long *prefix;        // [kFMaxB + 1] first attention unit of each sequence
    int *ub, *cpos;           // [kFMaxB] 16-token units, cache_pos
    float *nq, *nk;           // q_norm / k_norm as fp32 [d]
    double *invf;             // RoPE inverse frequencies [rd / 2]
    uint8_t *pq;              // producer: bytes held by each live ring entry
};

constexpr int kMiscBytes = 3840 + 1536;
constexpr int kRedBytes = 2 * kFW * 64 * 4;
constexpr int kStgBytes = kFW * 256 * 4;
constexpr int kKvnBytes = 2 * kFMaxB * 256 * 2;
// merge scratch inside the phase scratch
constexpr int kMergePairs = 16;
constexpr int kMergeFct = 0;                                        // [16][kFMaxContrib] floats
constexpr int kMergeStage = kMergeFct + kMergePairs * kFMaxContrib * 4;   // [8][128] halves
constexpr int kMergeComb = kMergeStage + 8 * 128 * 2;               // [256] floats
constexpr int kMergeInfo = kMergeComb + 256 * 4;                    // [16] x 4 ints
constexpr int kMergeBytes = kMergeInfo + kMergePairs * 16;
constexpr int kXSlotBytes = 2048;

// This CTA's share of the three stream-K work lists.
struct Plan {
    int c, P;
    // every list is cut over at most as many CTAs as it has items, so each
    // participating CTA owns at least one and a row block's contributors are
    // consecutive CTAs
    long long Ta, Ga, ia0, ia1; // q|k|v items: (row block, k unit), row block major
    long long Tb, G, ub0, ub1;  // attention units, cut over G <= P CTAs
    long long To, Go, io0, io1; // o_proj items: (k unit, row block), k unit major
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

// One thread streams everything this CTA reads, in the order the consumers
// use it: x, the q|k|v weight stages, the K/V tiles (4-D tensor copies; rows
// this step appends are patched in shared memory by the consumers), the o_proj
// weight stages.  Nothing it copies is written by this kernel.
__device__ __forceinline__ void producer(const FusedArgs &a, const CUtensorMap *kmap,
                                         const CUtensorMap *vmap, const Smem &sm, const Plan &pl)
{
    constexpr int E = kFEntries;
    // loop invariants in registers (the asm statements below clobber memory)
    const int RB = a.ring_bytes, DB = a.d / 64;
    uint8_t *const ring = sm.ring;
    uint64_t *const full = sm.full, *const empty = sm.empty;
    volatile int *const abort = sm.flags;
    unsigned *const gabort = a.sync + 1, *const status = a.status;
    const uint8_t *const wa = a.wa, *const wo = a.wo;
    const int step_a = a.step_a, step_o = a.step_o, nku_a = a.nku_a, nku_o = a.nku_o;
    const uint64_t pol = l2_evict_first_policy();
    int h = 0, in_use = 0, e = 0, nfree = 0;
    // bytes each live entry holds, in shared memory (the L1 beside the ring is small)
    int *const held = reinterpret_cast<int *>(sm.pq);
    bool dead = false;
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);

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
            if (reclaim()) {
                t0 = 0;
                continue;
            }
            if (*abort || *reinterpret_cast<volatile unsigned *>(gabort)) {
                *abort = 1;
                return false;
            }
            __nanosleep(32);
            const unsigned long long now = global_ns();
            if (!t0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(status, kStatusTimeout);
                atomicExch(gabort, 1u);
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
    // B: K/V tiles of up to three 16-token units
    for (long long pos = pl.ub0; pos < pl.ub1 && !dead;) {
        const Piece p = find_piece(sm.prefix, sm.ub, a.B, a.Hk, a.nrb, pos, pl.ub1);
        for (int u = p.u0; u < p.u1; u += 3) {
            const int nun = min(3, p.u1 - u);
            const int bytes = kv_entry_bytes(DB, nun);
            const int off = take(bytes, (uint32_t)bytes);
            if (off < 0) {
                dead = true;
                break;
            }
            uint64_t *bar = &full[e & (E - 1)];
            uint8_t *dst = ring + off;
            const int bs = nun * 2048;              // bytes per 64-wide box of this tile
            for (int ui = 0; ui < nun; ++ui) {
                const int t = (u + ui) * kAttnUnit;
                for (int db = 0; db < DB; ++db) {
                    tensor4d_g2s(dst + db * bs + ui * 2048, kmap, db * 64, t, p.kh, p.b, bar, pol);
                    tensor4d_g2s(dst + (DB + db) * bs + ui * 2048, vmap, db * 64, t, p.kh, p.b, bar,
                                 pol);
                }
            }
            ++e;
        }
        pos = p.seg_start + p.u1;
    }
    // D: o_proj weight stages (item i = k unit * nrb + row block)
    const int eo = o_entry_bytes(step_o), nrb_o = a.nrb_o;
    const int io0 = (int)pl.io0, io1 = (int)pl.io1;
    for (int i = io0; i < io1 && !dead; ++i) {
        const int off = take(eo, (uint32_t)step_o);
        if (off < 0) {
            dead = true;
            break;
        }
        const int ku = i / nrb_o, rb = i - ku * nrb_o;
        bulk_g2s(ring + off, wo + ((size_t)rb * nku_o + ku) * step_o, (uint32_t)step_o,
                 &full[e & (E - 1)], pol);
        ++e;
    }
    // every copy into this CTA's shared memory lands before the CTA may exit
    // (one time limit for all of them)
    const unsigned long long t0 = global_ns();
    for (int j = nfree; j < e; ++j)
        while (!mbar_try(&full[j & (E - 1)], (uint32_t)((j >> 5) & 1)) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
}

// -------------------------------------------------- q|k|v operand slots

// The operand fragments of every k unit of this CTA's q|k|v items (slot s
// holds k unit (ku0 + s) mod nku), from the raw x rows that the producer put in
// the ring's first entry.  fp32 x splits exactly into an fp16
// high part (column m) and low part (column M + m); bf16 x converts exactly.
__device__ __forceinline__ CRing build_x_slots(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                            CRing rg)
{
    const int n = (int)(pl.ia1 - pl.ia0);
    if (n <= 0)
        return rg;
    const int ns = min(n, a.nku_a), M = a.M, Mx = a.Mx, x_f32 = a.x_f32;
    const int tid = threadIdx.x, lane = tid & 31;
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
    return rg;
}

// ------------------------------------------------- q|k|v projection values
//
// The q|k|v partials stay in their slots; whoever needs final values (the
// attention CTAs for their heads' query and new K/V rows, the merge for the
// gate) waits for the pieces of the rows' epilogue groups and sums the slots
// itself, in CTA order.  No CTA hands normalized values to another.

// Pieces (CTAs) that contribute to row block rb of the q|k|v projection (items
// cut stream-K over G <= T CTAs, none of them empty); *cf = the first.
__device__ __forceinline__ int rb_pieces(int rb, int nku, int T, int G, int *cf)
{
    const int f = (int)(((unsigned)(rb * nku + 1) * (unsigned)G - 1u) / (unsigned)T);
    const int l = (int)(((unsigned)(rb * nku + nku) * (unsigned)G - 1u) / (unsigned)T);
    *cf = f;
    return l - f + 1;
}

// Pieces of q|k|v epilogue group grp (GR rows = whole heads).
__device__ __forceinline__ unsigned group_pieces(const FusedArgs &a, const Plan &pl, int grp)
{
    unsigned n = 0;
    int cf;
    for (int q = grp * a.GR / kRBR; q < (grp + 1) * a.GR / kRBR; ++q)
        n += rb_pieces(q, a.nku_a, (int)pl.Ta, (int)pl.Ga, &cf);
    return n;
}

// Bounded wait until every piece of group grp is in its slot.
__device__ __forceinline__ bool wait_group(const FusedArgs &a, const Smem &sm, const Plan &pl, int grp)
{
    return flag_wait(a.sync + a.s_cnt_a + grp, group_pieces(a, pl, grp), a.sync + 1, sm.flags,
                     a.status);
}

// Final value of q|k|v row rb * 128 + rr, column m, whose block has np pieces
// starting at CTA cf: the partial slots summed in CTA order (each piece's low
// plane of fp32 x right after its high plane).  Up to four pieces are loaded
// together before the sum; more are added one by one.
__device__ __forceinline__ float qkv_sum(const FusedArgs &a, int rb, int rr, int m, int cf, int np)
{
    const float *sp = a.part_a + (size_t)(cf + rb) * 1024 + rr;
    const bool lo = a.x_f32 != 0;
    float hv[4], lv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        hv[j] = j < np ? __ldcg(sp + (size_t)j * 1024 + m * 128) : 0.f;
        lv[j] = (lo && j < np) ? __ldcg(sp + (size_t)j * 1024 + (m + a.M) * 128) : 0.f;
    }
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v += hv[j];
        v += lv[j];
    }
    for (int j = 4; j < np; ++j) {
        v += __ldcg(sp + (size_t)j * 1024 + m * 128);
        if (lo)
            v += __ldcg(sp + (size_t)j * 1024 + (m + a.M) * 128);
    }
    return v;
}

__device__ __forceinline__ float qkv_value(const FusedArgs &a, const Plan &pl, int n, int m)
{
    int cf;
    const int np = rb_pieces(n >> 7, a.nku_a, (int)pl.Ta, (int)pl.Ga, &cf);
    return qkv_sum(a, n >> 7, n & 127, m, cf, np);
}

// Rows n0 + lane + 32 i (i < d / 32) of column m into v, n0 a multiple of 64:
// the head spans at most three row blocks, whose piece ranges are found once;
// every row's loads are in flight together.
__device__ __forceinline__ void head_rows(const FusedArgs &a, const Plan &pl, int n0, int m,
                                          int lane, float (&v)[8])
{
    const int per = a.d >> 5, rb0 = n0 >> 7;
    int cf[3], np[3];
#pragma unroll
    for (int q = 0; q < 3; ++q)
        np[q] = rb_pieces(rb0 + q, a.nku_a, (int)pl.Ta, (int)pl.Ga, &cf[q]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = 0.f;
        if (i < per) {
            const int n = n0 + lane + 32 * i, q = (n >> 7) - rb0;
            const int c0 = q == 0 ? cf[0] : (q == 1 ? cf[1] : cf[2]);
            const int n0p = q == 0 ? np[0] : (q == 1 ? np[1] : np[2]);
            v[i] = qkv_sum(a, n >> 7, n & 127, m, c0, n0p);
        }
    }
}

// RMSNorm over the head (x / sqrt(mean(x^2) + eps) * w) and the partial rotary
// embedding on dims [0, rd) at position pos (pairs (j, j + rd/2)), in place on
// the lane-strided values v; st is this warp's staging row (partners, and the
// final values on return).
__device__ __forceinline__ void norm_rope(float (&v)[8], const FusedArgs &a, const float *w,
                                          const double *invf, double pos, float *st, int lane)
{
    const int d = a.d, per = d >> 5, rd = a.rd, half = rd >> 1;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        ss = fmaf(v[i], v[i], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / (float)d + a.eps);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < per) {
            v[i] = v[i] * inv * w[lane + 32 * i];
            st[lane + 32 * i] = v[i];
        }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int j = lane + 32 * i;
        if (i < per && j < rd) {
            const int fi = j < half ? j : j - half;
            const float partner = st[j < half ? j + half : j - half];
            const double ang = pos * invf[fi];
            const double turns = rint(ang * 0.15915494309189535);
            const float red = (float)fma(-turns, 6.283185307179586, ang);
            float sn, cs;
            __sincosf(red, &sn, &cs);   // |red| <= pi: hardware path
            v[i] = j < half ? v[i] * cs - partner * sn : v[i] * cs + partner * sn;
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < per)
            st[lane + 32 * i] = v[i];
    __syncwarp();
}

// 8 staged floats starting at st[8 c] as one 16-byte chunk of bf16.
__device__ __forceinline__ uint4 bf16_chunk(const float *st, int c)
{
    const float4 lo = *reinterpret_cast<const float4 *>(st + 8 * c);
    const float4 hi = *reinterpret_cast<const float4 *>(st + 8 * c + 4);
    return make_uint4(pack_bf16x2(lo.x, lo.y), pack_bf16x2(lo.z, lo.w), pack_bf16x2(hi.x, hi.y),
                      pack_bf16x2(hi.z, hi.w));
}

// Test taps of q|k|v group grp (raw projection values), by its last piece.
__device__ __forceinline__ void taps_a(const FusedArgs &a, const Plan &pl, int grp)
{
    for (int idx = threadIdx.x; idx < a.M * a.GR; idx += kFW * 32) {
        const int m = idx / a.GR, n = grp * a.GR + idx % a.GR;
        a.tap_y[(long long)m * a.Na + n] = qkv_value(a, pl, n, m);
    }
}

// o_proj epilogue of row block rb: the sum over k units of its items' partial
// slots (slot = item = k unit * nrb + rb), bf16 out (zero rows for sequences
// whose position is out of the cache's range).  Each element's k units are
// split between two threads (loads in flight together), combined in `comb`.
__device__ __forceinline__ void epilogue_o(const FusedArgs &a, const Smem &sm, int rb)
{
    const int nku = a.nku_o, nrb = a.nrb_o, tid = threadIdx.x;
    float *comb = reinterpret_cast<float *>(sm.u + kMergeComb);
    const int total = a.M * kRBR;
    for (int base = 0; base < total; base += kFW * 16) {
        const int idx = base + (tid >> 1), half = tid & 1;
        float v = 0.f;
        if (idx < total) {
            const int m = idx >> 7, rr = idx & 127;
            const float *sp = a.part_o + (size_t)rb * 1024 + m * 128 + rr;
            const int k0 = half ? nku / 2 : 0, k1 = half ? nku : nku / 2;
            float t[16];
            int ku = k0;
            for (; ku + 16 <= k1; ku += 16) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    t[u] = __ldcg(sp + (size_t)(ku + u) * nrb * 1024);
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    v += t[u];
            }
            for (; ku < k1; ++ku)
                v += __ldcg(sp + (size_t)ku * nrb * 1024);
        }
        comb[tid] = v;
        named_bar_sync(1, kFW * 32);
        if (half == 0 && idx < total) {
            const int m = idx >> 7, rr = idx & 127;
            const int b = m / a.R;
            const int pb = sm.cpos[b];
            const bool valid = pb >= 0 && pb + a.R <= a.cap;
            const float o = comb[tid] + comb[tid + 1];
            a.out[(long long)m * a.No + rb * kRBR + rr] = __float2bfloat16_rn(valid ? o : 0.f);
        }
        named_bar_sync(1, kFW * 32);
    }
}

// End of a q|k|v piece (this CTA's items of one row block): the warps' rows go
// to partial slot (c + rb) and the row block's epilogue group counts one more
// piece (readers wait for the count, see group_pieces).  With taps on, the
// group's last piece writes the raw values.
__device__ __forceinline__ void flush_piece(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                            int rb, float y0, float y1, float y2, float y3)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, cq = lane & 3;
    float *sp = a.part_a + (long long)(pl.c + rb) * 1024;
    const int row = (warp >> 1) * 32 + (warp & 1) * 16 + g, col = 2 * cq;
    sp[col * 128 + row] = y0;
    sp[(col + 1) * 128 + row] = y1;
    sp[col * 128 + row + 8] = y2;
    sp[(col + 1) * 128 + row + 8] = y3;
    named_bar_sync(1, kFW * 32);
    const int grp = rb * kRBR / a.GR;
    if (tid == 0) {
        // acq_rel: releases this CTA's partials (ordered before it by the barrier)
        const unsigned old = atom_add_acq_rel(a.sync + a.s_cnt_a + grp, 1u);
        sm.flags[1] = (a.tap_y && old + 1 == group_pieces(a, pl, grp)) ? 1 : 0;
    }
    if (a.tap_y) {
        named_bar_sync(1, kFW * 32);
        if (sm.flags[1])
            taps_a(a, pl, grp);
        named_bar_sync(1, kFW * 32);
    }
}

// A: this CTA's q|k|v items in order (row block major), flushed per row block.
template <int BITS, int GROUP>
__device__ __forceinline__ CRing proj_phase_a(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                              CRing rg)
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
    const int i0 = (int)pl.ia0, i1 = (int)pl.ia1;
    const int nku = a.nku_a, ubytes = a.ubytes_a, eb = round1k(a.step_a);
    int rb = i0 / nku, ku = i0 % nku, xslot = 0;
    float Y[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = i0; i < i1; ++i) {
        const int slot = rg.e & (E - 1);
        const uint32_t par = (uint32_t)((rg.e >> 5) & 1);
        int held;
        const int off = ring_next(rg.h, eb, RB, held);
        ++rg.e;
        const uint8_t *ent = ring + off;
        const uint2 *xf = reinterpret_cast<const uint2 *>(xa + xslot * kXSlotBytes);
        if (mbar_wait(&full[slot], par, abort, status)) {
            if (mt == 0)
                unit_rows<BITS, GROUP, 0>(ent + uw * ubytes, xf, lane, Y);
            else
                unit_rows<BITS, GROUP, 1>(ent + uw * ubytes, xf, lane, Y);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
        if (++xslot == nku)
            xslot = 0;
        if (++ku == nku || i + 1 == i1) {
            flush_piece(a, sm, pl, rb, Y[0], Y[1], Y[2], Y[3]);
            Y[0] = Y[1] = Y[2] = Y[3] = 0.f;
        }
        if (ku == nku) {
            ku = 0;
            ++rb;
        }
    }
    return rg;
}

// D: this CTA's o_proj items (k unit major, each its own partial slot), the
// operand of each k unit already merged into an x slot.  Row-block counters are
// raised together at the end; the last item of a row block runs its epilogue.
template <int BITS, int GROUP>
__device__ __forceinline__ CRing proj_phase_o(const FusedArgs &a, const Smem &sm, const Plan &pl,
                                              CRing rg)
{
    constexpr int E = kFEntries;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = warp & 1, uw = warp >> 1, g = lane >> 2, cq = lane & 3;
    uint8_t *const ring = sm.ring;
    const uint8_t *const xa = sm.xa;
    uint64_t *const full = sm.full, *const empty = sm.empty;
    volatile int *const abort = sm.flags;
    unsigned *const status = a.status;
    float *const part = a.part_o;
    const int RB = a.ring_bytes;
    const int i0 = (int)pl.io0, i1 = (int)pl.io1;
    const int nrb = a.nrb_o, ubytes = a.ubytes_o, eb = o_entry_bytes(a.step_o);
    const int ku0 = i0 / nrb;
    const int row = uw * 32 + mt * 16 + g, col = 2 * cq;
    for (int i = i0; i < i1; ++i) {
        const int slot = rg.e & (E - 1);
        const uint32_t par = (uint32_t)((rg.e >> 5) & 1);
        int held;
        const int off = ring_next(rg.h, eb, RB, held);
        ++rg.e;
        const uint8_t *ent = ring + off;
        const uint2 *xf = reinterpret_cast<const uint2 *>(xa + (i / nrb - ku0) * kXSlotBytes);
        float Y[4] = {0.f, 0.f, 0.f, 0.f};
        if (mbar_wait(&full[slot], par, abort, status)) {
            if (mt == 0)
                unit_rows<BITS, GROUP, 0>(ent + uw * ubytes, xf, lane, Y);
            else
                unit_rows<BITS, GROUP, 1>(ent + uw * ubytes, xf, lane, Y);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
        float *sp = part + (size_t)i * 1024;
        sp[col * 128 + row] = Y[0];
        sp[(col + 1) * 128 + row] = Y[1];
        sp[col * 128 + row + 8] = Y[2];
        sp[(col + 1) * 128 + row + 8] = Y[3];
    }
    named_bar_sync(1, kFW * 32);
    // one arrival per item on its row block; every k unit contributes one item
    if (tid < i1 - i0) {
        const int rb = (i0 + tid) % nrb;
        const unsigned old = atom_add_acq_rel(a.sync + a.s_cnt_o + rb, 1u);
        if (old + 1 == (unsigned)a.nku_o)
            atomicOr(reinterpret_cast<unsigned *>(sm.flags + 3) + (tid >> 5), 1u << (tid & 31));
    }
    named_bar_sync(1, kFW * 32);
    const int n = i1 - i0;
    for (int j = 0; j < n && j < 64; ++j)
        if (sm.flags[3 + (j >> 5)] & (1 << (j & 31)))
            epilogue_o(a, sm, (i0 + j) % nrb);
    return rg;
}

// ---------------------------------------------------------------- attention

// B: this CTA's pieces of the attention segments.  Per piece the query rows
// (nh heads x R rows of one KV group) are read once their epilogue groups are
// ready; per K/V tile S = q K^T and O += P V run on bf16 mma.sync with an
// online softmax in the log2 domain; the piece's partial (m, l, O) goes to
// slot (segment + c) and the segment's counter is raised.
template <int MT, int DB>
__device__ __forceinline__ CRing attn_phase(const FusedArgs &a, const Smem &sm, const Plan &pl,
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
    const int R = a.R, B = a.B, Hk = a.Hk, nrb = a.nrb, gqa = a.gqa, RB = a.ring_bytes;
    const int d2 = 2 * a.d, GR = a.GR, Nq = a.Nq, Nkv = a.Nkv;
    const float scale_log2 = a.scale_log2;
    float *const ws = a.ws;
    float *const stg = sm.stg + warp * 256;
    __nv_bfloat16 *const kvn = sm.kvn;
    unsigned *const seg_cnt = a.sync + a.s_seg;
    const long long c = pl.c, ub1 = pl.ub1;
    constexpr int CH = D / 8;   // 16-byte chunks per row
    for (long long pos = pl.ub0; pos < ub1;) {
        const Piece p = find_piece(prefix, ubp, B, Hk, nrb, pos, ub1);
        const int nh = a.rb_nh[p.rb];
        const int h0 = p.kh * gqa + a.rb_h0[p.rb];
        const int nrows = nh * R;
        const int p0 = cpos[p.b];
        const int Lb = p0 + R;

        // this piece's units reach the rows this step appends (positions p0 .. p0 + R - 1)
        const bool kv_new = p.u1 * kAttnUnit > p0 && p.u0 * kAttnUnit < Lb;
        // the piece holding the last new row appends the new rows to the cache
        const bool appender = kv_new && p.u1 * kAttnUnit >= Lb;
        const int kgrp = (Nq + p.kh * D) / GR, vgrp = (Nq + Nkv + p.kh * D) / GR;

        // ---- every piece of the q|k|v rows this segment needs is in its slot
        if (tid == 0) {
            bool ok = true;
            for (int h = h0; h < h0 + nh && ok; ++h)
                ok = wait_group(a, sm, pl, (h * d2) / GR);
            if (kv_new && ok)
                ok = wait_group(a, sm, pl, kgrp) && wait_group(a, sm, pl, vgrp);
        }
        named_bar_sync(1, kFW * 32);

        // ---- query rows (a warp per row: head h0 + i / R, verify row i % R):
        //      sums of the partials, RMSNorm, partial RoPE, bf16 into the q tile
        for (int i = warp; i < MT * 16; i += kFW) {
            if (i < nrows) {
                const int r = i % R;
                float v[8];
                head_rows(a, pl, (h0 + i / R) * d2, p.b * R + r, lane, v);
                norm_rope(v, a, sm.nq, sm.invf, (double)(p0 + r), stg, lane);
                for (int cc = lane; cc < CH; cc += 32)
                    *reinterpret_cast<uint4 *>(qs + i * (D * 2) + ((cc ^ (i & 7)) << 4)) =
                        bf16_chunk(stg, cc);
                __syncwarp();
            } else {
                for (int cc = lane; cc < CH; cc += 32)
                    *reinterpret_cast<uint4 *>(qs + i * (D * 2) + ((cc ^ (i & 7)) << 4)) =
                        make_uint4(0, 0, 0, 0);
            }
        }
        // ---- the new K (RMSNorm + RoPE) and V rows of this KV head, staged as bf16;
        //      the appender also writes them to the cache
        if (kv_new) {
            for (int t = warp; t < 2 * R; t += kFW) {
                const int kind = t / R, r = t % R;        // 0: K, 1: V
                float v[8];
                head_rows(a, pl, (kind ? Nq + Nkv : Nq) + p.kh * D, p.b * R + r, lane, v);
                if (kind == 0) {
                    norm_rope(v, a, sm.nk, sm.invf, (double)(p0 + r), stg, lane);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i < DB * 2)
                            stg[lane + 32 * i] = v[i];
                    __syncwarp();
                }
                __nv_bfloat16 *row = kvn + (kind * kFMaxB + r) * 256;
                __nv_bfloat16 *dst = (kind ? a.vc : a.kc) + (long long)p.b * a.st_batch +
                                     (long long)p.kh * a.st_head + (long long)(p0 + r) * a.st_tok;
                for (int cc = lane; cc < CH; cc += 32) {
                    const uint4 ch = bf16_chunk(stg, cc);
                    *reinterpret_cast<uint4 *>(row + cc * 8) = ch;
                    if (appender)
                        *reinterpret_cast<uint4 *>(dst + cc * 8) = ch;
                }
                __syncwarp();
            }
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

            // rows this step appends: the tile holds the cache's old contents there
            if (ok && kv_new && t0 + ntok > p0 && t0 < Lb) {
                const int r0 = p0 > t0 ? p0 - t0 : 0, r1 = Lb - t0 < ntok ? Lb - t0 : ntok;
                for (int idx = tid; idx < (r1 - r0) * 2 * CH; idx += kFW * 32) {
                    const int row = r0 + idx / (2 * CH), rest = idx % (2 * CH);
                    const int kind = rest / CH, cc = rest % CH;
                    const uint4 ch = *reinterpret_cast<const uint4 *>(
                        kvn + (kind * kFMaxB + (t0 + row - p0)) * 256 + cc * 8);
                    *reinterpret_cast<uint4 *>((kind ? vst : kst) + (cc >> 3) * bs + row * 128 +
                                               (((cc & 7) ^ (row & 7)) << 4)) = ch;
                }
                fence_proxy_async_smem();
                named_bar_sync(1, kFW * 32);
            }
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

// ------------------------------------------------------------------- merge

// C: o_proj k unit j = operand columns [128 j, 128 j + 128) of heads x head_dim,
// merged by every CTA whose o_proj items use it, into its own x slot `xs`.
// Per (row m, head h) pair the contributors of h's segment left m_c, l_c and
// O_c; with M = max m_c, attn = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
// The factors 2^(m_c - M) / L are formed once per pair (a warp over the
// contributors), then threads own columns so each partial row is one coalesced
// read.  a = attn * sigmoid(gate) goes to the slot in fragment order.
__device__ __forceinline__ void merge_unit(const FusedArgs &a, const Smem &sm, const Plan &pl, int j,
                                           uint8_t *xs)
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
            ok = wait_group(a, sm, pl, (h * 2 * d + d) / a.GR);
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
        const int h = k / d;
        const float gt = qkv_value(a, pl, h * 2 * d + d + (k - h * d), m);
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
        for (; c + 15 * split < n; c += 16 * split) {   // sixteen loads in flight
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                v[u] = __ldcg(base + (long long)(c + u * split) * slotf);
#pragma unroll
            for (int u = 0; u < 16; ++u)
                acc = fmaf(f[c + u * split], v[u], acc);
        }
        for (; c + 3 * split < n; c += 4 * split) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = __ldcg(base + (long long)(c + u * split) * slotf);
#pragma unroll
            for (int u = 0; u < 4; ++u)
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

    // ---- operand fragments (thread = (k16-step, lane))
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
        reinterpret_cast<uint2 *>(xs)[tid] = v;
    }
    // the slot's next reader is the o_proj phase of this CTA
    named_bar_sync(1, kFW * 32);
}

}  // namespace

// ------------------------------------------------------------------ kernel

// One instance per (q|k|v bits, group, o_proj bits, group, attention m-tiles,
// head_dim / 64): every phase is inlined, so no call frames or spills go
// through local memory.
template <int BQ, int GQ, int BO, int GO, int MT, int DB>
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
    sm.stg = reinterpret_cast<float *>(base + a.off_red + kRedBytes);
    sm.kvn = reinterpret_cast<__nv_bfloat16 *>(base + a.off_red + kRedBytes + kStgBytes);
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
    sm.pq = misc + 3840;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kFEntries; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kFW);
        }
        sm.flags[0] = sm.flags[1] = sm.flags[2] = sm.flags[3] = sm.flags[4] = 0;
        fence_mbar_init();
    }
    if (tid < a.B) {
        const int p0 = a.cache_pos[tid];
        const bool valid = p0 >= 0 && p0 + a.R <= a.cap;
        sm.cpos[tid] = p0;
        sm.ub[tid] = valid ? (p0 + a.R + kAttnUnit - 1) / kAttnUnit : 0;
        // a sequence out of the cache's range is skipped (no attention, no
        // append, zero output rows) and reported
        if (!valid && blockIdx.x == 0)
            atomicOr(a.status, kStatusRange);
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
        rg = proj_phase_a<BQ, GQ>(a, sm, pl, rg);
        rg = attn_phase<MT, DB>(a, sm, pl, rg);
        if (pl.io1 > pl.io0) {
            // the o_proj operand of this CTA's k units, into the (now free) x slots
            const int ku0 = (int)(pl.io0 / a.nrb_o), ku1 = (int)((pl.io1 - 1) / a.nrb_o);
            for (int j = ku0; j <= ku1; ++j)
                merge_unit(a, sm, pl, j, sm.xa + (size_t)(j - ku0) * kXSlotBytes);
            rg = proj_phase_o<BO, GO>(a, sm, pl, rg);
        }
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

template <int BQ, int GQ, int BO, int GO, int MT, int DB>
struct FusedInstance {
    static cudaError_t launch(const FusedArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
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
        return cudaLaunchKernelEx(&cfg, fused_kernel<BQ, GQ, BO, GO, MT, DB>, a, kmap, vmap);
    }
    static cudaError_t set_smem(int bytes)
    {
        return cudaFuncSetAttribute(fused_kernel<BQ, GQ, BO, GO, MT, DB>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    }
    static cudaError_t occupancy(int smem, int *blocks)
    {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks, fused_kernel<BQ, GQ, BO, GO, MT, DB>, kFThreads, smem);
    }
};

#define GATTN_FUSED_CASE(BQ_, GQ_, BO_, GO_, MT_, DB_)                                             \
    if (k.bits_a == BQ_ && k.group_a == GQ_ && k.bits_o == BO_ && k.group_o == GO_ &&             \
        k.MT == MT_ && k.DB == DB_) {                                                              \
        ops->launch = FusedInstance<BQ_, GQ_, BO_, GO_, MT_, DB_>::launch;                         \
        ops->set_smem = FusedInstance<BQ_, GQ_, BO_, GO_, MT_, DB_>::set_smem;                     \
        ops->occupancy = FusedInstance<BQ_, GQ_, BO_, GO_, MT_, DB_>::occupancy;                   \
        return true;                                                                               \
    }

}  // namespace gattn
