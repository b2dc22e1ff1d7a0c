// proj.cuh -- affine-dequant projection kernel: y[m][n] = sum_k W[n][k] x[m][k]
// with W = scale * code + bias per (row, group).
//
// Weights stream once from HBM: one producer warp issues 1-D TMA bulk copies
// of contiguous stages (all warps' units of one 128-wide k unit, plus the x
// fragments and group sums of that k unit) into a shared-memory ring; kWR
// consumer warps unpack the codes in registers straight into tensor-core A
// fragments (each code as the exact fp16 subnormal q * 2^-24, one mask or byte
// permute per register) and run mma.sync m16n8k16 against x (B fragments).
// Per group, D = sum code*x is folded as y += scale*D + bias*sum(x) in fp32, so
// no per-weight dequantization multiply is spent.
//
// Split-K inside a thread-block cluster: the cluster's CTAs share a block of
// rows (whole heads for the q|k|v projection) and split K; each CTA keeps its
// partial sums in its own shared memory and, after a cluster barrier, the
// epilogue reads the partials of the whole block through distributed shared
// memory.  No global scratch, no atomics, no waiting on other grids' CTAs.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "unpack.cuh"
#include "xconv.cuh"

namespace gattn {

// One stage: all 8 k16-steps of this warp's unit, folded into Y.
//
// Codes enter the tensor cores as exact fp16 subnormals (unpack_a_sub), so each
// group's MMA chain ends at 2^-24 * D, D = sum q * x (2^-20 * D on the 4-bit
// rows whose codes stay in the high nibble); the group folds as
// y += (scale * 2^24) * (2^-24 D) + bias * X, X the group sum of x.
// st: the stage's weights; xp: the x fragments of its k unit, group sums after.
template <int BITS, int NT, int GROUP>
__device__ __forceinline__ void proj_stage(const uint8_t *st, const uint8_t *xp, int ubytes, int w,
                                           int lane, float (&Y)[2][NT][4])
{
    const uint8_t *unit = st + w * ubytes;
    const uint8_t *sb = unit + unit_code_bytes(BITS);
    const uint2 *xf = reinterpret_cast<const uint2 *>(xp);
    const float *xs = reinterpret_cast<const float *>(xp + 2048 * NT);
    constexpr int kpg = GROUP / 16;     // k16-steps per group (compile time: no branches)
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
    // spread the k16-steps of a group over SPLIT independent accumulator sets
    // (more independent MMA chains per warp) and add the sets at the group end
    constexpr int SPLIT = (NT == 1 && kpg >= 2) ? 2 : 1;
    float D[SPLIT][2][NT][4];
#pragma unroll
    for (int sp = 0; sp < SPLIT; ++sp)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    D[sp][mt][nt][i] = 0.f;

#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int sp = ks % SPLIT;
        uint32_t A[2][4];
        unpack_a_sub<BITS>(cw, 2 * ks, A[0]);
        unpack_a_sub<BITS>(cw, 2 * ks + 1, A[1]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint2 b = xf[(nt * 8 + ks) * 32 + lane];
            mma_f16(D[sp][0][nt], A[0], b.x, b.y, D[sp][0][nt]);
            mma_f16(D[sp][1][nt], A[1], b.x, b.y, D[sp][1][nt]);
        }
        if ((ks % kpg) == kpg - 1) {
            const int gi = ks / kpg;
            const uint4 e = *reinterpret_cast<const uint4 *>(sb + (gi * 8 + g) * 16);
            // scale * 2^24 (2^20 for the high-nibble rows), exact powers of two
            constexpr float kLo = 16777216.f, kHi = BITS == 4 ? 1048576.f : 16777216.f;
            const float s[4] = {bf16_lo(e.x) * kLo, bf16_lo(e.y) * kHi, bf16_lo(e.z) * kLo,
                                bf16_lo(e.w) * kHi};
            const float bb[4] = {bf16_hi(e.x), bf16_hi(e.y), bf16_hi(e.z), bf16_hi(e.w)};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float2 xv = *reinterpret_cast<const float2 *>(xs + gi * 8 * NT + nt * 8 + 2 * c);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    float dd[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        dd[i] = D[0][mt][nt][i];
#pragma unroll
                        for (int q = 1; q < SPLIT; ++q)
                            dd[i] += D[q][mt][nt][i];
#pragma unroll
                        for (int q = 0; q < SPLIT; ++q)
                            D[q][mt][nt][i] = 0.f;
                    }
                    float *y = Y[mt][nt];
                    y[0] = fmaf(s[2 * mt], dd[0], fmaf(bb[2 * mt], xv.x, y[0]));
                    y[1] = fmaf(s[2 * mt], dd[1], fmaf(bb[2 * mt], xv.y, y[1]));
                    y[2] = fmaf(s[2 * mt + 1], dd[2], fmaf(bb[2 * mt + 1], xv.x, y[2]));
                    y[3] = fmaf(s[2 * mt + 1], dd[3], fmaf(bb[2 * mt + 1], xv.y, y[3]));
                }
            }
        }
    }
}

// Statics an epilogue needs, staged in shared memory before the main loop so
// the epilogue itself has no dependent global round trips.
struct EpiSmem {
    float *red;         // [MP][kRBR] this CTA's partial sums (aliases the stage ring)
    float *recv;        // partial sums pushed here by the cluster's CTAs (see below)
    float *vals;        // [eb_rows] final values of one column of the cluster's rows
    uint16_t *nq, *nk;  // q_norm / k_norm [d] (bf16 bits)
    float2 *invf;       // inv_freq [rd/2] as float (hi, lo) pairs
    int *cpos;          // cache_pos [B]
};

// Split-K reduction by pushing: after its main loop every CTA stores its
// partial sums straight into the shared memory of the CTA that finishes those
// values (st.async, no round trip), each store counting its bytes on the
// receiver's mbarrier `rbar`; a finishing CTA waits on its own rbar for the
// bytes it expects and adds the received partials in k-split order from its own
// shared memory.  No cluster-wide barrier between the main loop and the
// epilogue; one at the very end keeps every CTA resident until all receivers
// have their bytes.
//
// q|k|v: column m of the cluster's rows is finished by CTA m % csize; its
// receive area holds, per local column lc = m / csize and part (0; 1 for the
// low fp16 plane of fp32 x), per k split, the cluster's eb_rows rows:
// recv[((lc * P + part) * ks + kr) * eb_rows + row].
__device__ __forceinline__ void push_qkv(const ProjArgs &a, const EpiSmem &sm, const uint64_t *rbar,
                                         int rank, int csize, int tid)
{
    const int P = a.xsplit ? 2 : 1;
    const int rbl = rank / a.ks, kr = rank % a.ks;
    for (int idx = tid; idx < a.M * P * (kRBR / 4); idx += kWR * 32) {
        const int r4 = idx % (kRBR / 4), mp = idx / (kRBR / 4);
        const int m = mp / P, part = mp % P;
        const float4 v = *reinterpret_cast<const float4 *>(sm.red + (m + part * a.xsplit) * kRBR + r4 * 4);
        const int lc = m / csize;
        float *dst = sm.recv + ((long long)(lc * P + part) * a.ks + kr) * a.eb_rows + rbl * kRBR + r4 * 4;
        const uint32_t owner = (uint32_t)(m % csize);
        st_async_v4(dsmem_addr(dst, owner), v, dsmem_addr(rbar, owner));
    }
}

// Bytes the q|k|v receive area of CTA `rank` expects: every CTA of the cluster
// sends its kRBR rows of each column the rank finishes (x2 with low planes).
__device__ __forceinline__ uint32_t recv_bytes_qkv(const ProjArgs &a, int rank, int csize)
{
    const int cols = rank < a.M ? (a.M - rank + csize - 1) / csize : 0;
    return (uint32_t)cols * (a.xsplit ? 2u : 1u) * (uint32_t)csize * kRBR * 4u;
}

// o_proj: row r of the row block is finished by CTA r / rpr (rpr = ceil(128 /
// csize) rows each): recv[(kr * M + m) * rpr + r % rpr].
__device__ __forceinline__ void push_o(const ProjArgs &a, const EpiSmem &sm, const uint64_t *rbar,
                                       int rank, int csize, int tid)
{
    const int rpr = (kRBR + csize - 1) / csize;
    const int kr = rank;
    for (int idx = tid; idx < a.M * kRBR; idx += kWR * 32) {
        const int r = idx % kRBR, m = idx / kRBR;
        const int owner = r / rpr;
        float *dst = sm.recv + ((long long)kr * a.M + m) * rpr + (r - owner * rpr);
        st_async_f32(dsmem_addr(dst, (uint32_t)owner), sm.red[m * kRBR + r],
                     dsmem_addr(rbar, (uint32_t)owner));
    }
}

// Bytes the o_proj receive area of CTA `rank` expects: its rows from every
// k split, all columns.
__device__ __forceinline__ uint32_t recv_bytes_o(const ProjArgs &a, int rank, int csize)
{
    const int rpr = (kRBR + csize - 1) / csize;
    const int rows = max(0, min(rpr, kRBR - rank * rpr));
    return (uint32_t)csize * (uint32_t)a.M * (uint32_t)rows * 4u;
}

// q|k|v epilogue of the cluster's rows (whole heads): this CTA takes the
// columns m with m % cluster_size == rank.  Per column: the final values (the
// received partials added in k-split order) into shared memory, then per head
// one warp splits query / gate / k / v, applies RMSNorm + partial RoPE to
// query and k, and writes q (bf16), the gate (fp32) and the new cache rows
// (bf16).
template <int MP>
static __device__ void epilogue_qkv(const ProjArgs &a, const EpiQKV &e, const EpiSmem &sm, int row0,
                                    int rank, int csize, int warp, int lane, int tid)
{
    const int d = e.d, half = e.rd >> 1, heads = a.eb_rows / d, per = d >> 5;
    const int Ny = e.Nq + 2 * e.Nkv;
    // up to kWR / heads of this CTA's columns at a time, so that every warp has
    // a (column, head) to finish even when the cluster spans a single head
    const int mper = heads >= kWR ? 1 : kWR / heads;
    const int ebr = a.eb_rows, ks = a.ks, P = a.xsplit ? 2 : 1;
    for (int m0 = rank; m0 < a.M; m0 += csize * mper) {
        // the pass's columns m0 + j csize, j < nm (only those that exist)
        const int nm = min(mper, (a.M - m0 + csize - 1) / csize);
        for (int idx = tid; idx < nm * ebr; idx += kWR * 32) {
            const int j = idx / ebr, r = idx - j * ebr;
            const int lc = m0 / csize + j;              // (m0 + j csize) / csize
            const float *hi = sm.recv + (lc * P * ks) * ebr + r;
            float v = 0.f;
            if (P == 1) {
                for (int k = 0; k < ks; ++k)
                    v += hi[k * ebr];
            } else {
                for (int k = 0; k < ks; ++k) {
                    v += hi[k * ebr];
                    v += hi[(ks + k) * ebr];
                }
            }
            sm.vals[idx] = v;
        }
        named_bar_sync(1, kWR * 32);
        for (int wi = warp; wi < mper * heads; wi += kWR) {
            const int j = wi / heads, hb = wi - j * heads;
            const int m = m0 + j * csize;
            const int n0 = row0 + hb * d;
            if (m >= a.M || n0 >= a.N)
                continue;
            const float *hv = sm.vals + j * a.eb_rows + hb * d;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = i < per ? hv[lane + 32 * i] : 0.f;
            if (e.tap_y) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < per)
                        e.tap_y[(long long)m * Ny + n0 + lane + 32 * i] = v[i];
            }
            const int b = m / e.R, r = m % e.R;
            const int p0 = sm.cpos[b];
            const bool valid = p0 >= 0 && p0 + e.R <= e.cap;
            int kind, head;    // 0 query, 1 gate, 2 k, 3 v
            if (n0 < e.Nq) {
                head = n0 / (2 * d);
                kind = ((n0 % (2 * d)) >= d) ? 1 : 0;
            } else if (n0 < e.Nq + e.Nkv) {
                head = (n0 - e.Nq) / d;
                kind = 2;
            } else {
                head = (n0 - e.Nq - e.Nkv) / d;
                kind = 3;
            }
            if (kind == 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < per)
                        e.gate[(long long)m * e.H * d + head * d + lane + 32 * i] = v[i];
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
                const float inv = rsqrtf(ss / (float)d + e.eps);
                const uint16_t *nw = kind == 0 ? sm.nq : sm.nk;
                // partial rotary on dims [0, rd): pairs (j, j + rd/2) at position p0 + r.
                // The angle pos * inv_freq is formed as an unevaluated float pair
                // (inv_freq split in hi + lo on the host, the product's rounding
                // error recovered with an fma) and reduced modulo 2 pi with a
                // two-constant Cody-Waite step, so the reduced angle is good to a
                // few 1e-7 rad for positions far past 1e5 with no double math
                const float pos = (float)(p0 + r);      // exact below 2^24
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = lane + 32 * i;
                    o[i] = i < per ? v[i] * inv * bf16_bits_to_float(nw[j]) : 0.f;
                    if (i < per && j < e.rd) {
                        const int fi = j < half ? j : j - half;
                        const int jp = j < half ? j + half : j - half;
                        const float partner = hv[jp] * inv * bf16_bits_to_float(nw[jp]);
                        const float2 fq = sm.invf[fi];
                        const float ph = pos * fq.x;
                        const float pl = fmaf(pos, fq.x, -ph) + pos * fq.y;
                        const float turns = rintf(ph * 0.15915494f);
                        float red = fmaf(-turns, 6.2831855f, ph);     // 2 pi = 6.2831855f
                        red = fmaf(-turns, -1.7484555e-07f, red);    //   + -1.7484555e-07f
                        red += pl;
                        float sn, cs;
                        __sincosf(red, &sn, &cs);   // |red| <= pi + 1e-6: hardware path
                        o[i] = j < half ? o[i] * cs - partner * sn : o[i] * cs + partner * sn;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = o[i];
            }
            if (kind == 0) {
                __nv_bfloat16 *q = e.qn + (((long long)b * e.R + r) * e.H + head) * d;
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
            if ((kind == 3 && e.vq_codes) || (kind == 2 && e.kq_codes)) {
                // Turbo4 cache: quantize the bf16 row (turbo.cuh); V always, K for
                // the symmetric format (after its norm and rotary embedding)
                float xq[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    xq[i] = i < per ? __bfloat162float(__float2bfloat16_rn(v[i])) : 0.f;
                const long long row = p0 + r;
                uint8_t *qc = kind == 3 ? e.vq_codes + b * e.cq_batch + head * e.cq_head
                                        : e.kq_codes + b * e.kcq_batch + head * e.kcq_head;
                uint8_t *qs = kind == 3 ? e.vq_scales + b * e.sq_batch + head * e.sq_head
                                        : e.kq_scales + b * e.ksq_batch + head * e.ksq_head;
                turbo4_quantize_warp(xq, per, lane, e.tq, qc + row * (d / 2), qs + row * (d / 16));
                continue;
            }
            __nv_bfloat16 *dst = (kind == 2 ? e.kc : e.vc) + (long long)b * e.st_batch +
                                 (long long)head * e.st_head + (long long)(p0 + r) * e.st_tok;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < per)
                    dst[lane + 32 * i] = __float2bfloat16_rn(v[i]);
        }
        named_bar_sync(1, kWR * 32);
    }
}

// o_proj epilogue: the cluster's single row block, rows split across its CTAs
// (ceil(128 / cluster size) per rank); thread t takes row rank * rpr + t % rpr
// and the columns t / rpr + j * (128 / rpr), adding the received partials in
// k-split order.
template <int MP>
static __device__ void epilogue_o(const ProjArgs &a, const EpiO &e, const EpiSmem &sm, int row0,
                                  int rank, int csize, int tid)
{
    const int rpr = (kRBR + csize - 1) / csize;   // rows per rank
    const int lanes_m = (kWR * 32) / rpr;         // column lanes per row
    if (tid >= lanes_m * rpr)
        return;
    const int r = rank * rpr + tid % rpr;
    const int n = row0 + r;
    if (r >= kRBR || n >= a.N)
        return;
    for (int m = tid / rpr; m < a.M; m += lanes_m) {
        const int b = m / e.R;
        const int pb = sm.cpos[b];
        const bool valid = pb >= 0 && pb + e.R <= e.cap;
        float v = 0.f;
        if (valid) {
            const float *pr = sm.recv + (long long)m * rpr + (r - rank * rpr);
            for (int k = 0; k < a.ks; ++k)
                v += pr[(long long)k * a.M * rpr];
        }
        if (e.resid) {
            const long long ri = (long long)m * a.N + n;
            v += e.resid_f32 ? static_cast<const float *>(e.resid)[ri]
                             : __uint_as_float((uint32_t)static_cast<const uint16_t *>(e.resid)[ri]
                                               << 16);
        }
        e.out[(long long)m * a.N + n] = __float2bfloat16_rn(v);
    }
}

// Decoder-block post-norm inside the o_proj launch, after the cluster's last
// barrier (the stage ring is free again).  Each CTA adds up the squares of the
// bf16 rows it stored (its own writes, in a fixed order) into its slot of
// ss_part; the CTA that takes the last ticket sums the slots in CTA order and
// writes out_n = bf16(out * rsqrt(mean(out^2) + eps) * post_w).  Nothing
// waits: CTAs that are not last just leave.
template <int MP>
static __device__ void postnorm_tail(const ProjArgs &a, const EpiO &e, float *scratch, int row0,
                                     int rank, int csize)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kWarps = (int)(blockDim.x >> 5);
    const int rpr = (kRBR + csize - 1) / csize;
    const int r0 = rank * rpr;
    const int nr = max(0, min(min(rpr, kRBR - r0), a.N - (row0 + r0)));
    __syncthreads();            // this CTA's out stores are visible to all its threads
    for (int m = warp; m < a.M; m += kWarps) {
        float ss = 0.f;
        for (int j = lane; j < nr; j += 32) {
            const float v = __bfloat162float(e.out[(long long)m * a.N + row0 + r0 + j]);
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0)
            e.ss_part[(long long)blockIdx.x * a.M + m] = ss;
    }
    __threadfence();
    __syncthreads();
    unsigned *last = reinterpret_cast<unsigned *>(scratch);
    if (tid == 0)
        *last = atomicAdd(e.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!*last)
        return;
    __threadfence();
    float *inv = scratch + 32;
    for (int m = warp; m < a.M; m += kWarps) {
        float ss = 0.f;
        for (int c = lane; c < (int)gridDim.x; c += 32)
            ss += __ldcg(e.ss_part + (long long)c * a.M + m);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0)
            inv[m] = rsqrtf(ss / (float)a.N + e.eps);
    }
    __syncthreads();
    const int vpr = a.N / 8;    // 16-byte vectors per row
    for (int i = tid; i < a.M * vpr; i += kWarps * 32) {
        const int m = i / vpr, c8 = i - m * vpr;
        const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(e.out + (long long)m * a.N) + c8);
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(e.post_w) + c8);
        const uint32_t uu[4] = {u.x, u.y, u.z, u.w}, ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
        const float f = inv[m];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(bf16_lo(uu[j]) * f * bf16_lo(ww[j]),
                                                          bf16_hi(uu[j]) * f * bf16_hi(ww[j]));
            o[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(e.out_n + (long long)m * a.N)[c8] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid == 0)
        *e.ticket = 0u;         // ready for the next launch
}


// Two CTAs per SM at least; the four-column-tile instances, whose grids are
// short of CTAs at two per SM, ask for three.
template <int BITS, int NT, int MODE, int GROUP>
__global__ void __launch_bounds__(proj_threads(NT), NT >= 4 ? 3 : 2)
    proj_kernel(const ProjArgs a, const EpiQKV eq, const EpiO eo)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int MP = 8 * NT;
    constexpr int kProducer = kWR;            // the producer warp
    const int S = a.stages;
    uint8_t *stages = smem;
    uint8_t *tail = smem + (size_t)S * a.stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(tail);             // [S <= 8]
    uint64_t *empty = full + 8;                                       // [8]
    int *flags = reinterpret_cast<int *>(tail + 128);                 // [0] abort
    uint64_t *rbar = reinterpret_cast<uint64_t *>(tail + 192);        // split-K receive
    EpiSmem sm;
    sm.red = reinterpret_cast<float *>(smem);                         // after the main loop
    sm.vals = reinterpret_cast<float *>(tail + 256);
    sm.nq = reinterpret_cast<uint16_t *>(sm.vals + kValsFloats);
    sm.nk = sm.nq + 256;
    sm.invf = reinterpret_cast<float2 *>(sm.vals + kValsFloats + 256);
    sm.cpos = reinterpret_cast<int *>(sm.invf + 128);
    sm.recv = reinterpret_cast<float *>(tail + proj_tail_bytes(a.eb_rows));
    uint8_t *xtab = reinterpret_cast<uint8_t *>(sm.recv + a.recv_cap);   // a.xtab_bytes
    const bool xfold = MODE == kModeQKV && a.xtab_bytes > 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int csize = a.rbc * a.ks;
    const int rank = (int)cluster_ctarank();
    const int cluster = blockIdx.x / csize;
    const int rb = cluster * a.rbc + rank / a.ks, kr = rank % a.ks;
    const int ku0 = (int)((long long)kr * a.nku / a.ks), ku1 = (int)((long long)(kr + 1) * a.nku / a.ks);
    const long long beg = (long long)rb * a.nku + ku0, end = (long long)rb * a.nku + ku1;

    const uint32_t rbytes = MODE == kModeQKV ? recv_bytes_qkv(a, rank, csize)
                                             : recv_bytes_o(a, rank, csize);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWR);
        }
        mbar_init(rbar, 1);
        if (rbytes)
            mbar_arrive_expect_tx(rbar, rbytes);
        flags[0] = 0;
        fence_mbar_init();
    }
    // the cluster's CTAs may signal rbar once everyone is past this point
    cluster_arrive_relaxed();
    // o_proj lets the next step's kernels launch at once: their pre-wait work
    // (weight streaming) reads nothing this kernel writes
    if constexpr (MODE == kModeO)
        pdl_launch_dependents();
    // epilogue statics: layer weights and the step's cache_pos (a step input),
    // copied asynchronously: nothing waits for them before the epilogue
    if (threadIdx.x < kWR * 32) {
        const int t = threadIdx.x;
        if constexpr (MODE == kModeQKV) {
            for (int j = t; j < eq.d / 8; j += kWR * 32) {
                cp_async<16>(sm.nq + 8 * j, eq.q_norm + 8 * j);
                cp_async<16>(sm.nk + 8 * j, eq.k_norm + 8 * j);
            }
            for (int j = t; j < eq.rd / 2; j += kWR * 32)
                cp_async<8>(sm.invf + j, eq.inv_freq2 + j);
            if (t < (a.M + eq.R - 1) / eq.R)
                cp_async<4>(sm.cpos + t, eq.cache_pos + t);
        } else {
            if (t < (a.M + eo.R - 1) / eo.R)
                cp_async<4>(sm.cpos + t, eo.cache_pos + t);
        }
    }
    __syncthreads();

    const int xbytes = 2048 * NT, sbytes = (kKU / GROUP) * 4 * MP;
    volatile int *abort = flags;
    float Y[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Y[mt][nt][i] = 0.f;

    if (warp == kProducer) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            long long it = 0;
            // weights do not depend on the previous kernel: start streaming them
            // before waiting for it, then fetch x once it is visible.
            const long long pre = (end - beg) < S ? (end - beg) : S;
            // bytes a stage brings: weights, and x unless the CTA converts x itself
            const uint32_t stage_tx = a.step_bytes + (xfold ? 0 : xbytes + sbytes);
            // failure test hook: CTA 0 never issues its last stage
            const long long withhold_at = a.withhold && blockIdx.x == 0 ? end - 1 - beg : -1;
            long long withheld = -1;
            for (; it < pre; ++it) {
                const long long s = beg + it;
                if (it == withhold_at) {
                    withheld = it;
                    continue;
                }
                uint8_t *st = stages + (size_t)(it % S) * a.stage_bytes;
                mbar_arrive_expect_tx(&full[it % S], stage_tx);
                bulk_g2s(st, a.w + s * a.step_bytes, a.step_bytes, &full[it % S], pol);
            }
            pdl_wait();
            for (long long i = 0; i < pre && !xfold; ++i) {
                if (i == withheld)
                    continue;
                const int ku = (int)((beg + i) % a.nku);
                uint8_t *st = stages + (size_t)(i % S) * a.stage_bytes;
                bulk_g2s(st + a.step_bytes, a.x16 + (long long)ku * NT * 1024, xbytes,
                         &full[i % S], pol);
                bulk_g2s(st + a.step_bytes + xbytes, a.xsum + (long long)ku * (kKU / GROUP) * MP,
                         sbytes, &full[i % S], pol);
            }
            for (; beg + it < end; ++it) {
                const long long s = beg + it;
                const int slot = (int)(it % S);
                const uint32_t ph = (uint32_t)((it / S) & 1);
                if (!mbar_wait(&empty[slot], ph ^ 1u, abort, a.status, a.wait_ns))
                    break;
                if (it == withhold_at) {
                    withheld = it;          // never issued: its consumers' wait runs out
                    continue;
                }
                const int ku = (int)(s % a.nku);
                uint8_t *st = stages + (size_t)slot * a.stage_bytes;
                mbar_arrive_expect_tx(&full[slot], stage_tx);
                bulk_g2s(st, a.w + s * a.step_bytes, a.step_bytes, &full[slot], pol);
                if (!xfold) {
                    bulk_g2s(st + a.step_bytes, a.x16 + (long long)ku * NT * 1024, xbytes,
                             &full[slot], pol);
                    bulk_g2s(st + a.step_bytes + xbytes,
                             a.xsum + (long long)ku * (kKU / GROUP) * MP, sbytes, &full[slot], pol);
                }
            }
            // let every copy this CTA issued land before the ring is reused
            const long long first = it > S ? it - S : 0;
            for (long long i = first; i < it; ++i) {
                if (i == withheld)
                    continue;
                unsigned long long t0 = global_ns();
                while (!mbar_try(&full[i % S], (uint32_t)((i / S) & 1)) &&
                       global_ns() - t0 < a.wait_ns) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        // the arguments read after the wait are brought into the constant cache
        // while waiting, each block of them by another warp
        if (lane == 0 && warp < 2) {
            unsigned h;
            if (warp == 0)
                h = arg_fold(a);
            else if constexpr (MODE == kModeQKV)
                h = arg_fold(eq);
            else
                h = arg_fold(eo);
            reinterpret_cast<volatile unsigned *>(flags)[4 + warp] = h;
        }
        // the x table of this CTA's k units (fp16 fragments and group sums of
        // every operand column): zeroed while waiting, so that only the columns
        // that carry input are converted after the wait
        const int xe = xbytes + sbytes;
        const int nk = ku1 - ku0;
        if (xfold) {
            uint4 *t4 = reinterpret_cast<uint4 *>(xtab);
            for (int i = threadIdx.x; i < nk * xe / 16; i += kWR * 32)
                t4[i] = make_uint4(0u, 0u, 0u, 0u);
            named_bar_sync(1, kWR * 32);
        }
        pdl_wait();
        // q|k|v: dependents (attention) may launch only once the previous kernels
        // have completed, so that attention can prefetch cache rows before waiting
        if constexpr (MODE == kModeQKV)
            pdl_launch_dependents();
        // items (k unit, column with input) of 128 k, eight lanes each, sixteen
        // per pass; the loads of two passes are issued together (one round trip
        // for up to 32 items: the decode and verify shapes)
        if (xfold) {
            const int mx = a.xsplit ? 2 * a.M : a.M;            // columns with input
            const int xd = a.x_f32 ? 0 : 1, K = a.nku * kKU, part = threadIdx.x & 7;
            for (int b0 = 0; b0 < nk * mx; b0 += 2 * kWR * 4) {
                int kl[2], m[2];
                bool live[2];
                XRaw raw[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int item = b0 + q * kWR * 4 + (threadIdx.x >> 3);
                    live[q] = item < nk * mx;
                    kl[q] = live[q] ? item / mx : 0;
                    m[q] = live[q] ? item % mx : 0;
                    raw[q] = x_chunk_load(a.xraw, xd, a.M, K, (ku0 + kl[q]) * kKU, m[q], part,
                                          live[q]);
                }
                // a warp none of whose items carry input skips the conversion
                // as a whole (its shuffles name every lane of the warp)
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (__any_sync(0xffffffffu, live[q]))
                        x_chunk_convert(raw[q], xd, a.M, GROUP, NT, (ku0 + kl[q]) * kKU, m[q], part,
                                        1.f, nullptr, reinterpret_cast<__half *>(xtab + kl[q] * xe),
                                        reinterpret_cast<float *>(xtab + kl[q] * xe + xbytes),
                                        live[q]);
            }
            named_bar_sync(1, kWR * 32);
        }
        for (long long it = 0; beg + it < end; ++it) {
            const int slot = (int)(it % S);
            const uint32_t ph = (uint32_t)((it / S) & 1);
            const uint8_t *st = stages + (size_t)slot * a.stage_bytes;
            if (mbar_wait(&full[slot], ph, abort, a.status, a.wait_ns))
                proj_stage<BITS, NT, GROUP>(st, xfold ? xtab + it * xe : st + a.step_bytes,
                                            a.unit_bytes, warp, lane, Y);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }
    }
    // the ring is drained: it now holds this CTA's partial sums [MP][kRBR]; the
    // epilogue statics have landed
    cp_async_wait_all();
    __syncthreads();
    if (warp < kWR) {
        const int g = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int row = warp * 32 + mt * 16 + g, col = nt * 8 + 2 * cq;
                sm.red[col * kRBR + row] = Y[mt][nt][0];
                sm.red[(col + 1) * kRBR + row] = Y[mt][nt][1];
                sm.red[col * kRBR + row + 8] = Y[mt][nt][2];
                sm.red[(col + 1) * kRBR + row + 8] = Y[mt][nt][3];
            }
    }
    __syncthreads();
    cluster_wait();     // every receive barrier of the cluster is initialized
    if (warp < kWR) {
        if constexpr (MODE == kModeQKV)
            push_qkv(a, sm, rbar, rank, csize, threadIdx.x);
        else
            push_o(a, sm, rbar, rank, csize, threadIdx.x);
    }
    // every partial this CTA finishes has landed; then the cluster barrier that
    // keeps each CTA resident until every receiver has its bytes (a CTA's shared
    // memory must outlive the stores sent to it), waited on only at the end
    // (not cut short by an aborted main loop: every CTA pushes its bytes, and
    // this CTA must see them all land before it may leave).  A sender whose own
    // stage wait ran out pushes about one limit late, so this wait is bounded by
    // four limits: it ends before the bytes land only if a copy never lands.
    if (warp < kWR && rbytes)
        mbar_wait_all(rbar, 0, a.status, 4 * a.wait_ns);
    cluster_arrive();
    if (warp < kWR && rbytes) {
        const int row0 = cluster * a.eb_rows;
        if constexpr (MODE == kModeQKV)
            epilogue_qkv<MP>(a, eq, sm, row0, rank, csize, warp, lane, threadIdx.x);
        else
            epilogue_o<MP>(a, eo, sm, row0, rank, csize, threadIdx.x);
    }
    if constexpr (MODE == kModeO) {
        if (eo.out_n)
            postnorm_tail<MP>(a, eo, reinterpret_cast<float *>(stages), cluster * a.eb_rows, rank,
                              csize);
    }
    cluster_wait();
}

template <int BITS, int NT, int MODE, int GROUP>
cudaError_t launch_proj_t(const ProjArgs &a, const EpiQKV &eq, const EpiO &eo, int grid, bool pdl,
                          cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(proj_threads(NT));
    cfg.dynamicSmemBytes = proj_smem_bytes(a);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.rbc * a.ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, proj_kernel<BITS, NT, MODE, GROUP>, a, eq, eo);
}

// the kernel instantiation for runtime (NT, mode, group)
template <int BITS, typename F>
cudaError_t with_proj_kernel(int NT, int mode, int group, F &&f)
{
#define GATTN_K(nt, md, gr)                                                                        \
    if (NT == nt && mode == md && group == gr)                                                     \
        return f(proj_kernel<BITS, nt, md, gr>, launch_proj_t<BITS, nt, md, gr>);
#define GATTN_G(nt, md) GATTN_K(nt, md, 32) GATTN_K(nt, md, 64) GATTN_K(nt, md, 128)
    GATTN_G(1, kModeQKV) GATTN_G(2, kModeQKV) GATTN_G(4, kModeQKV)
    GATTN_G(1, kModeO) GATTN_G(2, kModeO) GATTN_G(4, kModeO)
#undef GATTN_G
#undef GATTN_K
    return cudaErrorInvalidValue;
}

}  // namespace gattn
