// merge.cu -- combine the attention partials of every segment, apply the
// output gate, and write the o_proj operand.
//
// One CTA per (segment, query row).  Every contributor (the CTAs whose unit
// ranges touched the segment) left m_j (the log2-domain row maximum), l_j and
// O_j; with M = max m_j,
//   attn = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j.
// Two dependent rounds of loads: one warp loads every (m_j, l_j) at once and
// leaves the factors 2^(m_j - M) / L in shared memory; then two threads per
// head_dim column each load half of the contributors' O_j values (all in
// flight together; a warp's loads are one coalesced line per contributor) and
// their sums are added.
//
//   attn = O / l,   a = attn * sigmoid(gate)   (the layer's output gate)
//
// Over a Bf16KTurbo4V cache the V rows were attended in their Walsh-Hadamard
// basis, so attn is first rotated back: attn = H (O / l) / sqrt(d).
//
// `a` goes to the o_proj input in fp16 tensor-core fragment order, with the
// group sums of those fp16 values that the projection's bias term needs.
#include "common.cuh"
#include "kernels.cuh"

namespace gattn {

constexpr int kMergeMaxContrib = 160;       // contributors per segment (>= attention grid)

__global__ void __launch_bounds__(512) attn_merge_kernel(const AttnArgs a)
{
    __shared__ long long prefix[33];
    __shared__ int ub[32];
    __shared__ float gsum_sm[8];
    __shared__ float fct[kMergeMaxContrib];
    __shared__ float comb[512];
    // the o_proj launches at once to stream its weights; this kernel's own
    // pre-wait work reads only cache_pos (a step input)
    pdl_launch_dependents();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = a.d;
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

    const int seg = blockIdx.x;                       // (b, kh, rb)
    const int rb = seg % a.nrb, kh = (seg / a.nrb) % a.Hk, b = seg / (a.nrb * a.Hk);
    const int nrows = a.rb_nh[rb] * a.R;
    const int i = blockIdx.y;                         // row within the segment
    if (b >= a.B || i >= nrows || ub[b] == 0)
        return;
    const long long T = prefix[a.B];
    const long long G = attn_ranges(T, a.grid, a.min_units);
    const long long U = ub[b];
    const long long seg_start = prefix[b] + (long long)(kh * a.nrb + rb) * U;
    const long long cf = sk_owner(seg_start, T, G), cl = sk_owner(seg_start + U - 1, T, G);
    const int n = (int)(cl - cf + 1);
    const int slot_floats = attn_slot_floats(D);
    const float *base = a.ws + (seg + cf) * (long long)slot_floats;

    const int hl = i / a.R, r = i % a.R;
    const int h = kh * (a.H / a.Hk) + a.rb_h0[rb] + hl;
    const int m = b * a.R + r;
    const int half = tid / D, jd = tid - half * D;    // column and contributor half
    const long long Ktot = (long long)a.H * D;

    pdl_wait();                 // partials (attention) and the gate (q|k|v projection)
    const float gt = a.gate[(long long)m * Ktot + (long long)h * D + jd];

    // ---- factors 2^(m_j - M) / L (one warp, every contributor's loads at once)
    if (warp == 0) {
        constexpr int kPer = kMergeMaxContrib / 32;
        float mv[kPer], lv[kPer];
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int j = lane + 32 * u;
            mv[u] = j < n ? base[(long long)j * slot_floats + i] : -INFINITY;
            lv[u] = j < n ? base[(long long)j * slot_floats + kAttnMaxRows + i] : 0.f;
            mx = fmaxf(mx, mv[u]);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float L = 0.f;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            mv[u] = mv[u] == -INFINITY ? 0.f : exp2f(mv[u] - mx);
            L = fmaf(mv[u], lv[u], L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            L += __shfl_xor_sync(0xffffffffu, L, o);
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int j = lane + 32 * u;
            if (j < n)
                fct[j] = mv[u] * inv;
        }
    }
    __syncthreads();

    // ---- weighted sum of the O_j of column jd over this thread's contributors
    //      (j = half, half + 2, ...), sixteen loads in flight at a time
    const float *po = base + 2 * kAttnMaxRows + (long long)i * D + jd;
    float acc = 0.f;
    int j = half;
    for (; j + 30 < n; j += 32) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            v[u] = __ldcg(po + (long long)(j + 2 * u) * slot_floats);
#pragma unroll
        for (int u = 0; u < 16; ++u)
            acc = fmaf(fct[j + 2 * u], v[u], acc);
    }
    for (; j < n; j += 2)
        acc = fmaf(fct[j], __ldcg(po + (long long)j * slot_floats), acc);
    comb[tid] = acc;
    __syncthreads();
    if (half != 0)
        return;
    float o = comb[jd] + comb[jd + D];
    if (a.vq) {
        // Turbo4 V cache: the values were attended in the rotated basis; rotate
        // the output row back, H o / sqrt(d) (butterflies over the d columns:
        // within a warp by shuffles, across warps through shared memory)
#pragma unroll
        for (int h2 = 1; h2 < 32; h2 <<= 1) {
            const float p = __shfl_xor_sync(0xffffffffu, o, h2);
            o = (lane & h2) ? p - o : o + p;
        }
        for (int h2 = 32; h2 < D; h2 <<= 1) {
            named_bar_sync(2, D);       // the partner has read this slot's last value
            comb[jd] = o;
            named_bar_sync(2, D);
            const float p = comb[jd ^ h2];
            o = (jd & h2) ? p - o : o + p;
        }
        o *= a.inv_sqrt_d;
    }
    const float gated = o * (1.f / (1.f + __expf(-gt)));
    const __half hv = __float2half_rn(gated);
    const int k = h * D + jd;
    a.x16[x16_offset(m, k, a.NT)] = hv;
    if (a.tap_attn)
        a.tap_attn[(long long)m * Ktot + k] = o;

    // group sums of the fp16 operand values (groups of gs columns within the
    // head); only the first D threads (warps 0 .. D/32 - 1) remain
    const int gs = a.group_o, MP = 8 * a.NT, c0 = warp * 32;
    float gsum = __half2float(hv);
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1)
        if (o2 < gs)
            gsum += __shfl_xor_sync(0xffffffffu, gsum, o2);
    if (gs <= 32) {
        if ((lane % gs) == 0) {
            const int k0 = k;
            a.xsum[((long long)(k0 >> 7) * (kKU / gs) + ((k0 & 127) / gs)) * MP + m] = gsum;
        }
    } else {
        if (lane == 0)
            gsum_sm[warp] = gsum;
        named_bar_sync(1, D);
        const int wpg = gs / 32;                 // warps per group
        if (lane == 0 && (warp % wpg) == 0) {
            float t = 0.f;
            for (int w2 = warp; w2 < warp + wpg; ++w2)
                t += gsum_sm[w2];
            const int k0 = h * D + c0;
            a.xsum[((long long)(k0 >> 7) * (kKU / gs) + ((k0 & 127) / gs)) * MP + m] = t;
        }
    }
}

cudaError_t launch_attn_merge(const AttnArgs &a, int max_rows, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B * a.Hk * a.nrb, max_rows);
    cfg.blockDim = dim3(2 * a.d);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel, a);
}

}  // namespace gattn
