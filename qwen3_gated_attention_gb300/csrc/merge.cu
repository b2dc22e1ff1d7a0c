// merge.cu -- combine the attention partials of every segment, apply the
// output gate, and write the o_proj operand.
//
// One CTA per (segment, query row), one warp per 32 head_dim columns.  The
// lanes of a warp split the segment's contributors (the CTAs whose unit ranges
// touched it), so a segment cut into many pieces merges in about one memory
// round trip: each lane folds its contributors (m_j, l_j, O_j) with a running
// log2-domain maximum, the lanes agree on M = max m, rescale by 2^(m - M), and
// a shuffle reduce-scatter sums O and l across lanes (column c lands on lane c).
//
//   attn = O / l,   a = attn * sigmoid(gate)   (the layer's output gate)
//
// `a` goes to the o_proj input in fp16 tensor-core fragment order, with the
// group sums of those fp16 values that the projection's bias term needs.
#include "common.cuh"
#include "kernels.cuh"

namespace gattn {

__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnArgs a)
{
    __shared__ long long prefix[33];
    __shared__ int ub[32];
    __shared__ float gsum_sm[8];
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
    const int c0 = warp * 32;
    const long long Ktot = (long long)a.H * D;

    pdl_wait();                 // partials (attention) and the gate (q|k|v projection)
    const float gt = a.gate[(long long)m * Ktot + (long long)h * D + c0 + lane];
    // one pass per lane over its contributors with a running maximum
    float mloc = -INFINITY, lloc = 0.f;
    float acc[32];
#pragma unroll
    for (int cidx = 0; cidx < 32; ++cidx)
        acc[cidx] = 0.f;
    // contributors j and j + 32 are loaded together (one memory round trip for
    // up to 64 contributors), then folded
    for (int j0 = lane; j0 < n; j0 += 64) {
        float mj[2], lj[2];
        float4 v[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j = j0 + 32 * u;
            const bool live = j < n;
            const float *pj = base + (long long)(live ? j : j0) * slot_floats;
            mj[u] = live ? __ldcg(pj + i) : -INFINITY;
            lj[u] = __ldcg(pj + kAttnMaxRows + i);
            const float4 *src = reinterpret_cast<const float4 *>(pj + 2 * kAttnMaxRows +
                                                                 (long long)i * D + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                v[u][q] = __ldcg(src + q);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float mnew = fmaxf(mloc, mj[u]);
            const float sa = (mloc == -INFINITY) ? 0.f : exp2f(mloc - mnew);
            const float sb = (mj[u] == -INFINITY) ? 0.f : exp2f(mj[u] - mnew);
            mloc = mnew;
            lloc = lloc * sa + lj[u] * sb;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                acc[4 * q] = acc[4 * q] * sa + v[u][q].x * sb;
                acc[4 * q + 1] = acc[4 * q + 1] * sa + v[u][q].y * sb;
                acc[4 * q + 2] = acc[4 * q + 2] * sa + v[u][q].z * sb;
                acc[4 * q + 3] = acc[4 * q + 3] * sa + v[u][q].w * sb;
            }
        }
    }
    float M = mloc;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float sc = (mloc == -INFINITY) ? 0.f : exp2f(mloc - M);
    float L = lloc * sc;
#pragma unroll
    for (int cidx = 0; cidx < 32; ++cidx)
        acc[cidx] *= sc;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, o);
    // reduce-scatter: after the step with offset `off`, the lane keeps the half
    // of its columns selected by lane bit `off`; column c0 + lane ends on lane
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int cidx = 0; cidx < off; ++cidx) {
            const float send = upper ? acc[cidx] : acc[cidx + off];
            const float keep = upper ? acc[cidx + off] : acc[cidx];
            acc[cidx] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    const int jd = c0 + lane;
    const float o = L > 0.f ? acc[0] / L : 0.f;
    const float gated = o * (1.f / (1.f + __expf(-gt)));
    const __half hv = __float2half_rn(gated);
    const int k = h * D + jd;
    a.x16[x16_offset(m, k, a.NT)] = hv;
    if (a.tap_attn)
        a.tap_attn[(long long)m * Ktot + k] = o;

    // group sums of the fp16 operand values (groups of gs columns within the head)
    const int gs = a.group_o, MP = 8 * a.NT;
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
        __syncthreads();
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
    cfg.blockDim = dim3(a.d);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel, a);
}

}  // namespace gattn
