// pack.cu -- one-time weight repacking into the projection tile layout, the
// debug decoders, and the per-step x operand preparation.
#include "common.cuh"
#include "kernels.cuh"
#include "proj.cuh"
#include "xconv.cuh"

namespace gattn {

// code k of an interchange row (LSB-first bitstream of little-endian words)
__device__ __forceinline__ uint32_t row_code(const uint32_t *row, long long k, int bits)
{
    const long long bit = k * bits;
    const long long w = bit >> 5;
    const int sh = (int)(bit & 31);
    unsigned long long v = row[w];
    if (sh + bits > 32)
        v |= (unsigned long long)row[w + 1] << 32;
    return (uint32_t)((v >> sh) & ((1u << bits) - 1u));
}

// lane-stream code index -> (row in the 32-row tile, k in the 128-wide unit)
__device__ __forceinline__ void lane_code_pos(int p, int bits, int lane, int &row, int &k)
{
    const int mi = p >> 3;
    int v = p & 7;
    if (bits == 4) {
        // nibble n of a word holds fragment value: 0,2,4,6,1,3,5,7
        const int nib = v;
        v = (nib < 4) ? 2 * nib : 2 * (nib - 4) + 1;
    }
    const int ks = mi >> 1, mt = mi & 1;
    const int g = lane >> 2, c = lane & 3;
    row = mt * 16 + g + 8 * ((v >> 1) & 1);
    k = ks * 16 + 2 * c + 8 * (v >> 2) + (v & 1);
}

// One thread per (row block, k unit, warp, lane) writes that lane's code stream
// (16*bits bytes) and, for lanes < 8*(128/group)... the unit's scale/bias table.
__global__ void repack_kernel(const RepackSrc src, int K, int bits, int group, int nrb,
                              uint8_t *dst)
{
    const long long nku = K / kKU;
    const long long total = (long long)nrb * nku * kWR * 32;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total)
        return;
    const int lane = (int)(t & 31);
    const int w = (int)((t >> 5) % kWR);
    const long long step = (t >> 5) / kWR;
    const int rb = (int)(step / nku), ku = (int)(step % nku);
    const int ub = unit_bytes(bits, group);
    uint8_t *unit = dst + (step * kWR + w) * (long long)ub;
    const int words_per_row = K * bits / 32;

    auto src_row = [&](int n, int &which, int &local) -> bool {
        int base = 0;
        for (int i = 0; i < src.nsrc; ++i) {
            if (n < base + src.rows[i]) {
                which = i;
                local = n - base;
                return true;
            }
            base += src.rows[i];
        }
        return false;
    };

    uint32_t words[32];
    for (int i = 0; i < 32; ++i)
        words[i] = 0;
    for (int p = 0; p < 128; ++p) {
        int row, k;
        lane_code_pos(p, bits, lane, row, k);
        const int n = rb * kRBR + w * 32 + row;
        int which, local;
        uint32_t code = 0;
        if (src_row(n, which, local))
            code = row_code(src.packed[which] + (long long)local * words_per_row,
                            (long long)ku * kKU + k, bits);
        const int bit = p * bits, wi = bit >> 5, sh = bit & 31;
        words[wi] |= code << sh;
        if (sh + bits > 32)
            words[wi + 1] |= code >> (32 - sh);
    }
    for (int i = 0; i < bits; ++i) {
        uint4 v = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
        *reinterpret_cast<uint4 *>(unit + (i * 32 + lane) * 16) = v;
    }
    // scale/bias table: entry (gi, g, rs) for gi < 128/group
    const int ngr = kKU / group;
    const int gpr = K / group;
    uint32_t *sb = reinterpret_cast<uint32_t *>(unit + unit_code_bytes(bits));
    for (int gi = 0; gi < ngr; ++gi) {
        const int g = lane >> 2, rs = lane & 3;
        const int row = g + 8 * rs;
        const int n = rb * kRBR + w * 32 + row;
        int which, local;
        uint32_t e = 0;
        if (src_row(n, which, local)) {
            const long long idx = (long long)local * gpr + ((long long)ku * kKU) / group + gi;
            e = (uint32_t)src.scales[which][idx] | ((uint32_t)src.biases[which][idx] << 16);
        }
        sb[(gi * 8 + g) * 4 + rs] = e;
    }
}

cudaError_t launch_repack(const RepackSrc &src, int K, int bits, int group, int nrb, uint8_t *dst,
                          cudaStream_t s)
{
    const long long total = (long long)nrb * (K / kKU) * kWR * 32;
    const int threads = 128;
    const long long blocks = (total + threads - 1) / threads;
    return launch_plain(repack_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, src, K, bits,
                        group, nrb, dst);
}

// Dequantize from the tile layout with the projection kernel's own unpack:
// one warp per unit, w = fp32(scale * code + bias).
template <int BITS>
__global__ void dequant_tiles_kernel(const uint8_t *w, int N, int K, int group, int nrb, float *out)
{
    const long long nku = K / kKU;
    const long long units = (long long)nrb * nku * kWR;
    const long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (u >= units)
        return;
    const int ub = unit_bytes(BITS, group);
    const uint8_t *unit = w + u * ub;
    const int wi = (int)(u % kWR);
    const long long step = u / kWR;
    const int rb = (int)(step / nku), ku = (int)(step % nku);
    uint32_t cw[4 * BITS];
    for (int i = 0; i < BITS; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(unit + (i * 32 + lane) * 16);
        cw[4 * i] = v.x;
        cw[4 * i + 1] = v.y;
        cw[4 * i + 2] = v.z;
        cw[4 * i + 3] = v.w;
    }
    const uint32_t *sb = reinterpret_cast<const uint32_t *>(unit + unit_code_bytes(BITS));
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 16; ++mi) {
        uint32_t A[4];
        unpack_a<BITS>(cw, mi, A);
        const int ks = mi >> 1, mt = mi & 1;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&A[r]);
            const float q[2] = {__low2float(h), __high2float(h)};
            const int row_off = (r & 1) ? 8 : 0, k_off = (r & 2) ? 8 : 0;
            const int row = mt * 16 + g + row_off;
            const int k = ks * 16 + 2 * c + k_off;
            const int gi = k / group;
            const uint32_t e = sb[(gi * 8 + g) * 4 + (mt * 2 + (row_off ? 1 : 0))];
            const long long n = (long long)rb * kRBR + wi * 32 + row;
            if (n < N) {
                for (int j = 0; j < 2; ++j)
                    out[n * K + (long long)ku * kKU + k + j] = fmaf(bf16_lo(e), q[j], bf16_hi(e));
            }
        }
    }
}

cudaError_t launch_dequant_tiles(const uint8_t *w, int N, int K, int bits, int group, int nrb,
                                 float *out, cudaStream_t s)
{
    const long long units = (long long)nrb * (K / kKU) * kWR;
    const unsigned blocks = (unsigned)((units * 32 + 127) / 128);
    auto go = [&](auto kern) {
        return launch_plain(kern, dim3(blocks), dim3(128), 0, s, w, N, K, group, nrb, out);
    };
    switch (bits) {
    case 2: return go(dequant_tiles_kernel<2>);
    case 3: return go(dequant_tiles_kernel<3>);
    case 4: return go(dequant_tiles_kernel<4>);
    case 5: return go(dequant_tiles_kernel<5>);
    case 6: return go(dequant_tiles_kernel<6>);
    case 8: return go(dequant_tiles_kernel<8>);
    default: return cudaErrorInvalidValue;
    }
}

__global__ void unpack_codes_kernel(const uint32_t *packed, long long N, long long K, int bits,
                                    uint8_t *codes)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * K)
        return;
    const long long n = i / K, k = i % K;
    codes[i] = (uint8_t)row_code(packed + n * (K * bits / 32), k, bits);
}

cudaError_t launch_unpack_codes(const uint32_t *packed, long long N, long long K, int bits,
                                uint8_t *codes, cudaStream_t s)
{
    const long long total = N * K;
    if (total == 0)
        return cudaSuccess;
    return launch_plain(unpack_codes_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, s,
                        packed, N, K, bits, codes);
}

// x [M][K] (fp32 or bf16) -> fp16 B fragments + fp32 group sums of the fp16
// values.  One CTA per 128-wide k unit; thread (m, part) converts 16 elements.
// Row m's input RMSNorm factor 1 / sqrt(mean(x^2) + eps) over all K columns:
// one warp per row, four vector loads in flight per lane.
__device__ __forceinline__ float row_inv_rms(const void *x, int x_dtype, int m, int K, int lane,
                                             float eps)
{
    float ss = 0.f;
    if (x_dtype == 0) {
        const float4 *row = reinterpret_cast<const float4 *>(static_cast<const float *>(x) +
                                                             (long long)m * K);
#pragma unroll 4
        for (int i = lane; i < K / 4; i += 32) {
            const float4 f = row[i];
            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, fmaf(f.z, f.z, fmaf(f.w, f.w, ss))));
        }
    } else {
        const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(x) +
                                                           (long long)m * K);
#pragma unroll 4
        for (int i = lane; i < K / 8; i += 32) {
            const uint4 u = row[i];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
                ss = fmaf(a, a, fmaf(b, b, ss));
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    return rsqrtf(ss / (float)K + eps);
}

__global__ void __launch_bounds__(256) xprep_kernel(const void *x, int x_dtype, int M, int K,
                                                    int group, int NT, __half *x16, float *xsum,
                                                    const uint16_t *in_w, float eps)
{
    __shared__ float s_inv[32];
    // the next kernel (the q|k|v projection) may start streaming weights at once
    pdl_launch_dependents();
    pdl_wait();
    const int ku = blockIdx.x;
    const int m = threadIdx.x >> 3, part = threadIdx.x & 7;
    const int MP = 8 * NT;
    if (in_w) {                 // decoder-block input: per-row norm factors first
        for (int rr = threadIdx.x >> 5; rr < M; rr += blockDim.x >> 5) {
            const float inv = row_inv_rms(x, x_dtype, rr, K, threadIdx.x & 31, eps);
            if ((threadIdx.x & 31) == 0)
                s_inv[rr] = inv;
        }
        __syncthreads();
    }
    if (m >= MP)
        return;
    // fp32 input: columns [M, 2M) carry the exact remainder x - fp16(x)
    const bool lo_part = x_dtype == 0 && m >= M && m < 2 * M;
    const int src_m = lo_part ? m - M : m;
    // decoder-block input: the operand is RMSNorm(x) * input_ln
    const float scale = in_w && (m < M || lo_part) ? s_inv[src_m] : 1.f;
    const XRaw raw = x_chunk_load(x, x_dtype, M, K, ku * kKU, m, part);
    x_chunk_convert(raw, x_dtype, M, group, NT, ku * kKU, m, part, scale, in_w,
                    x16 + (long long)ku * NT * 1024, xsum + (long long)ku * (kKU / group) * MP);
}

cudaError_t launch_xprep(const void *x, int x_dtype, int M, int K, int group, int NT, __half *x16,
                         float *xsum, const uint16_t *in_w, float eps, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(K / kKU);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, xprep_kernel, x, x_dtype, M, K, group, NT, x16, xsum, in_w, eps);
}

}  // namespace gattn

namespace gattn {

// Post-attention RMSNorm of the decoder block: one CTA per row of the stored
// bf16 residual stream, out_n = bf16(r / sqrt(mean(r^2) + eps) * w).
__global__ void __launch_bounds__(256) postnorm_kernel(const __nv_bfloat16 *r, const uint16_t *w,
                                                       float eps, int N, __nv_bfloat16 *out_n)
{
    __shared__ float red[8];
    pdl_launch_dependents();
    pdl_wait();                 // r is the o_proj's output
    const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16 *row = r + (long long)m * N;
    float ss = 0.f;
    for (int i = tid; i < N; i += 256) {
        const float v = __bfloat162float(row[i]);
        ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0)
        red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2)
        tot += red[w2];
    const float inv = rsqrtf(tot / (float)N + eps);
    for (int i = tid; i < N; i += 256)
        out_n[(long long)m * N + i] = __float2bfloat16_rn(
            __bfloat162float(row[i]) * inv * __uint_as_float((uint32_t)w[i] << 16));
}

cudaError_t launch_postnorm(const __nv_bfloat16 *r, const uint16_t *w, float eps, int M, int N,
                            __nv_bfloat16 *out_n, bool pdl, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, postnorm_kernel, r, w, eps, N, out_n);
}

}  // namespace gattn
