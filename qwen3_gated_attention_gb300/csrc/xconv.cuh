// xconv.cuh -- the layer input x as the projections' tensor-core operand.
#pragma once

#include "common.cuh"

namespace gattn {

// The raw input of one 16-element chunk: 16 bf16 (two 16-byte words) or 16
// fp32 (four), loaded ahead of the conversion so that a thread's loads for
// several chunks are in flight together.
struct XRaw {
    uint4 w[4];
};

// Loads chunk `part` (16 elements from k0unit + 16 part) of operand column m
// (fp32: m >= M is the low plane of row m - M) for x_chunk_convert; columns
// with no input (and lanes with live false) load nothing.
__device__ __forceinline__ XRaw x_chunk_load(const void *x, int x_dtype, int M, int K, int k0unit,
                                            int m, int part, bool live = true)
{
    XRaw r;
    const int k0 = k0unit + part * 16;
    const bool lo_part = x_dtype == 0 && m >= M && m < 2 * M;
    if (live && (m < M || lo_part)) {
        const int src_m = lo_part ? m - M : m;
        if (x_dtype == 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const float *>(x) +
                                                               (long long)src_m * K + k0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                r.w[i] = src[i];
        } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(x) + (long long)m * K + k0);
            r.w[0] = src[0];
            r.w[1] = src[1];
        }
    }
    return r;
}

// One 16-element chunk of operand column m at one 128-wide k unit (loaded by
// x_chunk_load): x (fp32 or bf16, row-major [M][K]) to fp16 B-fragment halves,
// written into `frag` (that k unit's NT x 1024 halves in the order of
// x16_offset), and the group sums of the same fp16 values into `sums` (that k
// unit's (128 / group) x MP floats).  fp32 x: column m < M holds the nearest
// fp16, column M + m the exact remainder x - fp16(x).  in_w (bf16 [K], or
// null): decoder-block input, the operand is x * scale * in_w (scale the row's
// RMSNorm factor), rounded to bf16 for a bf16 stream.  Columns past the operand
// are zeros.  The eight lanes part = 0..7 of an aligned lane octet call this
// together (the group sums are shuffles among them); k0unit is the unit's first
// k in x.  A lane with live false only takes part in the shuffles (it writes
// nothing).
__device__ __forceinline__ void x_chunk_convert(const XRaw &r, int x_dtype, int M, int group,
                                                int NT, int k0unit, int m, int part, float scale,
                                                const uint16_t *in_w, __half *frag, float *sums,
                                                bool live = true)
{
    const int MP = 8 * NT;
    const int k0 = k0unit + part * 16;
    const bool lo_part = live && x_dtype == 0 && m >= M && m < 2 * M;
    float v[16];
    if (live && (m < M || lo_part)) {
        if (x_dtype == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[4 * i] = __uint_as_float(r.w[i].x);
                v[4 * i + 1] = __uint_as_float(r.w[i].y);
                v[4 * i + 2] = __uint_as_float(r.w[i].z);
                v[4 * i + 3] = __uint_as_float(r.w[i].w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t w[4] = {r.w[i].x, r.w[i].y, r.w[i].z, r.w[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * i + 2 * j] = bf16_lo(w[j]);
                    v[8 * i + 2 * j + 1] = bf16_hi(w[j]);
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = 0.f;
    }
    if (live && in_w && (m < M || lo_part)) {
        // the normed row is an activation of the residual stream's type: bf16
        // rows give a bf16 operand, fp32 rows keep fp32 (hi + lo columns)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = v[i] * scale * __uint_as_float((uint32_t)in_w[k0 + i] << 16);
            if (x_dtype != 0)
                v[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
        }
    }
    __half h[16];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half hi = __float2half_rn(v[i]);
        h[i] = lo_part ? __float2half_rn(v[i] - __half2float(hi)) : hi;
        sum += __half2float(h[i]);
    }
    // element q of this k16 step goes to lane (m%8)*4 + (q%8)/2, half slot (q/8)*2 + q%2
    const int base = ((m >> 3) * 8 + part) * 32;
#pragma unroll
    for (int cq = 0; cq < 4 && live; ++cq) {
        const int lane = ((m & 7) << 2) | cq;
        __half2 lo = __halves2half2(h[2 * cq], h[2 * cq + 1]);
        __half2 hi = __halves2half2(h[8 + 2 * cq], h[8 + 2 * cq + 1]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&lo);
        u.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(frag + (base + lane) * 4) = u;
    }
    // group sums: parts [gi*ppg, (gi+1)*ppg) of this column form group gi
    const int ppg = group >> 4;
    for (int o = 1; o < ppg; o <<= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (live && (part % ppg) == 0)
        sums[(part / ppg) * MP + m] = sum;
}

}  // namespace gattn
