// turbo.cuh -- the Turbo4 KV-cache format of the Atlas qwen3_5 forward page
// (MetalKvDtype / LayerKvCache): a row is stored in a Walsh-Hadamard-rotated
// basis as 4-bit Lloyd-Max codebook indices with one FP8 E4M3 scale per group
// of 16 coordinates ("matched-norm L2").  Bf16KTurbo4V stores V this way and
// keeps K in bf16; the symmetric Turbo4 format stores both.
//
// Per row of d values (the bf16 row the cache would otherwise hold):
//   y   = H v / sqrt(d)            H: Sylvester Hadamard of order d, natural order
//   per group g of 16 consecutive y:
//   u_i = y_i / rms(y_g)           idx_i = number of decision thresholds below u_i
//   s_g = ||y_g|| / ||c(idx_g)||   stored as E4M3 (nearest-even, saturating)
//   byte j/2 holds code j in its low (j even) or high (j odd) nibble
// The decisions are taken in fp32 in a fixed order -- butterfly stages h = 1,
// 2, 4, ..., the rounded 1/sqrt(d) factor after them, pairwise sums over a
// group ((a0 + a1) + (a2 + a3)) + ..., correctly rounded sqrt and division --
// written with explicit _rn intrinsics so nothing is contracted into an FMA.
// Dequantized: v = H (s * c(idx)) / sqrt(d).  The attention never rotates a
// cached row back: it rotates each output row once (values, by linearity) and
// each q row once (keys: q . H k / sqrt(d) = (H q / sqrt(d)) . k).
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace gattn {

// fp32 decision tables of the 16-level Lloyd-Max quantizer of N(0, 1)
struct TurboTables {
    float th[15];                  // thresholds between levels (ascending)
    float lv[16];                  // levels (ascending)
    float inv_sqrt_d;              // fp32(1 / sqrt(d))
};

// The unnormalized Walsh-Hadamard butterflies of one row of d = 32 * per
// values held by a warp (lane l holds elements l + 32 i, i < per), stages
// h = 1, 2, 4, ... in that order, each output one rounded fp32 add or subtract.
__device__ __forceinline__ void wht_warp(float (&x)[8], int per, int lane)
{
    // butterfly stages h < 32: partner lane l ^ h holds element e ^ h
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < per) {
                const float p = __shfl_xor_sync(0xffffffffu, x[i], h);
                x[i] = (lane & h) ? __fsub_rn(p, x[i]) : __fadd_rn(x[i], p);
            }
    }
    // stages h = 32, 64, 128: partner element in the same lane, register i ^ (h / 32)
#pragma unroll
    for (int hh = 1; hh < 8; hh <<= 1) {
        if (hh < per) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < per && !(i & hh)) {
                    const float a = x[i], b = x[i + hh];
                    x[i] = __fadd_rn(a, b);
                    x[i + hh] = __fsub_rn(a, b);
                }
        }
    }
}

// One warp quantizes one row of d = 32 * per values: lane l holds elements
// l + 32 i (i < per) in x (bf16-exact fp32 values).  Writes d/2 code bytes
// and d/16 scale bytes.
__device__ __forceinline__ void turbo4_quantize_warp(float (&x)[8], int per, int lane,
                                                     const TurboTables &t, uint8_t *codes,
                                                     uint8_t *scales)
{
    wht_warp(x, per, lane);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i >= per)
            break;
        const float y = __fmul_rn(x[i], t.inv_sqrt_d);
        // group (2i or 2i + 1) = lanes 0..15 or 16..31 of this register
        float ss = __fmul_rn(y, y);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        int k = 0;
        float lvl = t.lv[0];
        if (ss != 0.f) {
            const float r = __fsqrt_rn(__fmul_rn(ss, 0.0625f));
            const float u = __fdiv_rn(y, r);
            // the number of thresholds below u, using their exact symmetry about 0
            // (th[14 - j] = -th[j], th[7] = 0): n = positive thresholds that |u|
            // passes (strictly for u > 0, inclusively for u <= 0); code 8 + n or 7 - n
            const float au = fabsf(u);
            const bool pos = u > 0.f;
            int n = 0;
            float mag = t.lv[8];
#pragma unroll
            for (int j = 8; j < 15; ++j)
                if (pos ? au > t.th[j] : au >= t.th[j]) {
                    n = j - 7;
                    mag = t.lv[j + 1];
                }
            k = pos ? 8 + n : 7 - n;
            lvl = pos ? mag : -mag;
        }
        float cs = __fmul_rn(lvl, lvl);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
            cs = __fadd_rn(cs, __shfl_xor_sync(0xffffffffu, cs, o));
        const int hi = __shfl_down_sync(0xffffffffu, k, 1);
        const int e = lane + 32 * i;
        if (!(lane & 1))
            codes[e >> 1] = (uint8_t)(k | (hi << 4));
        if ((lane & 15) == 0)
            scales[e >> 4] = ss != 0.f ? (uint8_t)__nv_cvt_float_to_fp8(__fsqrt_rn(__fdiv_rn(ss, cs)),
                                                                        __NV_SATFINITE, __NV_E4M3)
                                       : (uint8_t)0;
    }
}

// Levels of 8 codes at once, in registers: w holds 8 nibbles (code j in
// nibble j).  The codebook is symmetric (level n = -level 15 - n), so nibble n
// names magnitude m = n - 8 (n >= 8) or 7 - n (n < 8) of the 8 positive fp16
// levels, whose low bytes are tl[0..1] and high bytes th[0..1] (byte m of the
// pair); byte permutes gather them and the sign bit comes from the nibble.
// o[k] = the fp16 pair (level of nibble 2k, level of nibble 2k + 1).
__device__ __forceinline__ void turbo4_levels8(uint32_t w, const uint32_t (&tl)[2],
                                               const uint32_t (&th)[2], uint32_t (&o)[4])
{
    const uint32_t neg = ~w & 0x88888888u;                      // nibble < 8: negative
    const uint32_t m = (w ^ ((neg >> 3) * 7u)) & 0x77777777u;   // magnitude index
    const uint32_t lo0 = __byte_perm(tl[0], tl[1], m), hi0 = __byte_perm(th[0], th[1], m);
    const uint32_t lo1 = __byte_perm(tl[0], tl[1], m >> 16), hi1 = __byte_perm(th[0], th[1], m >> 16);
    o[0] = __byte_perm(lo0, hi0, 0x5140) ^ (((neg << 12) & 0x8000u) | ((neg << 24) & 0x80000000u));
    o[1] = __byte_perm(lo0, hi0, 0x7362) ^ (((neg << 4) & 0x8000u) | ((neg << 16) & 0x80000000u));
    o[2] = __byte_perm(lo1, hi1, 0x5140) ^ (((neg >> 4) & 0x8000u) | ((neg << 8) & 0x80000000u));
    o[3] = __byte_perm(lo1, hi1, 0x7362) ^ (((neg >> 12) & 0x8000u) | (neg & 0x80000000u));
}

// fp16 value of an E4M3 byte (exact: every E4M3 value is an fp16 value)
__device__ __forceinline__ __half e4m3_to_half(uint8_t b)
{
    return __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3));
}

}  // namespace gattn
