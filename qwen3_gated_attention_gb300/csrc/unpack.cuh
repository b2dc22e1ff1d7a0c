// unpack.cuh -- packed affine codes -> exact fp16 tensor-core A fragments.
//
// Codes are unsigned integers below 2^bits <= 256; placed in the mantissa of
// fp16 1024 (0x6400) they give 1024 + q exactly, and one subtraction leaves q.
// The lane-stream code order of the device tile layout makes every fragment
// register one mask (4-bit), one byte permute (8-bit) or two funnel-shifted
// extracts (other widths) away from its packed word.
#pragma once

#include "common.cuh"

namespace gattn {

__device__ __forceinline__ uint32_t h2_sub_1024(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    h = __hsub2(h, __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<uint32_t *>(&h);
}

// (1024 + 16 n) / 16 - 64 = n, exact in fp16
__device__ __forceinline__ uint32_t h2_div16_sub64(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    h = __hfma2(h, __half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00)),
                __half2(__ushort_as_half(0xD400), __ushort_as_half(0xD400)));
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t *cw, int off)
{
    const int word = off >> 5, sh = off & 31;
    const uint32_t mask = (1u << BITS) - 1u;
    if (sh + BITS <= 32)
        return (cw[word] >> sh) & mask;
    return __funnelshift_r(cw[word], cw[word + 1], sh) & mask;
}

// Exact fp16 codes of the A fragment of MMA mi from the lane's code stream.
template <int BITS>
__device__ __forceinline__ void unpack_a(const uint32_t *cw, int mi, uint32_t (&A)[4])
{
    if constexpr (BITS == 8) {
        const uint32_t w0 = cw[2 * mi], w1 = cw[2 * mi + 1];
        A[0] = h2_sub_1024(__byte_perm(w0, 0x64646464u, 0x4140));
        A[1] = h2_sub_1024(__byte_perm(w0, 0x64646464u, 0x4342));
        A[2] = h2_sub_1024(__byte_perm(w1, 0x64646464u, 0x4140));
        A[3] = h2_sub_1024(__byte_perm(w1, 0x64646464u, 0x4342));
    } else if constexpr (BITS == 4) {
        const uint32_t w = cw[mi], w8 = w >> 8;
        A[0] = h2_sub_1024((w & 0x000F000Fu) | 0x64006400u);
        A[1] = h2_div16_sub64((w & 0x00F000F0u) | 0x64006400u);
        A[2] = h2_sub_1024((w8 & 0x000F000Fu) | 0x64006400u);
        A[3] = h2_div16_sub64((w8 & 0x00F000F0u) | 0x64006400u);
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int off = (mi * 8 + 2 * p) * BITS;
            const uint32_t c0 = code_at<BITS>(cw, off), c1 = code_at<BITS>(cw, off + BITS);
            A[p] = h2_sub_1024(c0 | (c1 << 16) | 0x64006400u);
        }
    }
}

// The A fragment of MMA mi with each code q as the fp16 bit pattern q itself:
// the subnormal q * 2^-24, exact (q < 2^10).  Products with fp16 x are exact in
// fp32, so the tensor cores return 2^-24 * sum q * x, which the projection
// scales back when it folds a group (scale * 2^24).  4-bit codes in the high
// nibble of a byte (A[1], A[3]: rows g + 8 of the fragment) stay in place,
// 16 q * 2^-24, and their rows fold with scale * 2^20.  One mask or one byte
// permute per register.
template <int BITS>
__device__ __forceinline__ void unpack_a_sub(const uint32_t *cw, int mi, uint32_t (&A)[4])
{
    if constexpr (BITS == 8) {
        const uint32_t w0 = cw[2 * mi], w1 = cw[2 * mi + 1];
        A[0] = __byte_perm(w0, 0u, 0x4140);
        A[1] = __byte_perm(w0, 0u, 0x4342);
        A[2] = __byte_perm(w1, 0u, 0x4140);
        A[3] = __byte_perm(w1, 0u, 0x4342);
    } else if constexpr (BITS == 4) {
        const uint32_t w = cw[mi], w8 = w >> 8;
        A[0] = w & 0x000F000Fu;
        A[1] = w & 0x00F000F0u;
        A[2] = w8 & 0x000F000Fu;
        A[3] = w8 & 0x00F000F0u;
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int off = (mi * 8 + 2 * p) * BITS;
            const uint32_t c0 = code_at<BITS>(cw, off), c1 = code_at<BITS>(cw, off + BITS);
            A[p] = c0 | (c1 << 16);
        }
    }
}

}  // namespace gattn
