// hostpack.cpp -- host quantizer + packer into the interchange layout
// (LSB-first code bitstream per row; bf16 scales/biases [N][K/group]).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "gattn.h"

namespace {

// Nearest-even bf16 of a double, by integer rounding of the 53-bit significand
// at the bf16 precision of its binade (7 fraction bits; fewer below 2^-126).
uint16_t bf16_rne(double x)
{
    uint64_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000);
    const int biased = (int)((u >> 52) & 0x7FF);
    const uint64_t frac = u & ((1ull << 52) - 1);
    if (biased == 0x7FF)
        return frac ? (uint16_t)0x7FC0 : (uint16_t)(sign | 0x7F80);
    if (biased == 0)            // double subnormals are far below bf16's range
        return sign;
    const int E = biased - 1023;
    const uint64_t sig = (1ull << 52) | frac;
    int drop = 45;              // 52 - 7 fraction bits
    if (E < -126)
        drop += -126 - E;
    if (drop > 54)
        return sign;
    uint64_t r = sig >> drop;
    const uint64_t rem = sig & ((1ull << drop) - 1);
    const uint64_t half = 1ull << (drop - 1);
    if (rem > half || (rem == half && (r & 1)))
        ++r;
    const double v = std::ldexp((double)r, E - 52 + drop);
    if (v >= 0x1p128)
        return sign | 0x7F80;
    const float f = (float)v;
    uint32_t b;
    std::memcpy(&b, &f, sizeof b);
    return sign | (uint16_t)((b >> 16) & 0x7FFF);
}

double bf16_value(uint16_t h)
{
    const uint32_t b = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &b, sizeof f);
    return (double)f;
}

}  // namespace

extern "C" gattn_status gattn_pack_affine_host(const float *w, int64_t N, int64_t K, int32_t bits,
                                               int32_t group, uint32_t *packed, uint16_t *scales,
                                               uint16_t *biases)
{
    if (!w || !packed || !scales || !biases || N <= 0 || K <= 0 || bits < 1 || bits > 8 ||
        group <= 0 || K % group || (K * bits) % 32)
        return GATTN_E_INVALID_ARG;
    const int64_t words = K * bits / 32, groups = K / group;
    const double levels = (double)((1u << bits) - 1u);
    std::memset(packed, 0, (size_t)(N * words) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n) {
        uint32_t *row = packed + n * words;
        for (int64_t g = 0; g < groups; ++g) {
            const float *src = w + n * K + g * group;
            double lo = src[0], hi = src[0];
            for (int j = 1; j < group; ++j) {
                lo = src[j] < lo ? src[j] : lo;
                hi = src[j] > hi ? src[j] : hi;
            }
            const uint16_t bb = bf16_rne(lo), sb = bf16_rne((hi - lo) / levels);
            biases[n * groups + g] = bb;
            scales[n * groups + g] = sb;
            const double b = bf16_value(bb), s = bf16_value(sb);
            for (int j = 0; j < group; ++j) {
                uint32_t code = 0;
                if (s != 0.0) {
                    double q = std::nearbyint(((double)src[j] - b) / s);
                    q = q < 0.0 ? 0.0 : (q > levels ? levels : q);
                    code = (uint32_t)q;
                }
                const int64_t bit = (g * group + j) * bits;
                const int64_t wi = bit >> 5;
                const int sh = (int)(bit & 31);
                row[wi] |= code << sh;
                if (sh + bits > 32)
                    row[wi + 1] |= code >> (32 - sh);
            }
        }
    }
    return GATTN_OK;
}
