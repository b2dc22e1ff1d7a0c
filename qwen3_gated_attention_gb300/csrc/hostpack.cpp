// hostpack.cpp -- host quantizer + packer into the interchange layout
// (LSB-first code bitstream per row; bf16 scales/biases [N][K/group]).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

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

// ------------------------------------------------------------- Turbo4 tables
//
// The 16-level Lloyd-Max quantizer of N(0, 1) (the codebook of the Turbo4
// V-cache format): symmetric, so only the 8 positive levels are iterated.
// Lloyd's iteration alternates the decision points (midpoints of adjacent
// levels; 0 between the two innermost) and the levels (the mean of N(0, 1)
// over each cell, phi(a) - phi(b) over its upper-tail mass Q(a) - Q(b)),
// starting from evenly spaced levels and running to its fixed point.
namespace {

void lloyd_max16(double pos[8])
{
    const double inv_sqrt_2pi = 0.39894228040143267794, inv_sqrt2 = 0.70710678118654752440;
    auto pdf = [&](double x) { return std::isinf(x) ? 0.0 : inv_sqrt_2pi * std::exp(-0.5 * x * x); };
    auto upper = [&](double x) { return 0.5 * std::erfc(x * inv_sqrt2); };
    for (int k = 0; k < 8; ++k)
        pos[k] = 3.0 * (k + 0.5) / 8.0;
    for (int round = 0; round < 4000; ++round) {
        double edge[9];
        edge[0] = 0.0;
        for (int k = 1; k < 8; ++k)
            edge[k] = 0.5 * (pos[k - 1] + pos[k]);
        edge[8] = INFINITY;
        for (int k = 0; k < 8; ++k)
            pos[k] = (pdf(edge[k]) - pdf(edge[k + 1])) / (upper(edge[k]) - upper(edge[k + 1]));
    }
}

}  // namespace

extern "C" gattn_status gattn_turbo4_codebook(float levels[16], float thresholds[15])
{
    if (!levels || !thresholds)
        return GATTN_E_INVALID_ARG;
    static double pos[8];
    static std::once_flag once;
    std::call_once(once, [] { lloyd_max16(pos); });
    double c[16];
    for (int k = 0; k < 8; ++k) {
        c[8 + k] = pos[k];
        c[7 - k] = -pos[k];
    }
    for (int j = 0; j < 16; ++j)
        levels[j] = (float)c[j];
    for (int j = 0; j < 15; ++j)
        thresholds[j] = (float)(0.5 * (c[j] + c[j + 1]));
    return GATTN_OK;
}
