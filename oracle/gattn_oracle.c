/*
 * gattn_oracle.c -- the parity oracle for the gated full-attention decoder layer
 * (Qwen3.5 family) at decode / speculative-verify time.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded float64 CPU
 * statement of what the layer computes.  It shares no code, header, table or
 * constant generator with the CUDA library; only the tests, the smoke check and
 * the bench's CPU-baseline leg may load it.  The product path never calls it.
 *
 * Sources (page titles, with the section of each page that fixes the step):
 *   [mlxd#99]   "feat(engine): stage D6 - qwen3_5 dense full-attn deltas"
 *               (Summary; Audit table; review Issue 2 and the rope-dims reply)
 *   [DS4#113]   DS4Server issue 113, "Reproduction and boundary" (head-chunk plan)
 *   [TF#503]    TensorFold issue 503, "Option C: a generic affine row decoder"
 *   [atlas-mod] Atlas spark_model/forward/qwen3_5/mod.rs (Qwen35ForwardConfig,
 *               q_total/q_only/kv_dim, LayerKvCache, FullAttentionScratch)
 *
 * Readings taken where the pages are silent (each is listed with its reason in
 * the design notes):
 *   - packed codes: each weight row is an LSB-first bitstream of `bits`-wide
 *     unsigned codes stored as little-endian uint32 words; scales and biases
 *     are bf16 [N][K/group]; w = scale*q + bias  ([TF#503] "packed-row affine").
 *   - q_proj rows of head h: [h*2d, h*2d+d) are the query, [h*2d+d, (h+1)*2d)
 *     the gate (contiguous halves of the [num_heads, 2*head_dim] view).
 *   - RMSNorm: x / sqrt(mean(x^2) + eps) * w (stored weight, no 1+w offset).
 *   - RoPE: rotate-half pairs (i, i+rd/2) inside the first rd dims,
 *     inv_freq_i = theta^(-2i/rd), plain 1-D position cache_pos + r.
 *   - softmax scale 1/sqrt(head_dim); KV head of query head h is h / gqa.
 *   - new K/V rows are rounded to bf16 (nearest-even) into the cache and the
 *     attention reads them back from the cache.
 *   - verify rows: row r attends cache positions t <= cache_pos + r.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_E_ARG 1
#define ORC_E_RANGE 2

/* ---------------------------------------------------------------- bf16 */

double orc_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double straight to bf16 (8 significant bits, float's exponent
 * range), ties to even.  No intermediate float rounding. */
uint16_t orc_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isinf(ax))
        return sign | 0x7F80;
    if (ax == 0.0)
        return sign;
    int e;
    frexp(ax, &e);             /* ax = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;          /* spacing of 8-bit significands at this binade */
    if (qexp < -133)           /* bf16 subnormal spacing */
        qexp = -133;
    double r = nearbyint(ldexp(ax, -qexp));  /* ties-to-even (default mode) */
    r = ldexp(r, qexp);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r;        /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ------------------------------------------------- affine group quantization */

static void put_code(uint32_t *row, int64_t j, int bits, uint32_t code)
{
    int64_t p = j * bits;
    int64_t w = p >> 5;
    int off = (int)(p & 31);
    row[w] |= code << off;
    if (off + bits > 32)
        row[w + 1] |= code >> (32 - off);
}

static uint32_t get_code(const uint32_t *row, int64_t j, int bits)
{
    int64_t p = j * bits;
    int64_t w = p >> 5;
    int off = (int)(p & 31);
    uint64_t lo = row[w];
    if (off + bits > 32)
        lo |= (uint64_t)row[w + 1] << 32;
    return (uint32_t)((lo >> off) & ((1u << bits) - 1u));
}

static int quant_args_ok(int64_t N, int64_t K, int bits, int group)
{
    if (N <= 0 || K <= 0 || bits < 1 || bits > 8 || group <= 0)
        return 0;
    if (K % group != 0 || (K * bits) % 32 != 0)
        return 0;
    return 1;
}

/* Synthetic-weight quantizer (only used to make inputs): per (row, group)
 * bias = bf16(min), scale = bf16((max-min)/(2^bits-1)),
 * q = clamp(nearest-even((w-bias)/scale), 0, 2^bits-1), q = 0 when scale = 0. */
int orc_quantize_affine(const double *w, int64_t N, int64_t K, int bits, int group,
                        uint32_t *packed, uint16_t *scales, uint16_t *biases)
{
    if (!quant_args_ok(N, K, bits, group))
        return ORC_E_ARG;
    int64_t words = K * bits / 32, G = K / group;
    double qmax = (double)((1u << bits) - 1u);
    memset(packed, 0, (size_t)(N * words) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const double *wg = w + n * K + g * group;
            double mn = wg[0], mx = wg[0];
            for (int j = 1; j < group; ++j) {
                if (wg[j] < mn) mn = wg[j];
                if (wg[j] > mx) mx = wg[j];
            }
            uint16_t bb = orc_bf16_from_double(mn);
            uint16_t sb = orc_bf16_from_double((mx - mn) / qmax);
            scales[n * G + g] = sb;
            biases[n * G + g] = bb;
            double b = orc_bf16_to_double(bb), s = orc_bf16_to_double(sb);
            for (int j = 0; j < group; ++j) {
                double q = 0.0;
                if (s != 0.0) {
                    q = nearbyint((wg[j] - b) / s);
                    if (q < 0.0) q = 0.0;
                    if (q > qmax) q = qmax;
                }
                put_code(packed + n * words, g * group + j, bits, (uint32_t)q);
            }
        }
    }
    return ORC_OK;
}

int orc_unpack_codes(const uint32_t *packed, int64_t N, int64_t K, int bits, uint8_t *codes)
{
    if (!quant_args_ok(N, K, bits, 32 / 32))
        return ORC_E_ARG;
    int64_t words = K * bits / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)get_code(packed + n * words, k, bits);
    return ORC_OK;
}

/* one dequantized row: w[k] = scale[g] * q[k] + bias[g] */
static void dequant_row(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                        int64_t n, int64_t K, int bits, int group, double *wrow)
{
    int64_t words = K * bits / 32, G = K / group;
    const uint32_t *row = packed + n * words;
    for (int64_t g = 0; g < G; ++g) {
        double s = orc_bf16_to_double(scales[n * G + g]);
        double b = orc_bf16_to_double(biases[n * G + g]);
        for (int j = 0; j < group; ++j) {
            int64_t k = g * group + j;
            wrow[k] = s * (double)get_code(row, k, bits) + b;
        }
    }
}

int orc_dequantize(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                   int64_t N, int64_t K, int bits, int group, double *W)
{
    if (!quant_args_ok(N, K, bits, group))
        return ORC_E_ARG;
    for (int64_t n = 0; n < N; ++n)
        dequant_row(packed, scales, biases, n, K, bits, group, W + n * K);
    return ORC_OK;
}

/* y[m][n] = sum_k W[n][k] x[m][k] for M input rows, W dequantized row by row. */
static void qmatvec(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                    int64_t N, int64_t K, int bits, int group,
                    const double *x, int M, double *y, int64_t ystride, double *wrow)
{
    for (int64_t n = 0; n < N; ++n) {
        dequant_row(packed, scales, biases, n, K, bits, group, wrow);
        for (int m = 0; m < M; ++m) {
            const double *xm = x + (int64_t)m * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += wrow[k] * xm[k];
            y[(int64_t)m * ystride + n] = acc;
        }
    }
}

int orc_qmatvec(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                int64_t N, int64_t K, int bits, int group, const double *x, int M, double *y)
{
    if (!quant_args_ok(N, K, bits, group) || M <= 0)
        return ORC_E_ARG;
    double *wrow = (double *)malloc((size_t)K * sizeof(double));
    if (!wrow)
        return ORC_E_ARG;
    qmatvec(packed, scales, biases, N, K, bits, group, x, M, y, N, wrow);
    free(wrow);
    return ORC_OK;
}

/* ------------------------------------------------------ norm and rotary */

/* y = x / sqrt(mean(x^2) + eps) * w   ([mlxd#99] Audit: has_qk_norm) */
void orc_rms_norm(const double *x, int n, const double *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i)
        y[i] = x[i] * inv * w[i];
}

/* rotary dims = trunc(head_dim * partial_rotary_factor) ([mlxd#99] rope dims;
 * [atlas-mod] rotary_dim = head_dim * partial_rotary_factor) */
int orc_rotary_dims(int head_dim, double partial_rotary_factor)
{
    return (int)((double)head_dim * partial_rotary_factor);
}

/* Mutation switches: each plants one plausible mistake so the tests can show
 * that their pins and tolerances catch it.  0 = the layer as the pages define it. */
enum {
    ORC_MUT_NONE = 0,
    ORC_MUT_NO_GATE = 1,        /* o_proj(attn) instead of o_proj(attn*sigmoid(gate)) */
    ORC_MUT_ROTATE_ALL = 2,     /* rotary over all head_dim dims */
    ORC_MUT_PAIR_ADJACENT = 3,  /* pairs (2i, 2i+1) instead of (i, i+rd/2) */
    ORC_MUT_GQA_MODULO = 4,     /* kv head h % Hk instead of h / gqa */
    ORC_MUT_FREQ_BASE_D = 5,    /* inv_freq exponent over head_dim, not rd */
    ORC_MUT_NO_CAUSAL = 6,      /* every verify row sees all new rows */
    ORC_MUT_SPLIT_ALTERNATE = 7,/* query/gate taken element-wise alternating */
    ORC_MUT_NO_KNORM = 8,       /* skip the K RMSNorm */
    ORC_MUT_NO_BF16_CACHE = 9,  /* attend the new rows unrounded */
    ORC_MUT_TURBO_NO_IWHT = 10, /* Turbo4 V: dequantize without rotating back */
};

/* x[0..d) rotated in place at position pos; only dims [0, rd) move. */
static void rope_partial(double *x, int d, int rd, double pos, double theta, int mutate)
{
    if (mutate == ORC_MUT_ROTATE_ALL)
        rd = d;
    int half = rd / 2;
    double base_dims = (mutate == ORC_MUT_FREQ_BASE_D) ? (double)d : (double)rd;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / base_dims);
        double a = pos * inv_freq;
        double c = cos(a), s = sin(a);
        int i1 = i, i2 = i + half;
        if (mutate == ORC_MUT_PAIR_ADJACENT) {
            i1 = 2 * i;
            i2 = 2 * i + 1;
        }
        double x1 = x[i1], x2 = x[i2];
        x[i1] = x1 * c - x2 * s;
        x[i2] = x2 * c + x1 * s;
    }
}

void orc_rope(double *x, int d, int rd, double pos, double theta)
{
    rope_partial(x, d, rd, pos, theta, ORC_MUT_NONE);
}

/* ------------------------------------------------------ head-chunk plan */

/* [DS4#113] "Reproduction and boundary": when q_len * gqa > 32 and q_len <= 32
 * the query heads of each KV group are cut into chunks of
 * max(1, min(gqa, 32 / q_len)) heads (last chunk = the remainder), in head
 * order.  Otherwise (or with the route off) each KV group is one chunk.
 * Writes up to `cap` chunks; returns the chunk count, or -1 on bad input. */
int orc_head_chunk_plan(int q_len, int num_heads, int num_kv_heads, int enabled,
                        int32_t *first, int32_t *len, int cap)
{
    if (q_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
        return -1;
    int gqa = num_heads / num_kv_heads;
    int per = gqa;
    if (enabled && q_len * gqa > 32 && q_len <= 32) {
        per = 32 / q_len;
        if (per > gqa) per = gqa;
        if (per < 1) per = 1;
    }
    int count = 0;
    for (int g = 0; g < num_kv_heads; ++g) {
        for (int h0 = 0; h0 < gqa; h0 += per) {
            int n = (gqa - h0 < per) ? gqa - h0 : per;
            if (count < cap) {
                first[count] = g * gqa + h0;
                len[count] = n;
            }
            ++count;
        }
    }
    return count;
}

/* ------------------------------------------------------------- the layer */

typedef struct orc_layer {
    int32_t hidden, num_heads, num_kv_heads, head_dim;
    double partial_rotary_factor, rope_theta, rms_eps;
    int32_t bits[4], group[4];     /* q, k, v, o */
    int32_t head_chunk;            /* 1: attend chunk by chunk along the plan */
    int32_t mutate;                /* ORC_MUT_* (tests only) */
} orc_layer;

typedef struct orc_weights {
    const uint32_t *packed[4];
    const uint16_t *scales[4];
    const uint16_t *biases[4];
    const uint16_t *q_norm, *k_norm;   /* bf16 [head_dim] */
} orc_weights;

/* Causal scaled-dot-product attention of one query head, one verify row,
 * against the cache of its KV head: scores q.k/sqrt(d) over t in [0, last],
 * softmax exp(s - max)/sum, output sum p_t v_t. */
static void sdpa_row(const double *q, const uint16_t *kc, const uint16_t *vc, int64_t tstride,
                     int d, int last, const uint8_t *keep, double *o, double *scores)
{
    double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int t = 0; t <= last; ++t) {
        if (keep && !keep[t]) {
            scores[t] = -INFINITY;
            continue;
        }
        const uint16_t *kt = kc + (int64_t)t * tstride;
        double s = 0.0;
        for (int j = 0; j < d; ++j)
            s += q[j] * orc_bf16_to_double(kt[j]);
        s *= scale;
        scores[t] = s;
        if (s > mx) mx = s;
    }
    for (int j = 0; j < d; ++j)
        o[j] = 0.0;
    if (mx == -INFINITY)            /* every position masked out: a zero row */
        return;
    double z = 0.0;
    for (int t = 0; t <= last; ++t) {
        scores[t] = exp(scores[t] - mx);
        z += scores[t];
    }
    for (int t = 0; t <= last; ++t) {
        const uint16_t *vt = vc + (int64_t)t * tstride;
        double p = scores[t] / z;
        for (int j = 0; j < d; ++j)
            o[j] += p * orc_bf16_to_double(vt[j]);
    }
}

/* Public for the SDPA pins: rows x heads of one sequence.
 * q [n_heads][R][d] (query heads h0 .. h0+n_heads-1), cache [Hk][cap][d] bf16,
 * row r of every head attends t <= pos0 + r.  out [n_heads][R][d]. */
int orc_sdpa(const double *q, const uint16_t *cache_k, const uint16_t *cache_v,
             int num_heads, int num_kv_heads, int head_dim, int capacity,
             int h0, int n_heads, int R, int pos0, double *out)
{
    if (num_heads % num_kv_heads || pos0 < 0 || pos0 + R > capacity)
        return ORC_E_ARG;
    int gqa = num_heads / num_kv_heads;
    double *scores = (double *)malloc((size_t)capacity * sizeof(double));
    if (!scores)
        return ORC_E_ARG;
    for (int i = 0; i < n_heads; ++i) {
        int h = h0 + i, kh = h / gqa;
        const uint16_t *kc = cache_k + (int64_t)kh * capacity * head_dim;
        const uint16_t *vc = cache_v + (int64_t)kh * capacity * head_dim;
        for (int r = 0; r < R; ++r)
            sdpa_row(q + ((int64_t)i * R + r) * head_dim, kc, vc, head_dim, head_dim,
                     pos0 + r, NULL, out + ((int64_t)i * R + r) * head_dim, scores);
    }
    free(scores);
    return ORC_OK;
}

/* ------------------------------------------------ Turbo4 V cache
 *
 * [atlas-mod] MetalKvDtype / LayerKvCache: the Bf16KTurbo4V format keeps K as
 * raw bf16 and stores V in a Walsh-Hadamard-rotated basis as 4-bit Lloyd-Max
 * codebook indices (two per byte) with one FP8 E4M3 scale per group of 16
 * coordinates ("matched-norm L2"); the attention output is rotated back.  The
 * pages name the parts, not the formulas; the readings taken:
 *   - rotation: y = H v / sqrt(d), H the Sylvester Hadamard matrix of order d
 *     (natural order), by the fast transform with stages h = 1, 2, 4, ...
 *   - codebook: the 16-level Lloyd-Max quantizer of N(0, 1), levels ascending,
 *     index j for level j; a group's coordinates are divided by the group's RMS
 *     and each takes the nearest level (a tie goes to the lower level).
 *   - scale: s = ||y_g|| / ||c(idx_g)||, so the dequantized group keeps the
 *     group's L2 norm; stored as E4M3 (nearest, ties to even, saturating).
 *   - input: the bf16 V row the cache would otherwise hold.  The quantizer's
 *     decisions (codes, scale byte) are taken in fp32 in a fixed order: the
 *     butterfly stages in order, the 1/sqrt(d) factor (rounded to fp32) after
 *     them, pairwise sums over each group ((a0+a1)+(a2+a3))+..., correctly
 *     rounded sqrt and division.  A kernel taking them the same way agrees
 *     bit for bit.
 *   - byte j/2 of a row holds code j in its low nibble (j even) or its high
 *     nibble (j odd); row r of a (sequence, KV head) is d/2 code bytes and d/16
 *     scale bytes, rows in token order.
 *   - dequantized row: v = H (s * c(idx)) / sqrt(d), in float64.
 */

/* E4M3 (OCP FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities, S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9. */
double orc_e4m3_to_double(uint8_t b)
{
    const int e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (b & 0x80) ? -v : v;
}

/* Nearest E4M3 value, ties to the even mantissa, magnitudes past 448
 * saturating to 448; NaN gives the NaN byte. */
uint8_t orc_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int e2;
    frexp(a, &e2);
    int be = e2 - 1;                    /* a in [2^be, 2^(be+1)) */
    if (be < -6)
        be = -6;                        /* subnormal quantum below 2^-6 */
    const double q = ldexp(1.0, be - 3);
    const double n = nearbyint(a / q);  /* a / q is exact; ties to even */
    const double v = n * q;
    if (v == 0.0)
        return sign;
    frexp(v, &e2);
    const int bv = e2 - 1;
    if (bv < -6)
        return sign | (uint8_t)(v / ldexp(1.0, -9));
    return sign | (uint8_t)((bv + 7) << 3) | (uint8_t)(v / ldexp(1.0, bv - 3) - 8.0);
}

static double gauss_pdf(double x)
{
    return isinf(x) ? 0.0 : exp(-0.5 * x * x) / sqrt(6.283185307179586476925);
}

/* P(a < X < b) for X ~ N(0, 1), from the tail on the side of the cell */
static double gauss_mass(double a, double b)
{
    const double r2 = 1.4142135623730950488;
    if (a >= 0.0)
        return 0.5 * (erfc(a / r2) - erfc(b / r2));
    return 0.5 * (erfc(-b / r2) - erfc(-a / r2));
}

/* The 16 levels of the Lloyd-Max quantizer of N(0, 1): Lloyd's iteration
 * (thresholds at the midpoints of the levels, each level the mean of N(0, 1)
 * over its cell) from 16 evenly spaced levels on [-3, 3], run to its fixed
 * point (it settles to rounding noise in under a thousand rounds). */
void orc_turbo4_codebook(double c[16])
{
    static double cached[16];
    static int have = 0;            /* the oracle is single-threaded */
    if (have) {
        memcpy(c, cached, sizeof(cached));
        return;
    }
    double lv[16], t[17];
    for (int j = 0; j < 16; ++j)
        lv[j] = -3.0 + 6.0 * (j + 0.5) / 16.0;
    for (int it = 0; it < 4000; ++it) {
        t[0] = -INFINITY;
        t[16] = INFINITY;
        for (int j = 1; j < 16; ++j)
            t[j] = 0.5 * (lv[j - 1] + lv[j]);
        for (int j = 0; j < 16; ++j)
            lv[j] = (gauss_pdf(t[j]) - gauss_pdf(t[j + 1])) / gauss_mass(t[j], t[j + 1]);
    }
    memcpy(cached, lv, sizeof(lv));
    have = 1;
    memcpy(c, lv, sizeof(lv));
}

/* fp32 levels and the 15 decision thresholds between them (midpoints taken
 * in double, then rounded) */
void orc_turbo4_tables_f32(float levels[16], float thresholds[15])
{
    double c[16];
    orc_turbo4_codebook(c);
    for (int j = 0; j < 16; ++j)
        levels[j] = (float)c[j];
    for (int j = 0; j < 15; ++j)
        thresholds[j] = (float)(0.5 * (c[j] + c[j + 1]));
}

static float pairwise16(const float *a)
{
    float t[16];
    memcpy(t, a, sizeof(t));
    for (int w = 1; w < 16; w <<= 1)
        for (int i = 0; i < 16; i += 2 * w)
            t[i] = t[i] + t[i + w];
    return t[0];
}

/* n rows of d bf16 values -> codes [n][d/2] and scales [n][d/16] */
int orc_turbo4_quantize_rows(const uint16_t *v, int64_t n, int d, uint8_t *codes, uint8_t *scales)
{
    if (d < 16 || d > 1024 || (d & (d - 1)) || n < 0)
        return ORC_E_ARG;
    float lv[16], th[15], y[1024], sq[16], cq[16];
    orc_turbo4_tables_f32(lv, th);
    const float sc = (float)(1.0 / sqrt((double)d));
    for (int64_t row = 0; row < n; ++row) {
        const uint16_t *vr = v + row * d;
        uint8_t *cr = codes + row * (d / 2), *sr = scales + row * (d / 16);
        for (int j = 0; j < d; ++j)
            y[j] = (float)orc_bf16_to_double(vr[j]);
        for (int h = 1; h < d; h <<= 1)
            for (int i = 0; i < d; ++i)
                if (!(i & h)) {
                    const float a = y[i], b = y[i + h];
                    y[i] = a + b;
                    y[i + h] = a - b;
                }
        for (int j = 0; j < d; ++j)
            y[j] = y[j] * sc;
        for (int g = 0; g < d / 16; ++g) {
            const float *yg = y + 16 * g;
            uint8_t idx[16];
            for (int i = 0; i < 16; ++i)
                sq[i] = yg[i] * yg[i];
            const float ss = pairwise16(sq);
            if (ss == 0.0f) {
                memset(idx, 0, sizeof(idx));
                sr[g] = 0;
            } else {
                const float r = sqrtf(ss * 0.0625f);
                for (int i = 0; i < 16; ++i) {
                    const float u = yg[i] / r;
                    int k = 0;
                    while (k < 15 && u > th[k])
                        ++k;
                    idx[i] = (uint8_t)k;
                    cq[i] = lv[k] * lv[k];
                }
                const float cs = pairwise16(cq);
                sr[g] = orc_e4m3_from_float(sqrtf(ss / cs));
            }
            for (int i = 0; i < 16; i += 2)
                cr[8 * g + i / 2] = (uint8_t)(idx[i] | (idx[i + 1] << 4));
        }
    }
    return ORC_OK;
}

/* n code rows -> float64 rows [n][d] in the original basis */
static void turbo4_dequant(const uint8_t *codes, const uint8_t *scales, int64_t n, int d,
                           const double *c, int mutate, double *out)
{
    const double sc = 1.0 / sqrt((double)d);
    for (int64_t row = 0; row < n; ++row) {
        const uint8_t *cr = codes + row * (d / 2), *sr = scales + row * (d / 16);
        double *y = out + row * d;
        for (int j = 0; j < d; ++j)
            y[j] = orc_e4m3_to_double(sr[j / 16]) * c[(cr[j / 2] >> (4 * (j & 1))) & 15];
        if (mutate == ORC_MUT_TURBO_NO_IWHT)
            continue;
        for (int h = 1; h < d; h <<= 1)
            for (int i = 0; i < d; ++i)
                if (!(i & h)) {
                    const double a = y[i], b = y[i + h];
                    y[i] = a + b;
                    y[i + h] = a - b;
                }
        for (int j = 0; j < d; ++j)
            y[j] *= sc;
    }
}

int orc_turbo4_dequant_rows(const uint8_t *codes, const uint8_t *scales, int64_t n, int d,
                            int mutate, double *out)
{
    if (d < 16 || d > 1024 || (d & (d - 1)) || n < 0)
        return ORC_E_ARG;
    double c[16];
    orc_turbo4_codebook(c);
    turbo4_dequant(codes, scales, n, d, c, mutate, out);
    return ORC_OK;
}

/* sdpa_row over V rows given in float64 (a dequantized cache); K rows from
 * the bf16 cache kc, or from float64 rows kd (a dequantized Turbo4 K cache) */
static void sdpa_row_vd(const double *q, const uint16_t *kc, int64_t tstride, const double *vd,
                        int d, int last, const uint8_t *keep, double *o, double *scores,
                        const double *kd)
{
    double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int t = 0; t <= last; ++t) {
        if (keep && !keep[t]) {
            scores[t] = -INFINITY;
            continue;
        }
        double s = 0.0;
        if (kd) {
            for (int j = 0; j < d; ++j)
                s += q[j] * kd[(int64_t)t * d + j];
        } else {
            const uint16_t *kt = kc + (int64_t)t * tstride;
            for (int j = 0; j < d; ++j)
                s += q[j] * orc_bf16_to_double(kt[j]);
        }
        s *= scale;
        scores[t] = s;
        if (s > mx) mx = s;
    }
    for (int j = 0; j < d; ++j)
        o[j] = 0.0;
    if (mx == -INFINITY)
        return;
    double z = 0.0;
    for (int t = 0; t <= last; ++t) {
        scores[t] = exp(scores[t] - mx);
        z += scores[t];
    }
    for (int t = 0; t <= last; ++t) {
        const double p = scores[t] / z;
        for (int j = 0; j < d; ++j)
            o[j] += p * vd[(int64_t)t * d + j];
    }
}

/*
 * One layer step for B sequences of R new rows each.
 *   x        [B][R][hidden]                     layer input (exact values)
 *   cache_k/v [B][Hk][capacity][head_dim] bf16  read and appended in place
 *   cache_pos [B]                               first new position of each sequence
 *   out      [B][R][hidden]                     o_proj output, float64
 *   tap_y    [B][R][2*H*d + 2*Hk*d] or NULL     q_full | k | v before norm
 *   tap_attn [B][R][H][d] or NULL               attention output before the gate
 * Returns ORC_OK, ORC_E_ARG for an inadmissible layer, ORC_E_RANGE when a
 * sequence would write past the capacity (nothing is written for it).
 */
/* An attention mask ([DS4#113] "broadcast/head-specific masks"): byte
 * m[b*stride_batch + hm*stride_head + r*stride_row + t], nonzero = row r may
 * attend position t; hm = 0 for a broadcast mask (heads == 1), the query head
 * for a head-specific one (heads == num_heads).  Reading: a mask replaces the
 * causal rule (it carries it), positions run over [0, cache_pos + R), and a
 * row with no position left is a zero row.  len > 0: a row holds len
 * positions and the positions from len on are not attended (the library's
 * mask rows, `positions` long); len <= 0: every row covers [0, cache_pos + R). */
typedef struct orc_mask {
    const uint8_t *m;
    int32_t heads;
    int64_t stride_row, stride_head, stride_batch;
    int32_t len;
} orc_mask;

/* the last position a masked row may attend: cache_pos + R - 1, cut at the row's length */
static int mask_last(const orc_mask *M, int p0, int R)
{
    int last = p0 + R - 1;
    if (M->len > 0 && last > M->len - 1)
        last = M->len - 1;
    return last;
}

#define ORC_E_MASK 3

/* k_codes / k_scales (with v_codes / v_scales): the symmetric Turbo4 cache of
 * [atlas-mod] MetalKvDtype::Turbo4, K quantized like V (same rotation, codebook
 * and scales) from the bf16 row of the normed, rotated key; scores then use
 * the dequantized K rows.  cache_k is unused then. */
static int layer_step(const orc_layer *L, const orc_weights *W, const double *x,
                      uint16_t *cache_k, uint16_t *cache_v, uint8_t *v_codes, uint8_t *v_scales,
                      uint8_t *k_codes, uint8_t *k_scales,
                      int capacity, const int32_t *cache_pos, int B, int R, const orc_mask *M,
                      double *out, double *tap_y, double *tap_attn)
{
    const int turbo = v_codes != NULL;
    const int kturbo = k_codes != NULL;
    if (kturbo && (!turbo || !k_scales))
        return ORC_E_ARG;
    const int Hd = L->hidden, H = L->num_heads, Hk = L->num_kv_heads, d = L->head_dim;
    if (Hd <= 0 || H <= 0 || Hk <= 0 || d <= 0 || H % Hk || B <= 0 || R <= 0)
        return ORC_E_ARG;
    if (!(L->partial_rotary_factor > 0.0 && L->partial_rotary_factor <= 1.0))
        return ORC_E_ARG;
    int rd = orc_rotary_dims(d, L->partial_rotary_factor);
    if (rd < 2 || (rd & 1))
        return ORC_E_ARG;
    const int gqa = H / Hk;
    const int64_t Nq = 2LL * H * d, Nkv = (int64_t)Hk * d, Ny = Nq + 2 * Nkv;
    const int64_t Ka = Hd, Ko = (int64_t)H * d;
    const int64_t Ns[4] = {Nq, Nkv, Nkv, Hd};
    const int64_t Ks[4] = {Ka, Ka, Ka, Ko};
    for (int p = 0; p < 4; ++p)
        if (!quant_args_ok(Ns[p], Ks[p], L->bits[p], L->group[p]))
            return ORC_E_ARG;
    int rc = ORC_OK;

    int64_t maxK = Ka > Ko ? Ka : Ko;
    double *wrow = (double *)malloc((size_t)maxK * sizeof(double));
    double *y = (double *)malloc((size_t)(R * Ny) * sizeof(double));
    double *qn = (double *)malloc((size_t)((int64_t)R * H * d) * sizeof(double));
    double *attn = (double *)malloc((size_t)((int64_t)R * H * d) * sizeof(double));
    double *ga = (double *)malloc((size_t)(R * Ko) * sizeof(double));
    double *tmp = (double *)malloc((size_t)d * sizeof(double));
    double *nq = (double *)malloc((size_t)d * sizeof(double));
    double *nk = (double *)malloc((size_t)d * sizeof(double));
    double *scores = (double *)malloc((size_t)capacity * sizeof(double) + 8);
    double *knew = (double *)malloc((size_t)((int64_t)R * Hk * d) * sizeof(double));
    double *vnew = (double *)malloc((size_t)((int64_t)R * Hk * d) * sizeof(double));
    int32_t *cf = (int32_t *)malloc((size_t)H * sizeof(int32_t));
    int32_t *cl = (int32_t *)malloc((size_t)H * sizeof(int32_t));
    double *vdq = NULL, *kdq = NULL, cbk[16];
    uint16_t *vb16 = (uint16_t *)malloc((size_t)d * sizeof(uint16_t));
    if (turbo) {
        if (d < 16 || d > 1024 || (d & (d - 1))) {
            rc = ORC_E_ARG;
            goto done;
        }
        orc_turbo4_codebook(cbk);
        vdq = (double *)malloc((size_t)capacity * d * sizeof(double) + 8);
        if (kturbo)
            kdq = (double *)malloc((size_t)capacity * d * sizeof(double) + 8);
    }
    if (!wrow || !y || !qn || !attn || !ga || !tmp || !nq || !nk || !scores || !knew || !vnew || !cf ||
        !cl || !vb16 || (turbo && !vdq) || (kturbo && !kdq)) {
        rc = ORC_E_ARG;
        goto done;
    }
    for (int j = 0; j < d; ++j) {
        nq[j] = orc_bf16_to_double(W->q_norm[j]);
        nk[j] = orc_bf16_to_double(W->k_norm[j]);
    }
    int nchunks = orc_head_chunk_plan(R, H, Hk, L->head_chunk, cf, cl, H);
    if (M && M->heads != 1 && M->heads != H) {
        rc = ORC_E_ARG;
        goto done;
    }
    /* [DS4#113] the head-chunked route hands the mask unchanged to every head
     * chunk: a broadcast mask fits each chunk, a mask over all H heads does not */
    if (M && M->heads > 1 && nchunks > Hk) {
        rc = ORC_E_MASK;
        goto done;
    }

    for (int b = 0; b < B; ++b) {
        const int p0 = cache_pos[b];
        if (p0 < 0 || p0 + R > capacity) {
            rc = ORC_E_RANGE;
            continue;
        }
        const double *xb = x + (int64_t)b * R * Hd;
        /* projections: q_full (doubled q_proj), k, v  ([atlas-mod] q_total = 2*H*d) */
        for (int p = 0; p < 3; ++p) {
            int64_t off = (p == 0) ? 0 : (p == 1 ? Nq : Nq + Nkv);
            qmatvec(W->packed[p], W->scales[p], W->biases[p], Ns[p], Ka, L->bits[p], L->group[p],
                    xb, R, y + off, Ny, wrow);
        }
        if (tap_y)
            memcpy(tap_y + (int64_t)b * R * Ny, y, (size_t)(R * Ny) * sizeof(double));

        uint16_t *kcb = kturbo ? NULL : cache_k + (int64_t)b * Hk * capacity * d;
        uint16_t *vcb = turbo ? NULL : cache_v + (int64_t)b * Hk * capacity * d;
        for (int r = 0; r < R; ++r) {
            const double *yr = y + (int64_t)r * Ny;
            double pos = (double)(p0 + r);
            /* query heads: split [query | gate], RMSNorm, partial RoPE */
            for (int h = 0; h < H; ++h) {
                const double *src = yr + (int64_t)h * 2 * d;
                if (L->mutate == ORC_MUT_SPLIT_ALTERNATE)
                    for (int j = 0; j < d; ++j) tmp[j] = src[2 * j];
                else
                    memcpy(tmp, src, (size_t)d * sizeof(double));
                double *dst = qn + ((int64_t)r * H + h) * d;
                orc_rms_norm(tmp, d, nq, L->rms_eps, dst);
                rope_partial(dst, d, rd, pos, L->rope_theta, L->mutate);
            }
            /* KV heads: RMSNorm + RoPE on k, raw v; append at cache_pos + r as bf16 */
            for (int kh = 0; kh < Hk; ++kh) {
                double *kr = knew + ((int64_t)r * Hk + kh) * d;
                double *vr = vnew + ((int64_t)r * Hk + kh) * d;
                const double *ksrc = yr + Nq + (int64_t)kh * d;
                const double *vsrc = yr + Nq + Nkv + (int64_t)kh * d;
                if (L->mutate == ORC_MUT_NO_KNORM)
                    memcpy(kr, ksrc, (size_t)d * sizeof(double));
                else
                    orc_rms_norm(ksrc, d, nk, L->rms_eps, kr);
                rope_partial(kr, d, rd, pos, L->rope_theta, L->mutate);
                memcpy(vr, vsrc, (size_t)d * sizeof(double));
                if (kturbo) {
                    for (int j = 0; j < d; ++j)
                        vb16[j] = orc_bf16_from_double(kr[j]);
                    const int64_t row = ((int64_t)b * Hk + kh) * capacity + p0 + r;
                    orc_turbo4_quantize_rows(vb16, 1, d, k_codes + row * (d / 2),
                                             k_scales + row * (d / 16));
                } else {
                    uint16_t *kdst = kcb + ((int64_t)kh * capacity + p0 + r) * d;
                    for (int j = 0; j < d; ++j)
                        kdst[j] = orc_bf16_from_double(kr[j]);
                }
                for (int j = 0; j < d; ++j)
                    vb16[j] = orc_bf16_from_double(vr[j]);
                if (turbo) {
                    const int64_t row = ((int64_t)b * Hk + kh) * capacity + p0 + r;
                    orc_turbo4_quantize_rows(vb16, 1, d, v_codes + row * (d / 2),
                                             v_scales + row * (d / 16));
                } else {
                    memcpy(vcb + ((int64_t)kh * capacity + p0 + r) * d, vb16,
                           (size_t)d * sizeof(uint16_t));
                }
            }
        }
        /* Turbo4 V: per KV head, dequantize its rows [0, p0 + R) back to the
         * original basis, then attend them as float64 rows */
        if (turbo) {
            for (int kh = 0; kh < Hk; ++kh) {
                const int64_t row0 = ((int64_t)b * Hk + kh) * capacity;
                turbo4_dequant(v_codes + row0 * (d / 2), v_scales + row0 * (d / 16), p0 + R, d, cbk,
                               L->mutate, vdq);
                if (kturbo)
                    turbo4_dequant(k_codes + row0 * (d / 2), k_scales + row0 * (d / 16), p0 + R, d,
                                   cbk, L->mutate, kdq);
                for (int h = 0; h < H; ++h) {
                    const int khh = (L->mutate == ORC_MUT_GQA_MODULO) ? h % Hk : h / gqa;
                    if (khh != kh)
                        continue;
                    for (int r = 0; r < R; ++r) {
                        int last = (L->mutate == ORC_MUT_NO_CAUSAL) ? p0 + R - 1 : p0 + r;
                        const uint8_t *keep = NULL;
                        if (M) {
                            last = mask_last(M, p0, R);
                            keep = M->m + b * M->stride_batch + (M->heads > 1 ? h : 0) * M->stride_head +
                                   r * M->stride_row;
                        }
                        sdpa_row_vd(qn + ((int64_t)r * H + h) * d,
                                    kturbo ? NULL : kcb + (int64_t)kh * capacity * d, d, vdq, d, last,
                                    keep, attn + ((int64_t)r * H + h) * d, scores,
                                    kturbo ? kdq : NULL);
                    }
                }
            }
        }
        /* attention, chunk by chunk along the head plan (one chunk per KV
         * group when the route is off or ineligible) */
        for (int c = 0; c < (turbo ? 0 : nchunks); ++c) {
            for (int h = cf[c]; h < cf[c] + cl[c]; ++h) {
                int kh = (L->mutate == ORC_MUT_GQA_MODULO) ? h % Hk : h / gqa;
                const uint16_t *kc = kcb + (int64_t)kh * capacity * d;
                const uint16_t *vc = vcb + (int64_t)kh * capacity * d;
                for (int r = 0; r < R; ++r) {
                    int last = p0 + r;
                    if (L->mutate == ORC_MUT_NO_CAUSAL)
                        last = p0 + R - 1;
                    double *o = attn + ((int64_t)r * H + h) * d;
                    const double *qv = qn + ((int64_t)r * H + h) * d;
                    if (L->mutate == ORC_MUT_NO_BF16_CACHE) {
                        /* attend the unrounded new rows: a scratch copy of the
                         * cache rows is not kept, so recompute with doubles */
                        double scale = 1.0 / sqrt((double)d), mx = -INFINITY, z = 0.0;
                        for (int t = 0; t <= last; ++t) {
                            double s = 0.0;
                            for (int j = 0; j < d; ++j) {
                                double kv = (t >= p0) ? knew[((int64_t)(t - p0) * Hk + kh) * d + j]
                                                      : orc_bf16_to_double(kc[(int64_t)t * d + j]);
                                s += qv[j] * kv;
                            }
                            scores[t] = s * scale;
                            if (scores[t] > mx) mx = scores[t];
                        }
                        for (int t = 0; t <= last; ++t) { scores[t] = exp(scores[t] - mx); z += scores[t]; }
                        for (int j = 0; j < d; ++j) o[j] = 0.0;
                        for (int t = 0; t <= last; ++t)
                            for (int j = 0; j < d; ++j) {
                                double vv = (t >= p0) ? vnew[((int64_t)(t - p0) * Hk + kh) * d + j]
                                                      : orc_bf16_to_double(vc[(int64_t)t * d + j]);
                                o[j] += scores[t] / z * vv;
                            }
                    } else if (M) {
                        sdpa_row(qv, kc, vc, d, d, mask_last(M, p0, R),
                                 M->m + b * M->stride_batch + (M->heads > 1 ? h : 0) * M->stride_head +
                                     r * M->stride_row, o, scores);
                    } else {
                        sdpa_row(qv, kc, vc, d, d, last, NULL, o, scores);
                    }
                }
            }
        }
        if (tap_attn)
            memcpy(tap_attn + (int64_t)b * R * H * d, attn, (size_t)((int64_t)R * H * d) * sizeof(double));
        /* output gate and o_proj: out = Wo (attn * sigmoid(gate)) */
        for (int r = 0; r < R; ++r) {
            const double *yr = y + (int64_t)r * Ny;
            for (int h = 0; h < H; ++h)
                for (int j = 0; j < d; ++j) {
                    double g = (L->mutate == ORC_MUT_SPLIT_ALTERNATE) ? yr[(int64_t)h * 2 * d + 2 * j + 1]
                                                                      : yr[(int64_t)h * 2 * d + d + j];
                    double a = attn[((int64_t)r * H + h) * d + j];
                    ga[(int64_t)r * Ko + (int64_t)h * d + j] =
                        (L->mutate == ORC_MUT_NO_GATE) ? a : a * (1.0 / (1.0 + exp(-g)));
                }
        }
        qmatvec(W->packed[3], W->scales[3], W->biases[3], Hd, Ko, L->bits[3], L->group[3],
                ga, R, out + (int64_t)b * R * Hd, Hd, wrow);
    }
done:
    free(wrow); free(y); free(qn); free(attn); free(ga); free(tmp); free(nq); free(nk);
    free(scores); free(knew); free(vnew); free(cf); free(cl); free(vdq); free(kdq); free(vb16);
    return rc;
}

int orc_layer_step(const orc_layer *L, const orc_weights *W, const double *x,
                   uint16_t *cache_k, uint16_t *cache_v, int capacity,
                   const int32_t *cache_pos, int B, int R,
                   double *out, double *tap_y, double *tap_attn)
{
    return layer_step(L, W, x, cache_k, cache_v, NULL, NULL, NULL, NULL, capacity, cache_pos, B, R,
                      NULL, out, tap_y, tap_attn);
}

/* orc_layer_step with an attention mask (orc_mask above): mask bytes, heads
 * (1 or num_heads) and strides in bytes.  ORC_E_MASK when a head-specific
 * mask meets the head-chunked route. */
int orc_layer_step_masked(const orc_layer *L, const orc_weights *W, const double *x,
                          uint16_t *cache_k, uint16_t *cache_v, int capacity,
                          const int32_t *cache_pos, int B, int R, const uint8_t *mask,
                          int32_t mask_heads, int64_t stride_row, int64_t stride_head,
                          int64_t stride_batch, double *out, double *tap_y, double *tap_attn)
{
    if (!mask)
        return ORC_E_ARG;
    const orc_mask M = {mask, mask_heads, stride_row, stride_head, stride_batch, 0};
    return layer_step(L, W, x, cache_k, cache_v, NULL, NULL, NULL, NULL, capacity, cache_pos, B, R,
                      &M, out, tap_y, tap_attn);
}

/* The layer step over a Bf16KTurbo4V cache: K as in orc_layer_step, V as
 * code rows [B][Hk][capacity][d/2] and scale rows [B][Hk][capacity][d/16]
 * (Turbo4 V cache above); the new V rows are quantized from their bf16
 * values, attention reads every V row dequantized. */
int orc_layer_step_turbo4v(const orc_layer *L, const orc_weights *W, const double *x,
                           uint16_t *cache_k, uint8_t *v_codes, uint8_t *v_scales, int capacity,
                           const int32_t *cache_pos, int B, int R,
                           double *out, double *tap_y, double *tap_attn)
{
    if (!v_codes || !v_scales)
        return ORC_E_ARG;
    return layer_step(L, W, x, cache_k, NULL, v_codes, v_scales, NULL, NULL, capacity, cache_pos, B,
                      R, NULL, out, tap_y, tap_attn);
}

/* ------------------------------------------------------ decoder block */

/* The steps on either side of the layer in a decoder block ([atlas-mod]
 * forward_full_attention: norm -> projections -> attention -> residual +
 * post-norm -> MLP): per row of x [B][R][hidden],
 *   h          = RMSNorm(x) * input_ln
 *   out        = x + layer(h)                       (the residual stream)
 *   out_normed = RMSNorm(bf16(out)) * post_ln       (the MLP's input)
 * The residual stream is stored as bf16, and the post-norm reads the stored
 * row.  h is an activation of the residual stream's type: h_bf16 != 0 rounds
 * it to bf16 (a bf16 stream, as the engine's x_norm buffer), 0 keeps it exact
 * (an fp32 stream).  input_ln / post_ln are bf16 [hidden]; post_ln and
 * out_normed may be NULL.  Cache behaviour is that of orc_layer_step. */
/* The layer step's optional parts together: a Bf16KTurbo4V V cache (v_codes
 * and v_scales, else cache_v is a bf16 V cache) and an attention mask (mask
 * NULL: causal; orc_mask above). */
typedef struct orc_step_ext {
    uint8_t *v_codes, *v_scales;
    uint8_t *k_codes, *k_scales;       /* with v_*: the symmetric Turbo4 cache */
    const uint8_t *mask;
    int32_t mask_heads;
    int64_t mask_row, mask_head, mask_batch;
    int32_t mask_len;                  /* positions per mask row (orc_mask.len) */
} orc_step_ext;

int orc_layer_step_ext(const orc_layer *L, const orc_weights *W, const double *x,
                       uint16_t *cache_k, uint16_t *cache_v, int capacity,
                       const int32_t *cache_pos, int B, int R, const orc_step_ext *e,
                       double *out, double *tap_y, double *tap_attn)
{
    orc_mask M;
    const orc_mask *mp = NULL;
    if (e && e->mask) {
        M.m = e->mask;
        M.heads = e->mask_heads;
        M.stride_row = e->mask_row;
        M.stride_head = e->mask_head;
        M.stride_batch = e->mask_batch;
        M.len = e->mask_len;
        mp = &M;
    }
    uint8_t *vc = e ? e->v_codes : NULL, *vs = e ? e->v_scales : NULL;
    uint8_t *kc = e ? e->k_codes : NULL, *ks = e ? e->k_scales : NULL;
    if ((vc == NULL) != (vs == NULL) || (kc == NULL) != (ks == NULL))
        return ORC_E_ARG;
    return layer_step(L, W, x, kc ? NULL : cache_k, vc ? NULL : cache_v, vc, vs, kc, ks, capacity,
                      cache_pos, B, R, mp, out, tap_y, tap_attn);
}

static int block_step(const orc_layer *L, const orc_weights *W, const double *x, int h_bf16,
                      const uint16_t *input_ln, const uint16_t *post_ln,
                      uint16_t *cache_k, uint16_t *cache_v, int capacity,
                      const int32_t *cache_pos, int B, int R, const orc_step_ext *e,
                      double *out, double *out_normed)
{
    const int Hd = L->hidden;
    const int64_t M = (int64_t)B * R;
    double *w = malloc((size_t)Hd * sizeof(double));
    double *h = malloc((size_t)(M * Hd) * sizeof(double));
    double *y = malloc((size_t)(M * Hd) * sizeof(double));
    double *rb = malloc((size_t)Hd * sizeof(double));
    int rc = ORC_OK;
    if (!w || !h || !y || !rb) {
        rc = ORC_E_ARG;
        goto done;
    }
    for (int i = 0; i < Hd; ++i)
        w[i] = orc_bf16_to_double(input_ln[i]);
    for (int64_t m = 0; m < M; ++m)
        orc_rms_norm(x + m * Hd, Hd, w, L->rms_eps, h + m * Hd);
    if (h_bf16)
        for (int64_t j = 0; j < M * Hd; ++j)
            h[j] = orc_bf16_to_double(orc_bf16_from_double(h[j]));
    rc = orc_layer_step_ext(L, W, h, cache_k, cache_v, capacity, cache_pos, B, R, e, y, NULL, NULL);
    if (rc != ORC_OK)
        goto done;
    for (int64_t j = 0; j < M * Hd; ++j)
        out[j] = x[j] + y[j];
    if (post_ln && out_normed) {
        for (int i = 0; i < Hd; ++i)
            w[i] = orc_bf16_to_double(post_ln[i]);
        for (int64_t m = 0; m < M; ++m) {
            for (int i = 0; i < Hd; ++i)
                rb[i] = orc_bf16_to_double(orc_bf16_from_double(out[m * Hd + i]));
            orc_rms_norm(rb, Hd, w, L->rms_eps, out_normed + m * Hd);
        }
    }
done:
    free(w); free(h); free(y); free(rb);
    return rc;
}

int orc_block_step(const orc_layer *L, const orc_weights *W, const double *x, int h_bf16,
                   const uint16_t *input_ln, const uint16_t *post_ln,
                   uint16_t *cache_k, uint16_t *cache_v, int capacity,
                   const int32_t *cache_pos, int B, int R, double *out, double *out_normed)
{
    return block_step(L, W, x, h_bf16, input_ln, post_ln, cache_k, cache_v, capacity, cache_pos, B,
                      R, NULL, out, out_normed);
}

/* orc_block_step with the optional parts of orc_step_ext */
int orc_block_step_ext(const orc_layer *L, const orc_weights *W, const double *x, int h_bf16,
                       const uint16_t *input_ln, const uint16_t *post_ln,
                       uint16_t *cache_k, uint16_t *cache_v, int capacity,
                       const int32_t *cache_pos, int B, int R, const orc_step_ext *e,
                       double *out, double *out_normed)
{
    return block_step(L, W, x, h_bf16, input_ln, post_ln, cache_k, cache_v, capacity, cache_pos, B,
                      R, e, out, out_normed);
}
