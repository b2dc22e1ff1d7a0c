/*
 * Test helper (CPU): drives the oracle and the library's host code (the
 * packer and the Turbo4 codebook of hostpack.cpp) through every entry point
 * on small inputs, for a build under AddressSanitizer and
 * UndefinedBehaviorSanitizer (tests/test_sanitize_host.py).  Exit 0 and no
 * sanitizer report = pass.  It includes the oracle's source to reach its
 * types; nothing here computes a reference value of its own.
 */
#include "../oracle/gattn_oracle.c"

#include <stdio.h>

#include "gattn.h"

static uint64_t rng_state = 88172645463325252ull;
static double urand(void)           /* xorshift64*, in [-1, 1) */
{
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (double)((rng_state * 2685821657736338717ull) >> 11) / 4503599627370496.0 - 1.0;
}

#define CHECK(c)                                                                                   \
    do {                                                                                           \
        if (!(c)) {                                                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c);                       \
            return 1;                                                                              \
        }                                                                                          \
    } while (0)

static int packers(void)
{
    const int N = 64, K = 256;
    double *w = malloc(sizeof(double) * N * K);
    float *wf = malloc(sizeof(float) * N * K);
    for (int i = 0; i < N * K; ++i) {
        w[i] = (double)(float)(0.02 * urand());
        wf[i] = (float)w[i];
    }
    const int bits[] = {2, 3, 4, 5, 6, 8}, groups[] = {32, 64, 128};
    for (int bi = 0; bi < 6; ++bi)
        for (int gi = 0; gi < 3; ++gi) {
            const int b = bits[bi], g = groups[gi], words = K * b / 32;
            uint32_t *p1 = calloc((size_t)N * words, 4), *p2 = calloc((size_t)N * words, 4);
            uint16_t *s1 = calloc((size_t)N * (K / g), 2), *s2 = calloc((size_t)N * (K / g), 2);
            uint16_t *b1 = calloc((size_t)N * (K / g), 2), *b2 = calloc((size_t)N * (K / g), 2);
            CHECK(orc_quantize_affine(w, N, K, b, g, p1, s1, b1) == 0);
            CHECK(gattn_pack_affine_host(wf, N, K, b, g, p2, s2, b2) == GATTN_OK);
            CHECK(memcmp(p1, p2, (size_t)N * words * 4) == 0);
            CHECK(memcmp(s1, s2, (size_t)N * (K / g) * 2) == 0);
            uint8_t *codes = malloc((size_t)N * K);
            double *dq = malloc(sizeof(double) * N * K), *y = malloc(sizeof(double) * N * 2);
            CHECK(orc_unpack_codes(p1, N, K, b, codes) == 0);
            CHECK(orc_dequantize(p1, s1, b1, N, K, b, g, dq) == 0);
            CHECK(orc_qmatvec(p1, s1, b1, N, K, b, g, w, 2, y) == 0);
            free(p1); free(p2); free(s1); free(s2); free(b1); free(b2); free(codes); free(dq); free(y);
        }
    CHECK(gattn_pack_affine_host(wf, N, K, 7, 64, NULL, NULL, NULL) != GATTN_OK);
    free(w);
    free(wf);
    return 0;
}

static int turbo(void)
{
    float lv[16], th[15], olv[16], oth[15];
    CHECK(gattn_turbo4_codebook(lv, th) == GATTN_OK);
    orc_turbo4_tables_f32(olv, oth);
    CHECK(memcmp(lv, olv, sizeof lv) == 0 && memcmp(th, oth, sizeof th) == 0);
    CHECK(gattn_turbo4_codebook(NULL, th) != GATTN_OK);
    for (int b = 0; b < 256; ++b)
        (void)orc_e4m3_to_double((uint8_t)b);
    const float xs[] = {0.f, -0.f, 1e-9f, 448.f, 1e30f, -3.5f, 0.0017f};
    for (int i = 0; i < 7; ++i)
        (void)orc_e4m3_from_float(xs[i]);
    const int ds[] = {64, 128, 256};
    for (int di = 0; di < 3; ++di) {
        const int d = ds[di], n = 40;
        uint16_t *v = malloc(sizeof(uint16_t) * n * d);
        for (int i = 0; i < n * d; ++i)
            v[i] = orc_bf16_from_double(i % 97 == 0 ? 0.0 : 3.0 * urand());
        for (int j = 0; j < d; ++j)
            v[j] = 0;                           /* a zero row */
        uint8_t *c = malloc((size_t)n * d / 2), *s = malloc((size_t)n * d / 16);
        double *r = malloc(sizeof(double) * n * d);
        CHECK(orc_turbo4_quantize_rows(v, n, d, c, s) == 0);
        CHECK(orc_turbo4_dequant_rows(c, s, n, d, 0, r) == 0);
        free(v); free(c); free(s); free(r);
    }
    CHECK(orc_turbo4_quantize_rows(NULL, 1, 48, NULL, NULL) != 0);
    return 0;
}

/* one small layer: hidden 128, H query heads over Hk KV heads, d 64, 4-bit
 * g64, B = 2 sequences of R rows; R * H / Hk > 32 takes the head-chunked route */
static int layers(int H, int Hk, int R)
{
    enum { Hd = 128, d = 64, B = 2, cap = 64 };
    orc_layer L = {Hd, H, Hk, d, 0.25, 10000.0, 1e-6, {4, 4, 4, 4}, {64, 64, 64, 64}, 1, 0};
    const int64_t Ns[4] = {2 * H * d, Hk * d, Hk * d, Hd}, Ks[4] = {Hd, Hd, Hd, H * d};
    orc_weights W;
    void *keep[16];
    int nk = 0;
    for (int p = 0; p < 4; ++p) {
        double *w = malloc(sizeof(double) * Ns[p] * Ks[p]);
        for (int64_t i = 0; i < Ns[p] * Ks[p]; ++i)
            w[i] = 0.05 * urand();
        uint32_t *pk = calloc((size_t)(Ns[p] * Ks[p] * 4 / 32), 4);
        uint16_t *sc = calloc((size_t)(Ns[p] * Ks[p] / 64), 2), *bi = calloc((size_t)(Ns[p] * Ks[p] / 64), 2);
        CHECK(orc_quantize_affine(w, Ns[p], Ks[p], 4, 64, pk, sc, bi) == 0);
        free(w);
        W.packed[p] = pk;
        W.scales[p] = sc;
        W.biases[p] = bi;
        keep[nk++] = pk; keep[nk++] = sc; keep[nk++] = bi;
    }
    uint16_t qn[d], kn[d], iln[Hd], pln[Hd];
    for (int j = 0; j < d; ++j) {
        qn[j] = orc_bf16_from_double(1.0 + 0.1 * urand());
        kn[j] = orc_bf16_from_double(1.0 + 0.1 * urand());
    }
    for (int j = 0; j < Hd; ++j) {
        iln[j] = orc_bf16_from_double(1.0 + 0.1 * urand());
        pln[j] = orc_bf16_from_double(1.0 + 0.1 * urand());
    }
    W.q_norm = qn;
    W.k_norm = kn;
    const int M = B * R;
    double *x = malloc(sizeof(double) * M * Hd), *out = malloc(sizeof(double) * M * Hd);
    double *on = malloc(sizeof(double) * M * Hd);
    double *ty = malloc(sizeof(double) * M * (2 * H * d + 2 * Hk * d));
    double *ta = malloc(sizeof(double) * M * H * d);
    for (int i = 0; i < M * Hd; ++i)
        x[i] = (double)(float)urand();
    const size_t cache = (size_t)B * Hk * cap * d;
    uint16_t *ck = malloc(cache * 2), *cv = malloc(cache * 2);
    uint8_t *kc = malloc(cache / 2), *ks = malloc(cache / 16), *vc = malloc(cache / 2), *vs = malloc(cache / 16);
    for (size_t i = 0; i < cache; ++i) {
        ck[i] = orc_bf16_from_double(urand());
        cv[i] = orc_bf16_from_double(urand());
    }
    for (size_t i = 0; i < cache / 2; ++i) {
        kc[i] = (uint8_t)(urand() * 127 + 128);
        vc[i] = (uint8_t)(urand() * 127 + 128);
    }
    for (size_t i = 0; i < cache / 16; ++i) {
        ks[i] = (uint8_t)(0x30 + (i % 16));
        vs[i] = (uint8_t)(0x30 + (i % 13));
    }
    const int32_t pos[B] = {20, cap - R};       /* the second sequence fills the cache */
    const int32_t bad[B] = {20, cap - R + 1};   /* one row past the capacity: a range error */
    uint8_t *mask = malloc((size_t)B * H * R * cap);
    for (size_t i = 0; i < (size_t)B * H * R * cap; ++i)
        mask[i] = urand() > -0.2;
    CHECK(orc_layer_step(&L, &W, x, ck, cv, cap, pos, B, R, out, ty, ta) == 0);
    CHECK(orc_layer_step(&L, &W, x, ck, cv, cap, bad, B, R, out, NULL, NULL) == ORC_E_RANGE);
    CHECK(orc_layer_step_masked(&L, &W, x, ck, cv, cap, pos, B, R, mask, 1, cap, R * cap, R * cap,
                                out, ty, ta) == 0);
    CHECK(orc_layer_step_turbo4v(&L, &W, x, ck, vc, vs, cap, pos, B, R, out, ty, ta) == 0);
    orc_step_ext e = {vc, vs, kc, ks, mask, 1, cap, R * cap, R * cap, cap};
    CHECK(orc_layer_step_ext(&L, &W, x, NULL, NULL, cap, pos, B, R, &e, out, ty, ta) == 0);
    CHECK(orc_block_step_ext(&L, &W, x, 1, iln, pln, ck, cv, cap, pos, B, R, NULL, out, on) == 0);
    orc_step_ext ev = {vc, vs, NULL, NULL, NULL, 0, 0, 0, 0, 0};
    CHECK(orc_block_step_ext(&L, &W, x, 0, iln, NULL, ck, NULL, cap, pos, B, R, &ev, out, NULL) == 0);
    L.head_chunk = 0;
    orc_step_ext eh = {NULL, NULL, NULL, NULL, mask, H, cap, (int64_t)R * cap, (int64_t)H * R * cap, 0};
    CHECK(orc_layer_step_ext(&L, &W, x, ck, cv, cap, pos, B, R, &eh, out, ty, ta) == 0);
    /* mask rows of 5 positions, shorter than every sequence's span */
    orc_step_ext es = {vc, vs, NULL, NULL, mask, 1, 5, (int64_t)R * 5, (int64_t)R * 5, 5};
    CHECK(orc_layer_step_ext(&L, &W, x, ck, NULL, cap, pos, B, R, &es, out, ty, ta) == 0);
    CHECK(orc_layer_step(&L, &W, x, ck, cv, cap, pos, B, R, out, NULL, NULL) == 0);
    int32_t cf[64], cl[64];
    for (int q = 1; q <= 33; ++q) {
        const int n = orc_head_chunk_plan(q, H, Hk, 1, cf, cl, 64);
        CHECK(n >= Hk && n <= H);
    }
    free(x); free(out); free(on); free(ty); free(ta); free(ck); free(cv); free(mask);
    free(kc); free(ks); free(vc); free(vs);
    for (int i = 0; i < nk; ++i)
        free(keep[i]);
    return 0;
}

int main(void)
{
    if (packers() || turbo() || layers(4, 2, 3) || layers(8, 2, 17) || layers(4, 4, 32))
        return 1;
    printf("sanitized host run ok\n");
    return 0;
}
