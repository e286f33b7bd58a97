/*
 * Every entry point of the C oracle on small and ragged inputs, built with AddressSanitizer
 * and UndefinedBehaviorSanitizer by tests/test_sanitizers.py (test infrastructure: it links
 * the oracle and nothing else). Besides memory and UB errors it checks two invariants the
 * oracle's pins also cover: prefix pieces merged with the Non-Shared part give the whole
 * decode, and a selection's scores come out in order. Exit 0 = clean.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t R, BW, Hq, Hkv, d, Lmax, S, Tmax;
    double scale;
} oracle_dims;

int oracle_partial_rows(const oracle_dims* D, const float* q, const float* shared_k, const float* shared_v,
                        const int32_t* shared_len, const float* pool_k, const float* pool_v,
                        const int32_t* beam_tok_idx, int32_t p_lo, int32_t p_hi, int32_t t_lo, int32_t t_hi,
                        const int64_t* rows, int64_t nrows, double* out, double* lse, int32_t nthreads);
int oracle_decode_rows(const oracle_dims* D, const float* q, const float* shared_k, const float* shared_v,
                       const int32_t* shared_len, const float* pool_k, const float* pool_v,
                       const int32_t* beam_tok_idx, int32_t step, const int64_t* rows, int64_t nrows, double* out,
                       double* lse, int32_t nthreads);
int oracle_merge(int32_t nparts, int64_t nrows, int32_t d, const double* part_out, const double* part_lse,
                 double* out, double* lse);
int oracle_beam_update(const oracle_dims* D, const int32_t* parent, const float* new_k, const float* new_v,
                       float* pool_k, float* pool_v, int32_t* idx, int32_t step);
int oracle_beam_select(int32_t R, int32_t BW, int32_t K, int32_t W, const float* beam_score, const float* cand_logp,
                       const int32_t* cand_token, int32_t* parent, int32_t* token, float* score);

/* xorshift64 (Marsaglia, "Xorshift RNGs", 2003) */
static uint64_t rs = 88172645463325252ull;
static uint64_t nxt(void) {
    rs ^= rs << 13;
    rs ^= rs >> 7;
    rs ^= rs << 17;
    return rs;
}
static float unif(void) { return (float)((nxt() >> 11) * (1.0 / 9007199254740992.0)) * 2.f - 1.f; }
static float* farr(size_t n) {
    float* p = (float*)malloc(sizeof(float) * (n ? n : 1));
    for (size_t i = 0; i < n; ++i) p[i] = unif();
    return p;
}

static int fail(const char* what) {
    fprintf(stderr, "oracle_san: %s\n", what);
    return 1;
}

static int one_case(int R, int BW, int Hq, int Hkv, int d, int Lmax, int T) {
    const int Tm = T > 0 ? T : 1;
    oracle_dims D = {R, BW, Hq, Hkv, d, Lmax, BW * Tm, Tm, 0.35};
    const size_t rows = (size_t)R * BW * Hq, tok = (size_t)Hkv * d;
    float* q = farr(rows * d);
    float* sk = farr((size_t)R * Lmax * tok);
    float* sv = farr((size_t)R * Lmax * tok);
    int32_t* slen = (int32_t*)malloc(sizeof(int32_t) * R);
    for (int r = 0; r < R; ++r) slen[r] = Lmax ? (int32_t)(r == 0 ? Lmax : nxt() % (uint64_t)(Lmax + 1)) : 0;
    float* pk = farr((size_t)R * D.S * tok);
    float* pv = farr((size_t)R * D.S * tok);
    int32_t* idx = (int32_t*)calloc((size_t)R * BW * Tm, sizeof(int32_t));
    int32_t* par = (int32_t*)malloc(sizeof(int32_t) * R * BW);
    float* nk = farr((size_t)R * BW * tok);
    float* nv = farr((size_t)R * BW * tok);
    for (int s = 0; s < T; ++s) {
        for (int i = 0; i < R * BW; ++i) par[i] = (int32_t)(nxt() % (uint64_t)BW);
        if (oracle_beam_update(&D, par, nk, nv, pk, pv, idx, s) != 0) return fail("beam_update rejected a valid step");
    }
    if (oracle_beam_update(&D, par, nk, nv, pk, pv, idx, Tm) != -1) return fail("beam_update accepted step >= Tmax");
    double* out = (double*)malloc(sizeof(double) * rows * d);
    double* lse = (double*)malloc(sizeof(double) * rows);
    if (oracle_decode_rows(&D, q, sk, sv, slen, pk, pv, idx, T, NULL, 0, out, lse, 2) != 0) return fail("decode");
    /* pieces: prefix halves and the Non-Shared part, merged */
    const int half = Lmax / 2;
    double* po = (double*)malloc(sizeof(double) * 3 * rows * d);
    double* pl = (double*)malloc(sizeof(double) * 3 * rows);
    if (oracle_partial_rows(&D, q, sk, sv, slen, pk, pv, idx, 0, half, 0, 0, NULL, 0, po, pl, 1) != 0 ||
        oracle_partial_rows(&D, q, sk, sv, slen, pk, pv, idx, half, Lmax, 0, 0, NULL, 0, po + rows * d, pl + rows,
                            1) != 0 ||
        oracle_partial_rows(&D, q, sk, sv, slen, pk, pv, idx, 0, 0, 0, T, NULL, 0, po + 2 * rows * d, pl + 2 * rows,
                            1) != 0)
        return fail("partial");
    double* mo = (double*)malloc(sizeof(double) * rows * d);
    double* ml = (double*)malloc(sizeof(double) * rows);
    if (oracle_merge(3, (int64_t)rows, d, po, pl, mo, ml) != 0) return fail("merge");
    for (size_t i = 0; i < rows; ++i) {
        if (isinf(lse[i]) != isinf(ml[i]) || (!isinf(lse[i]) && fabs(lse[i] - ml[i]) > 1e-9))
            return fail("split-and-merge LSE differs from the whole decode");
        for (int e = 0; e < d; ++e)
            if (fabs(out[i * d + e] - mo[i * d + e]) > 1e-9) return fail("split-and-merge output differs");
    }
    int64_t sel[2] = {0, (int64_t)rows - 1};
    if (oracle_decode_rows(&D, q, sk, sv, slen, pk, pv, idx, T, sel, 2, out, lse, 1) != 0) return fail("rows");
    int64_t bad_row = (int64_t)rows;
    if (oracle_decode_rows(&D, q, sk, sv, slen, pk, pv, idx, T, &bad_row, 1, out, lse, 1) != -1)
        return fail("decode accepted a row out of range");
    if (oracle_partial_rows(&D, q, sk, sv, slen, pk, pv, idx, 0, Lmax, 0, Tm + 1, NULL, 0, po, pl, 1) != -1)
        return fail("partial accepted t_hi > Tmax");
    free(q); free(sk); free(sv); free(slen); free(pk); free(pv); free(idx); free(par); free(nk); free(nv);
    free(out); free(lse); free(po); free(pl); free(mo); free(ml);
    return 0;
}

static int select_case(int R, int BW, int K, int W) {
    float* bs = farr((size_t)R * BW);
    float* lp = (float*)malloc(sizeof(float) * R * BW * K);
    int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * R * BW * K);
    for (int i = 0; i < R * BW; ++i) {
        float v = 0.f;
        for (int k = 0; k < K; ++k) {
            v -= (float)(nxt() % 4) / 8.f; /* non-increasing, with equal neighbours */
            lp[(size_t)i * K + k] = v;
            tok[(size_t)i * K + k] = (int32_t)(nxt() % 1000);
        }
    }
    int32_t* par = (int32_t*)malloc(sizeof(int32_t) * R * W);
    int32_t* tk = (int32_t*)malloc(sizeof(int32_t) * R * W);
    float* sc = (float*)malloc(sizeof(float) * R * W);
    if (oracle_beam_select(R, BW, K, W, bs, lp, tok, par, tk, sc) != 0) return fail("beam_select");
    for (int r = 0; r < R; ++r)
        for (int j = 1; j < W; ++j)
            if (sc[(size_t)r * W + j] > sc[(size_t)r * W + j - 1]) return fail("selection out of order");
    if (oracle_beam_select(R, BW, K, BW * K + 1, bs, lp, tok, par, tk, sc) != -1) return fail("W > BW*K accepted");
    free(bs); free(lp); free(tok); free(par); free(tk); free(sc);
    return 0;
}

int main(void) {
    const int cases[][7] = {{2, 3, 4, 2, 8, 5, 3}, {1, 1, 2, 1, 4, 0, 2}, {2, 4, 4, 4, 16, 17, 1},
                            {3, 2, 6, 2, 8, 9, 0}, {1, 6, 8, 2, 32, 40, 5}};
    for (size_t c = 0; c < sizeof(cases) / sizeof(cases[0]); ++c) {
        const int* k = cases[c];
        if (one_case(k[0], k[1], k[2], k[3], k[4], k[5], k[6])) return 1;
    }
    if (select_case(2, 5, 7, 9) || select_case(1, 1, 1, 1) || select_case(3, 17, 4, 68)) return 1;
    printf("oracle_san: ok\n");
    return 0;
}
