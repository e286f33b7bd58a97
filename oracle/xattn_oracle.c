/*
 * Plain fp64 CPU oracle for split Shared / Non-Shared beam-search decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU-baseline
 * leg load this library. The CUDA path shares no code, header or table with it.
 *
 * What it computes (xGR: Efficient Generative Recommendation Serving at Scale, section 2.1
 * "xAttention": the KV cache is split into a Shared part holding the user-history prompt,
 * stored once per request, and a Non-Shared part holding the tokens each beam generated,
 * managed per token; the staged Shared / Non-Shared / Merge computation combines local
 * scores and max/sum statistics with an online softmax). Staging and merging reach,
 * up to rounding, plain softmax attention over the concatenated key list, so this file
 * writes out that plain definition and nothing else:
 *
 *   for request r, beam b, query head h (KV head h_kv = h / G, G = Hq / Hkv):
 *     keys   J = shared_k[r, 0 .. shared_len[r]-1, h_kv]
 *                ++ pool_k[r, beam_tok_idx[r, b, i], h_kv]   for i < step
 *     (values gathered the same way)
 *     s_j    = scale * <q[r,b,h], k_j>                         (fp64)
 *     lse    = m + ln(sum_j exp(s_j - m)),  m = max_j s_j
 *     out    = sum_j exp(s_j - lse) * v_j
 *
 * Inputs are float32 arrays holding the exact input values (bf16 values are exact in
 * float32); every operation after loading is in double precision.
 *
 * Partial results (one stage, or one piece of the prefix) use the same definition over a
 * subset of the keys; an empty subset gives lse = -inf and out = 0. The merge of partials
 * is the log-sum-exp combine read from the "OnlineSoftmax" merging stage of that section:
 *   lse = ln(sum_i exp(lse_i)),  out = sum_i exp(lse_i - lse) * out_i.
 *
 * The beam update is the per-token Non-Shared management of the same section: the token a
 * beam emits at step s goes to the fresh pool slot s*BW + b (nothing is copied when beams
 * fork), and the beam's ancestry row becomes its parent's row followed by that slot:
 *   idx'[b, 0:s] = idx[parent[b], 0:s],   idx'[b, s] = s*BW + b,
 * computed from a snapshot of the old table (the pages' in-place update avoids
 * read-before-write hazards; only the resulting table and pool are fixed here).
 *
 * Compile-time ORACLE_MUTANT=n plants one deliberate mistake; the tests build those
 * variants to show that the pins catch each of them. Default 0 = the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
    int32_t R, BW, Hq, Hkv, d, Lmax, S, Tmax;
    double scale;
} oracle_dims;

static int dims_ok(const oracle_dims* D) {
    if (!D || D->R < 0 || D->BW <= 0 || D->Hq <= 0 || D->Hkv <= 0 || D->d <= 0) return 0;
    if (D->Hq % D->Hkv != 0 || D->Lmax < 0 || D->S < 0 || D->Tmax < 0) return 0;
    return 1;
}

static inline int kv_head_of(const oracle_dims* D, int h) {
#if ORACLE_MUTANT == 2
    return h % D->Hkv; /* planted: interleaved instead of consecutive grouping */
#else
    return h / (D->Hq / D->Hkv);
#endif
}

/* Attention of one query row over an explicit key list (pointers to float rows).
 * Writes out[0..d-1] and *lse. n == 0 gives out = 0, lse = -inf. */
static void attend(int d, double scale, const float* qrow, int n, const float* const* krows,
                   const float* const* vrows, double* scores, double* out, double* lse) {
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (n == 0) { *lse = -INFINITY; return; }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += (double)qrow[e] * (double)krows[j][e];
#if ORACLE_MUTANT == 3
        scores[j] = acc; /* planted: scale dropped */
        (void)scale;
#else
        scores[j] = scale * acc;
#endif
        if (scores[j] > m) m = scores[j];
    }
    double sum = 0.0;
    for (int j = 0; j < n; ++j) sum += exp(scores[j] - m);
#if ORACLE_MUTANT == 5
    double L = log(sum); /* planted: max term dropped from the log-sum-exp */
#else
    double L = m + log(sum);
#endif
    for (int j = 0; j < n; ++j) {
        double p = exp(scores[j] - L);
#if ORACLE_MUTANT == 5
        p = exp(scores[j] - m) / sum;
#endif
        for (int e = 0; e < d; ++e) out[e] += p * (double)vrows[j][e];
    }
    *lse = L;
}

/* Key list of row (r, b, h): prefix tokens [p_lo, p_hi) (clipped to shared_len[r]) then
 * Non-Shared positions [t_lo, t_hi) of the beam's ancestry row. Returns the count, or -1
 * when an index is out of range. */
static int gather_keys(const oracle_dims* D, int r, int b, int h, const float* shared_k,
                       const float* shared_v, const int32_t* shared_len, const float* pool_k,
                       const float* pool_v, const int32_t* idx, int p_lo, int p_hi, int t_lo,
                       int t_hi, const float** krows, const float** vrows) {
    const int d = D->d, Hkv = D->Hkv;
    const int hk = kv_head_of(D, h);
    int L = shared_len[r];
#if ORACLE_MUTANT == 6
    L = L - 1; /* planted: last prefix token dropped */
#endif
    if (L < 0 || L > D->Lmax) return -1;
    int lo = p_lo < 0 ? 0 : p_lo, hi = p_hi < L ? p_hi : L;
    int n = 0;
    for (int j = lo; j < hi; ++j) {
        size_t off = (((size_t)r * D->Lmax + j) * Hkv + hk) * (size_t)d;
        krows[n] = shared_k + off;
        vrows[n] = shared_v + off;
        ++n;
    }
#if ORACLE_MUTANT == 1
    t_hi = t_lo; /* planted: Non-Shared part dropped */
#endif
    for (int i = t_lo; i < t_hi; ++i) {
#if ORACLE_MUTANT == 4
        int slot = idx[((size_t)r * D->Tmax + i) * D->BW + b]; /* planted: table read as [R, T, BW] */
#else
        int slot = idx[((size_t)r * D->BW + b) * D->Tmax + i];
#endif
        if (slot < 0 || slot >= D->S) return -1;
        size_t off = (((size_t)r * D->S + slot) * Hkv + hk) * (size_t)d;
        krows[n] = pool_k + off;
        vrows[n] = pool_v + off;
        ++n;
    }
    return n;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Attention restricted to prefix tokens [p_lo, p_hi) and Non-Shared positions [t_lo, t_hi),
 * for the listed flat rows ((r*BW + b)*Hq + h), or all rows when rows == NULL.
 * out: [nrows, d] fp64, lse: [nrows] fp64. Returns 0, or -1 on bad arguments / indices. */
int oracle_partial_rows(const oracle_dims* D, const float* q, const float* shared_k,
                        const float* shared_v, const int32_t* shared_len, const float* pool_k,
                        const float* pool_v, const int32_t* beam_tok_idx, int32_t p_lo,
                        int32_t p_hi, int32_t t_lo, int32_t t_hi, const int64_t* rows,
                        int64_t nrows, double* out, double* lse, int32_t nthreads) {
    if (!dims_ok(D) || t_lo < 0 || t_hi > D->Tmax || t_lo > t_hi) return -1;
    const int64_t total = (int64_t)D->R * D->BW * D->Hq;
    if (!rows) nrows = total;
    const int maxkeys = D->Lmax + D->Tmax + 1;
    int err = 0;
    int nt = set_threads(nthreads);
#pragma omp parallel num_threads(nt) reduction(| : err)
    {
        const float** kr = (const float**)malloc(sizeof(float*) * (size_t)maxkeys);
        const float** vr = (const float**)malloc(sizeof(float*) * (size_t)maxkeys);
        double* sc = (double*)malloc(sizeof(double) * (size_t)maxkeys);
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t row = rows ? rows[i] : i;
            if (row < 0 || row >= total) { err |= 1; continue; }
            int h = (int)(row % D->Hq);
            int b = (int)((row / D->Hq) % D->BW);
            int r = (int)(row / ((int64_t)D->Hq * D->BW));
            int n = gather_keys(D, r, b, h, shared_k, shared_v, shared_len, pool_k, pool_v,
                                beam_tok_idx, p_lo, p_hi, t_lo, t_hi, kr, vr);
            if (n < 0) { err |= 1; continue; }
            const float* qrow = q + (size_t)row * D->d;
            attend(D->d, D->scale, qrow, n, kr, vr, sc, out + (size_t)i * D->d, lse + i);
        }
        free(kr); free(vr); free(sc);
    }
    return err ? -1 : 0;
}

/* The full decode attention of every listed row: the whole valid prefix plus the first
 * `step` tokens of the beam's ancestry row. */
int oracle_decode_rows(const oracle_dims* D, const float* q, const float* shared_k,
                       const float* shared_v, const int32_t* shared_len, const float* pool_k,
                       const float* pool_v, const int32_t* beam_tok_idx, int32_t step,
                       const int64_t* rows, int64_t nrows, double* out, double* lse,
                       int32_t nthreads) {
    return oracle_partial_rows(D, q, shared_k, shared_v, shared_len, pool_k, pool_v,
                               beam_tok_idx, 0, D->Lmax, 0, step, rows, nrows, out, lse, nthreads);
}

/* Log-sum-exp combine of nparts partials over nrows rows of width d.
 * part_out [nparts, nrows, d], part_lse [nparts, nrows]; lse_i = -inf means empty. */
int oracle_merge(int32_t nparts, int64_t nrows, int32_t d, const double* part_out,
                 const double* part_lse, double* out, double* lse) {
    if (nparts < 0 || nrows < 0 || d <= 0) return -1;
    for (int64_t i = 0; i < nrows; ++i) {
        double m = -INFINITY;
        for (int p = 0; p < nparts; ++p) {
            double l = part_lse[(size_t)p * nrows + i];
            if (l > m) m = l;
        }
        for (int e = 0; e < d; ++e) out[(size_t)i * d + e] = 0.0;
        if (m == -INFINITY) { lse[i] = -INFINITY; continue; }
        double sum = 0.0;
        for (int p = 0; p < nparts; ++p) sum += exp(part_lse[(size_t)p * nrows + i] - m);
        double L = m + log(sum);
        for (int p = 0; p < nparts; ++p) {
            double l = part_lse[(size_t)p * nrows + i];
#if ORACLE_MUTANT == 9
            double wgt = exp(l - m); /* planted: weights not normalised by the merged sum */
#else
            double wgt = exp(l - L);
#endif
            const double* o = part_out + ((size_t)p * nrows + i) * d;
            for (int e = 0; e < d; ++e) out[(size_t)i * d + e] += wgt * o[e];
        }
        lse[i] = L;
    }
    return 0;
}

/* One beam-search step of the Non-Shared bookkeeping, in place.
 * parent [R, BW] (ignored at step 0), new_k/new_v [R, BW, Hkv, d],
 * pool_k/pool_v [R, S, Hkv, d], idx [R, BW, Tmax]. Needs (step+1)*BW <= S and step < Tmax.
 * Returns 0, or -1 on bad arguments (nothing written then). */
int oracle_beam_update(const oracle_dims* D, const int32_t* parent, const float* new_k,
                       const float* new_v, float* pool_k, float* pool_v, int32_t* idx,
                       int32_t step) {
    if (!dims_ok(D) || step < 0 || step >= D->Tmax || (int64_t)(step + 1) * D->BW > D->S) return -1;
    const int BW = D->BW, T = D->Tmax;
    const size_t tok = (size_t)D->Hkv * D->d;
    if (step > 0)
        for (int r = 0; r < D->R; ++r)
            for (int b = 0; b < BW; ++b)
                if (parent[(size_t)r * BW + b] < 0 || parent[(size_t)r * BW + b] >= BW) return -1;
    int32_t* old = (int32_t*)malloc(sizeof(int32_t) * (size_t)BW * (size_t)(T > 0 ? T : 1));
    for (int r = 0; r < D->R; ++r) {
        int32_t* tab = idx + (size_t)r * BW * T;
        memcpy(old, tab, sizeof(int32_t) * (size_t)BW * T);
        for (int b = 0; b < BW; ++b) {
            int p = step > 0 ? parent[(size_t)r * BW + b] : b;
#if ORACLE_MUTANT == 8
            p = b; /* planted: ancestry not inherited from the parent */
#endif
            for (int i = 0; i < step; ++i) tab[(size_t)b * T + i] = old[(size_t)p * T + i];
#if ORACLE_MUTANT == 7
            int slot = step * BW + p; /* planted: token stored under the parent's slot */
#else
            int slot = step * BW + b;
#endif
            tab[(size_t)b * T + step] = slot;
            size_t dst = ((size_t)r * D->S + (size_t)(step * BW + b)) * tok;
            size_t src = ((size_t)r * BW + b) * tok;
            memcpy(pool_k + dst, new_k + src, sizeof(float) * tok);
            memcpy(pool_v + dst, new_v + src, sizeof(float) * tok);
        }
    }
    free(old);
    return 0;
}

/* Beam selection of one beam-search step (xGR: Efficient Generative Recommendation Serving at
 * Scale, section 2.2, xBeam "early sort termination": the Top-K sequences are chosen from the
 * pool of every beam's candidates; the pages prune that choice with a global min-heap because
 * the log-probabilities within a beam are already in order). The pruning only saves work;
 * the chosen set has a plain definition, which is what this function writes out:
 *   candidate (b, k) of request r, b < BW, k < K, scores
 *     s = beam_score[r, b] + cand_logp[r, b, k]        (one float32 addition)
 *   and the W candidates with the largest s are chosen, best first, equal scores ordered by
 *   the smaller flat index b*K + k (reading: the pages fix no tie rule).
 * Full sort of all BW*K candidates (qsort). Outputs [R, W]: parent = b, token =
 * cand_token[r, b, k], score = s. Returns 0, or -1 on bad sizes or a NaN score. */
typedef struct {
    float s;
    int32_t flat;
} sel_cand;

static int sel_cmp(const void* pa, const void* pb) {
    const sel_cand* a = (const sel_cand*)pa;
    const sel_cand* b = (const sel_cand*)pb;
    if (a->s != b->s) return a->s > b->s ? -1 : 1;
#if ORACLE_MUTANT == 10
    return a->flat > b->flat ? -1 : (a->flat < b->flat); /* planted: ties to the larger index */
#else
    return a->flat < b->flat ? -1 : (a->flat > b->flat);
#endif
}

int oracle_beam_select(int32_t R, int32_t BW, int32_t K, int32_t W, const float* beam_score,
                       const float* cand_logp, const int32_t* cand_token, int32_t* parent,
                       int32_t* token, float* score) {
    if (R < 1 || BW < 1 || K < 1 || W < 1 || (int64_t)BW * K > (1 << 30) || W > BW * K) return -1;
    const int n = BW * K;
    sel_cand* c = (sel_cand*)malloc(sizeof(sel_cand) * (size_t)n);
    if (!c) return -1;
    for (int r = 0; r < R; ++r) {
        for (int b = 0; b < BW; ++b)
            for (int k = 0; k < K; ++k) {
                const float lp = cand_logp[((size_t)r * BW + b) * K + k];
#if ORACLE_MUTANT == 11
                const float s = lp; /* planted: the beam's own score not added */
#else
                const float s = beam_score[(size_t)r * BW + b] + lp;
#endif
                if (s != s) {
                    free(c);
                    return -1;
                }
                c[b * K + k].s = s;
                c[b * K + k].flat = b * K + k;
            }
        qsort(c, (size_t)n, sizeof(sel_cand), sel_cmp);
        for (int j = 0; j < W; ++j) {
            const int b = c[j].flat / K, k = c[j].flat % K;
            parent[(size_t)r * W + j] = b;
            token[(size_t)r * W + j] = cand_token[((size_t)r * BW + b) * K + k];
            score[(size_t)r * W + j] = c[j].s;
        }
    }
    free(c);
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
