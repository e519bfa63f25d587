/*
 * qsa_oracle.c -- plain FP64 CPU oracle (TEST INFRASTRUCTURE ONLY; see
 * qsa_oracle.h).  Written for clarity, not speed: every query head walks its own
 * selection list, dequantises each selected cell from the paged INT8 pool in
 * FP64, and applies a textbook max-subtracted softmax.
 *
 * Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
 * PR #2808).  Section Summary defines the result (each position attends to
 * exactly the cells it selected; a cell is excluded, -inf, for positions that
 * did not select it) and the 8-position union with per-cell membership; section
 * Extra Notes fixes the union's storage (int32 cell, separate mask byte) and says
 * non-resident pages are masked.  Readings where the page is silent: scores are
 * scaled by 1/sqrt(d) (passed in as sm_scale), query head h uses KV head h/12,
 * K/V values are int8 times a per-cell per-KV-head FP16 scale, and a query with
 * no resident selected cell outputs zeros.
 */
#include "qsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { D = 128, HPK = 12, PAGE = 64, GROUP = 8 };

double qsa_ref_half_to_double(uint16_t h) {
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

double qsa_ref_bf16_to_double(uint16_t b) {
    /* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
    int sign = (b >> 15) & 1, e = (b >> 7) & 0xff, f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 128), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

int qsa_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Is `cell` in the sorted list lst[0:n]?  Plain binary search. */
static int list_has(const int32_t* lst, int32_t n, int32_t cell) {
    int32_t lo = 0, hi = n;
    while (lo < hi) {
        int32_t mid = lo + (hi - lo) / 2;
        if (lst[mid] < cell) lo = mid + 1;
        else hi = mid;
    }
    return lo < n && lst[lo] == cell;
}

int qsa_ref_union(const int32_t* sel, const int32_t* sel_count, int32_t n_q, int32_t sel_stride,
                  int32_t* ucell, uint8_t* umask, int32_t* ucount, int32_t ustride) {
    if (n_q < 0 || sel_stride <= 0 || ustride <= 0) return 1;
    if (n_q == 0) return 0;
    if (!sel || !sel_count || !ucell || !umask || !ucount) return 1;
    int32_t n_groups = (n_q + GROUP - 1) / GROUP;
    int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)GROUP * (size_t)sel_stride);
    if (!all) return 1;
    int rc = 0;
    for (int32_t g = 0; g < n_groups && rc == 0; ++g) {
        int32_t q_begin = g * GROUP;
        int32_t nj = n_q - q_begin < GROUP ? n_q - q_begin : GROUP;
        /* 1. gather every selected cell of the group's queries */
        size_t n_all = 0;
        for (int32_t j = 0; j < nj; ++j) {
            int32_t c = sel_count[q_begin + j];
            if (c < 0 || c > sel_stride) { rc = 1; break; }
            memcpy(all + n_all, sel + (size_t)(q_begin + j) * sel_stride, sizeof(int32_t) * (size_t)c);
            n_all += (size_t)c;
        }
        if (rc) break;
        /* 2. sort and drop repeats: the set union */
        qsort(all, n_all, sizeof(int32_t), cmp_i32);
        size_t n_u = 0;
        for (size_t t = 0; t < n_all; ++t)
            if (n_u == 0 || all[t] != all[n_u - 1]) all[n_u++] = all[t];
        if (n_u > (size_t)ustride) { rc = 3; break; }
        /* 3. membership byte: bit j set iff query q_begin+j selected the cell */
        for (size_t t = 0; t < n_u; ++t) {
            uint8_t m = 0;
            for (int32_t j = 0; j < nj; ++j)
                if (list_has(sel + (size_t)(q_begin + j) * sel_stride, sel_count[q_begin + j], all[t]))
                    m |= (uint8_t)(1u << j);
            ucell[(size_t)g * ustride + t] = all[t];
            umask[(size_t)g * ustride + t] = m;
        }
        ucount[g] = (int32_t)n_u;
    }
    free(all);
    return rc;
}

int qsa_attn_ref(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                 const uint16_t* k_scale, const uint16_t* v_scale,
                 const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                 const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                 const int32_t* q_index, int32_t n_index, double sm_scale,
                 double* out, int32_t n_threads) {
    if (n_q < 0 || n_kv <= 0 || n_lpages < 0 || n_ppages < 0 || sel_stride <= 0) return 1;
    int32_t n_rows = q_index ? n_index : n_q;
    if (n_rows <= 0) return n_rows < 0 ? 1 : 0;
    if (!q || !k_pool || !v_pool || !k_scale || !v_scale || !page_table || !sel || !sel_count || !out)
        return 1;
    for (int32_t t = 0; t < n_rows; ++t) {
        int32_t i = q_index ? q_index[t] : t;
        if (i < 0 || i >= n_q || sel_count[i] < 0 || sel_count[i] > sel_stride) return 1;
    }
    const int32_t n_heads = n_kv * HPK;
    const long long n_work = (long long)n_rows * n_heads;
    int bad = 0;
#ifdef _OPENMP
    int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt) reduction(| : bad)
#endif
    {
        double* score = (double*)malloc(sizeof(double) * (size_t)sel_stride);
        int32_t* row = (int32_t*)malloc(sizeof(int32_t) * (size_t)sel_stride);
        double qv[D], kc[D], acc[D];
        if (!score || !row) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
        for (long long w = 0; w < n_work; ++w) {
            if (!score || !row) continue;
            int32_t t = (int32_t)(w / n_heads), h = (int32_t)(w % n_heads);
            int32_t i = q_index ? q_index[t] : t;
            int32_t kh = h / HPK;
            const uint16_t* qrow = q + ((size_t)i * n_heads + h) * D;
            for (int d = 0; d < D; ++d) qv[d] = qsa_ref_bf16_to_double(qrow[d]);
            const int32_t* lst = sel + (size_t)i * sel_stride;
            int32_t n_sel = 0;
            double m = -INFINITY;
            /* scores of the query's own resident cells */
            for (int32_t s = 0; s < sel_count[i]; ++s) {
                int32_t c = lst[s];
                if (c < 0 || c / PAGE >= n_lpages) { bad = 1; continue; }
                int32_t pp = page_table[c / PAGE];
                if (pp < 0) continue;                      /* not resident: masked */
                if (pp >= n_ppages) { bad = 1; continue; }
                size_t r = ((size_t)pp * n_kv + kh) * PAGE + (size_t)(c % PAGE);
                double ks = qsa_ref_half_to_double(k_scale[r]);
                for (int d = 0; d < D; ++d) kc[d] = (double)k_pool[r * D + d] * ks;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qv[d] * kc[d];
                score[n_sel] = dot * sm_scale;
                row[n_sel] = (int32_t)r;
                if (score[n_sel] > m) m = score[n_sel];
                ++n_sel;
            }
            double* o = out + ((size_t)t * n_heads + h) * D;
            if (n_sel == 0) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                continue;
            }
            /* softmax weights (max subtracted) applied to the dequantised values */
            double z = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int32_t s = 0; s < n_sel; ++s) {
                double p = exp(score[s] - m);
                size_t r = (size_t)row[s];
                double vs = qsa_ref_half_to_double(v_scale[r]);
                z += p;
                for (int d = 0; d < D; ++d) acc[d] += p * ((double)v_pool[r * D + d] * vs);
            }
            for (int d = 0; d < D; ++d) o[d] = acc[d] / z;
        }
        free(score);
        free(row);
    }
    return bad ? 1 : 0;
}
