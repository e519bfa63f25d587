/*
 * qsa_oracle.h -- plain FP64 CPU oracle for selected-cell (QSA union) prompt
 * attention.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg are its only users.  It shares no code, header,
 * table or helper with the CUDA path (libqsa.so), and the CUDA path never calls it.
 *
 * What it computes follows "sycl: prompt attention over 8-query selection unions
 * on XMX" (Strata PR #2808), section Summary: each prompt position attends to
 * exactly its own selected cells (the union path must reach the same result as
 * the per-position FP32 kernel), and for every 8 neighbouring positions the
 * union of their selections is sorted and each cell marked with the positions
 * that chose it (section Extra Notes: int32 cell + a separate membership byte).
 *
 * Layouts (row-major, all host memory owned by the caller):
 *   q          uint16 [n_q][n_kv*12][128]      BF16 bit patterns
 *   k_pool     int8   [n_ppages][n_kv][64][128]
 *   v_pool     int8   [n_ppages][n_kv][64][128]
 *   k_scale    uint16 [n_ppages][n_kv][64]       FP16 bit patterns
 *   v_scale    uint16 [n_ppages][n_kv][64]       FP16 bit patterns
 *   page_table int32  [n_lpages]                 physical page, < 0 = not resident
 *   sel        int32  [n_q][sel_stride]          sorted cell ids
 *   sel_count  int32  [n_q]
 * Return value: 0 on success, 1 on a bad argument, 3 when a union does not fit.
 */
#ifndef QSA_ORACLE_H
#define QSA_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* FP16 / BF16 bit pattern -> double, decoded from the IEEE-754 field layout. */
double qsa_ref_half_to_double(uint16_t h);
double qsa_ref_bf16_to_double(uint16_t b);

/* Per group g of 8 consecutive queries (8g .. min(8g+8, n_q)-1): the sorted set
 * union of their lists into ucell[g][0:ucount[g]] and, for each union cell, a
 * byte whose bit j says that query 8g+j selected it. */
int qsa_ref_union(const int32_t* sel, const int32_t* sel_count, int32_t n_q, int32_t sel_stride,
                  int32_t* ucell, uint8_t* umask, int32_t* ucount, int32_t ustride);

/* out[t][h][:] (FP64) = softmax over the resident cells c of query i's own list
 * of (q_i,h . k_c) * sm_scale, applied to v_c, with k_c = int8 K * FP16 scale of
 * KV head h/12 (likewise v_c); 0 when no resident cell is selected.
 * i = q_index[t] for t < n_index, or t itself for t < n_q when q_index is NULL.
 * n_threads <= 0 uses every OpenMP thread. */
int qsa_attn_ref(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                 const uint16_t* k_scale, const uint16_t* v_scale,
                 const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                 const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                 const int32_t* q_index, int32_t n_index, double sm_scale,
                 double* out, int32_t n_threads);

/* Number of OpenMP threads a call with n_threads <= 0 would use. */
int qsa_ref_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
