/*
 * qsa.h -- C ABI of libqsa.so: selected-cell (QSA union) prompt attention over a
 * paged INT8 KV cache, on GB300 (sm_103a).
 *
 * Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
 * PR #2808).  Section Summary: every prompt position attends only to its own
 * sorted selection of at most 2,051 K/V cells; for every 8 neighbouring
 * positions a first kernel builds the sorted union of their selections with each
 * cell marked by the positions that chose it, and a second kernel dequantises the
 * INT8 K/V of 64-cell chunks of that union once and runs S = Q K^T and O += P V
 * for all 96 rows (8 positions x 12 heads) with FP32 sums, setting a cell to
 * -inf for the positions that did not select it.  Section Extra Notes: a union
 * cell is an int32 with its 8-position mask in a separate byte; non-resident
 * pages are masked.  Section "What changed": the entry point carries the prompt
 * attention contract (query, paged K/V and scales, page table, per-position
 * selection lists and counts).
 *
 * Conventions shared by every entry point below
 *   - Device pointers point to CUDA global memory of the current device; host
 *     pointers are marked "host".  The caller owns all memory; the library
 *     allocates nothing, keeps no state between calls and never synchronises.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it; the call returns before it runs.
 *   - Shapes are fixed by the method: head dim d = 128, 12 query heads per KV
 *     head, 64-cell pages, groups of 8 consecutive queries starting at query 0
 *     (the last group may be ragged).
 *   - Layouts (row-major, no padding unless a stride is given):
 *       q          bf16  [n_q][n_kv*12][128]
 *       k_pool     int8  [n_ppages][n_kv][64][128]      (one KV head's page = 8 KB)
 *       v_pool     int8  [n_ppages][n_kv][64][128]
 *       k_scale    fp16  [n_ppages][n_kv][64]           per-cell per-KV-head scale
 *       v_scale    fp16  [n_ppages][n_kv][64]
 *       page_table int32 [n_lpages]   physical page of logical page c>>6; < 0 = not resident
 *       sel        int32 [n_q][sel_stride]   strictly increasing cell ids >= 0
 *       sel_count  int32 [n_q]               0 <= count <= sel_stride
 *       union_cells int32 [n_groups][union_stride], union_mask uint8 [..], union_count int32 [n_groups]
 *       out        fp32  [n_q][n_kv*12][128]
 *     with n_groups = ceil(n_q / 8).  K/V value of cell c for KV head h is
 *     int8 * scale at [page_table[c>>6]][h][c&63]; query head i uses KV head i/12.
 *   - bf16 / fp16 tensors are passed as uint16_t bit patterns.
 *   - Pointers to q, k_pool, v_pool and out must be 16-byte aligned.
 *   - Errors: a non-zero qsa_status is returned before anything is enqueued when
 *     an argument is invalid; QSA_ERR_CUDA reports a launch failure.  Problems that
 *     only the device can see (a bad count, cell or page-table entry, a union that
 *     does not fit, a device wait that ran out) never cause an out-of-bounds
 *     access: the offending cell is masked or the count clamped, and the matching
 *     QSA_DEV_* bit is OR-ed into *dev_status when dev_status is not NULL.
 */
#ifndef QSA_H
#define QSA_H
#include <stddef.h>
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_ARG = 1,          /* null pointer, negative size, bad alignment or stride */
    QSA_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels are built for */
    QSA_ERR_CAPACITY = 3,     /* workspace too small */
    QSA_ERR_CUDA = 4,         /* a CUDA launch or device query failed */
    QSA_ERR_DEVICE_CHECK = 5  /* reserved for callers decoding *dev_status */
} qsa_status;

/* Bits OR-ed into the optional device status word (int32 in device memory). */
enum {
    QSA_DEV_BAD_SEL_COUNT = 1,     /* a selection count outside [0, sel_stride] (clamped) */
    QSA_DEV_UNION_OVERFLOW = 2,    /* a union longer than union_stride (truncated) */
    QSA_DEV_BAD_CELL = 4,          /* a cell < 0 or on a page >= n_lpages (masked) */
    QSA_DEV_BAD_PAGE = 8,          /* a page-table entry >= n_ppages (masked) */
    QSA_DEV_BAD_UNION_COUNT = 16,  /* a union count outside [0, union_stride] (clamped) */
    QSA_DEV_WAIT_TIMEOUT = 32      /* a pipelined kernel gave up waiting; its output is invalid */
};

/* Attention kernel variants (all sm_103a).  QSA_ATTN_DEFAULT picks the fastest. */
enum {
    QSA_ATTN_DEFAULT = 0,
    QSA_ATTN_TCGEN05 = 1,   /* tcgen05.mma with TMEM accumulators, warp-specialised pipeline,
                               one CTA per (group, KV head), 64-cell chunks, two CTAs per SM */
    QSA_ATTN_TCGEN05_SM = 2 /* tcgen05, one CTA per (group, KV head) and per SM: Q, an O per
                               softmax set and three S/P buffers in TMEM, two softmax warp sets
                               on alternating chunks, combined at the end (the kernel
                               qsa_fused_attn runs with the union built in-CTA) */
};

/* The variant QSA_ATTN_DEFAULT resolves to in this build (one of the values above). */
int qsa_attn_default_variant(void);

/* Human-readable name of a qsa_status value.  Never NULL. */
const char* qsa_status_str(int status);

/* Bytes of one workspace holding the union arrays for n_q queries:
 * union_cells, then union_mask, then union_count, each 256-byte aligned.
 * Returns 0 for n_q < 0 or union_stride <= 0. */
size_t qsa_union_workspace_bytes(int32_t n_q, int32_t union_stride);

/* Union build (first kernel).  Defined by "sycl: prompt attention over 8-query
 * selection unions on XMX" (Strata PR #2808), section Summary (the sorted union of
 * 8 neighbouring positions' selections, each cell marked by the positions that
 * chose it) and section Extra Notes (a union cell is an int32 with its 8-position
 * mask in a separate byte).  For each group g of up to 8 consecutive queries:
 * union_cells[g][0:union_count[g]] = the sorted set union of their selection lists,
 * union_mask[g][u] bit j = query 8g+j selected union_cells[g][u] (bits of absent
 * ragged queries are 0).  Entries past union_count[g] are left unspecified.
 * Bit-exact and deterministic (no order-dependent atomics).
 * Requires union_stride % 64 == 0 and sel_stride >= 1; union_stride >= 8*sel_stride
 * guarantees that every union fits.  n_q == 0 returns QSA_OK with no launch. */
int qsa_union_build(const int32_t* sel, const int32_t* sel_count, int32_t n_q, int32_t sel_stride,
                    int32_t* union_cells, uint8_t* union_mask, int32_t* union_count,
                    int32_t union_stride, int32_t* dev_status, void* stream);

/* Union attention (second kernel).  Defined by "sycl: prompt attention over
 * 8-query selection unions on XMX" (Strata PR #2808), section Summary: for
 * query i (group g = i/8, j = i%8) and query head hq, out[i][hq][:] = sum over
 * union cells c with bit j of the mask set and a resident page of
 * softmax(q . k_c * sm_scale) * v_c, with k_c, v_c the dequantised K/V of KV
 * head hq/12; zeros when no such cell exists (our reading for the empty case).
 * One CTA per (group, KV head) covers 96 rows; K/V chunks of 64 union cells are
 * gathered through the page table and dequantised once.  Both variants compute
 * S = Q K^T on FP16 operands (Q converted from BF16, exact, with an exact
 * power-of-two row scale for rows outside FP16's comfortable range; K as the
 * exact INT8 integers, its scale applied to the score column in FP32) and
 * O += P V with FP32 accumulation (QSA_ATTN_TCGEN05: P = p * v_scale rounded to
 * BF16 against exact BF16 V; QSA_ATTN_TCGEN05_SM: P rounded to FP16 against exact
 * FP16 V, the V scale carried by a per-chunk power of two).  Typically
 * sm_scale = 1/sqrt(128).  `variant` is one of the QSA_ATTN_* values.
 * n_q == 0 returns QSA_OK. */
int qsa_union_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                   const uint16_t* k_scale, const uint16_t* v_scale,
                   const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                   const int32_t* union_cells, const uint8_t* union_mask, const int32_t* union_count,
                   int32_t union_stride, int32_t n_q, float sm_scale, float* out,
                   int32_t variant, int32_t* dev_status, void* stream);

/* Whole prompt-attention step: qsa_union_build into `workspace` (device memory
 * of at least qsa_union_workspace_bytes(n_q, union_stride) bytes, 256-byte
 * aligned, owned by the caller) followed by qsa_union_attn, both on `stream`.
 * Returns QSA_ERR_CAPACITY when workspace_bytes is too small. */
int qsa_prompt_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                    const uint16_t* k_scale, const uint16_t* v_scale,
                    const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                    const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                    float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                    int32_t union_stride, int32_t variant, int32_t* dev_status, void* stream);

/* The whole prompt-attention step in one launch, with each group's union built
 * inside the attention CTA ("sycl: prompt attention over 8-query selection unions
 * on XMX", Strata PR #2808, section Summary: the union of 8 neighbouring
 * positions' sorted selections; section What changed: there the union and the
 * attention run as a launch pair).  No union arrays reach global memory and no
 * workspace is needed.  The result is that of qsa_prompt_attn with
 * variant = QSA_ATTN_TCGEN05_SM, bit for bit: each CTA first builds its group's
 * union in shared memory with the union kernel's own algorithm, then runs that
 * variant's attention pipeline on it.
 *   - Arguments and layouts are those of qsa_prompt_attn without the workspace,
 *     union stride and variant.  Lists must be strictly increasing (the union
 *     build's precondition); counts outside [0, sel_stride] are clamped and
 *     reported as QSA_DEV_BAD_SEL_COUNT.  Device checks as in qsa_union_attn.
 *   - The union of 8 lists (up to 8 x sel_stride entries, 5 bytes each) must fit
 *     the CTA's shared memory next to the pipeline's (sm_103's per-block limit
 *     of 227 KB): sel_stride up to about 2,800 (2,056 holds the method's
 *     2,051-cell cap); QSA_ERR_UNSUPPORTED, before any CUDA call, above that,
 *     and for more than 65,535 groups (n_q > 524,280).
 *   - n_q == 0 returns QSA_OK with no launch. */
int qsa_fused_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                   const uint16_t* k_scale, const uint16_t* v_scale,
                   const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                   const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                   float sm_scale, float* out, int32_t* dev_status, void* stream);

/* Per-position selected-cell attention without unions: out[i][hq][:] is the same
 * softmax over query i's own resident selected cells as qsa_union_attn computes,
 * but every position gathers its own cells ("sycl: prompt attention over 8-query
 * selection unions on XMX", Strata PR #2808, section Summary: the prompt path's
 * default, each position gathering its own ~2,051 cells; section Extra Notes
 * times it against the union kernel).  It is the baseline the union path
 * replaces, built on the warp-level tensor path (mma.sync, FP32 sums): S on FP16
 * operands (Q converted from BF16 with the union kernel's exact power-of-two row
 * scaling, K as the exact INT8 integers, its scale on the score column in FP32),
 * P V on BF16 operands (V exact, P = p * v_scale rounded to BF16 once).  Each
 * (query, KV head) list is split
 * over four warps whose partial softmax states are merged at the end, so the
 * summation order differs from a single walk of the list (results agree within
 * BF16 rounding of the weights).  Arguments and layouts are those of
 * qsa_prompt_attn (sel: [n_q][sel_stride] cells, sel_count: [n_q]); no workspace.
 * The lists need not be sorted.  Device checks as in qsa_union_attn
 * (QSA_DEV_BAD_SEL_COUNT, QSA_DEV_BAD_CELL, QSA_DEV_BAD_PAGE into *dev_status).
 * n_q == 0 returns QSA_OK with no launch. */
int qsa_select_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                    const uint16_t* k_scale, const uint16_t* v_scale,
                    const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                    const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                    float sm_scale, float* out, int32_t* dev_status, void* stream);

/* Decode-time selected-cell attention over a batch of sequences: query i is the
 * current position of sequence i and attends to its own selected cells through
 * its own page table.  The union pages leave decode untouched ("sycl: prompt
 * attention over 8-query selection unions on XMX", Strata PR #2808, section
 * Summary: the decode kernel gathers each position's own cells); this is that
 * computation -- the softmax of qsa_select_attn, per query -- with one page table
 * per query instead of one for the whole chunk.
 *   - q: [n_q][n_kv*12][128] BF16; out: [n_q][n_kv*12][128] FP32, written for
 *     every query (zeros when no selected cell is resident).
 *   - page_tables: query i's table is page_tables[i * pt_stride ...], n_lpages
 *     entries (logical page -> physical page in the shared pools, < 0 = not
 *     resident).  pt_stride == 0 gives every query one shared table (then this
 *     is qsa_select_attn); otherwise pt_stride >= n_lpages.
 *   - Pools, scales, sel / sel_count / sel_stride, sm_scale, dev_status and
 *     stream as in qsa_select_attn; lists need not be sorted.
 *   - Returns QSA_ERR_ARG for a negative pt_stride or 0 < pt_stride < n_lpages,
 *     otherwise as qsa_select_attn.  n_q == 0 returns QSA_OK with no launch. */
int qsa_decode_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                    const uint16_t* k_scale, const uint16_t* v_scale,
                    const int32_t* page_tables, int32_t pt_stride, int32_t n_lpages, int32_t n_ppages,
                    int32_t n_kv, const int32_t* sel, const int32_t* sel_count, int32_t sel_stride,
                    int32_t n_q, float sm_scale, float* out, int32_t* dev_status, void* stream);

/* Self-test of the bounded waits (not part of the method: the pages have no
 * counterpart).  Every pipelined kernel here waits on mbarriers with a wall-time
 * limit and, when one runs out, records QSA_DEV_WAIT_TIMEOUT in *dev_status and
 * returns instead of hanging.  This launches one warp that waits on an mbarrier
 * nothing arrives on, for limit_us microseconds, then records that bit: a test
 * can see the whole path -- the wait ending by time, the device status reaching
 * the host, the context staying usable -- without faulting anything.
 *   - limit_us in (0, 10^7]; dev_status: device int32, OR-ed into, required.
 *   - Returns QSA_ERR_ARG otherwise, QSA_ERR_CUDA if the launch fails. */
int qsa_wait_selftest(int32_t limit_us, int32_t* dev_status, void* stream);

/* Bytes of the static device scratch behind qsa_prompt_attn_static (32 MiB):
 * room for n_q <= 3256 queries at union_stride 16448, more at smaller strides. */
#define QSA_STATIC_SCRATCH_BYTES (32u << 20)

/* qsa_prompt_attn without a workspace argument and without any allocation.
 * The method's description has no counterpart of this call: it exists for
 * callers that cannot hand over device memory -- a plain C host with no device
 * allocator of its own, for which cudaMalloc / cudaFree around each step would
 * synchronise the device, or a caller inside a framework whose allocator it
 * cannot reach.  The union arrays go to a scratch of QSA_STATIC_SCRATCH_BYTES
 * in this library's static device memory (one per device), and the result is
 * that of qsa_prompt_attn on a workspace of that size.
 *   - Arguments, layouts and ownership are those of qsa_prompt_attn; the
 *     stream must belong to the current device (QSA_ERR_ARG otherwise).
 *   - Checks that need no CUDA call come first, in this order: sizes, shape
 *     arguments and variant (QSA_ERR_ARG), then capacity: QSA_ERR_CAPACITY when
 *     qsa_union_workspace_bytes(n_q, union_stride) > QSA_STATIC_SCRATCH_BYTES,
 *     then null pointers (QSA_ERR_ARG).  QSA_ERR_CUDA when the scratch's
 *     address cannot be resolved.
 *   - The first call on each device resolves the scratch's address with
 *     cudaGetSymbolAddress (this may load the library's device code on that
 *     device) and caches it for the life of the process; make that first call
 *     before any stream capture begins.  The cached address is not valid after
 *     cudaDeviceReset (the module is loaded again and the scratch may move):
 *     a process that resets a device must not call this entry point on that
 *     device afterwards.
 *   - Nothing in the scratch must start at zero (the union build writes all
 *     that the attention kernel reads), so no call clears it.
 *   - All calls on one device share the one scratch: two calls whose work can
 *     overlap on the device (different streams, or different host threads
 *     without ordering between their streams) race on it.  Order them. */
int qsa_prompt_attn_static(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                           const uint16_t* k_scale, const uint16_t* v_scale,
                           const int32_t* page_table, int32_t n_lpages, int32_t n_ppages, int32_t n_kv,
                           const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                           float sm_scale, float* out, int32_t union_stride, int32_t variant,
                           int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif
