// capi.cu -- the extern "C" boundary of libqsa.so (declared in include/qsa.h):
// argument validation, workspace carving and kernel launches.  No allocation,
// no synchronisation, no host fallback.
#include <cstdint>
#include <cuda_runtime.h>

#include "qsa_common.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

struct UnionLayout {
    size_t cells, mask, count, total;
};

UnionLayout union_layout(int32_t n_q, int32_t union_stride) {
    const size_t groups = (size_t)((n_q + qsa::kGroup - 1) / qsa::kGroup);
    UnionLayout L;
    L.cells = 0;
    L.mask = align_up(groups * (size_t)union_stride * sizeof(int32_t));
    L.count = L.mask + align_up(groups * (size_t)union_stride);
    L.total = L.count + align_up(groups * sizeof(int32_t));
    return L;
}

int check_union_args(int32_t n_q, int32_t union_stride) {
    if (n_q < 0 || union_stride <= 0 || union_stride % 64 != 0) return QSA_ERR_ARG;
    return QSA_OK;
}

int check_attn_args(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                    const uint16_t* v_scale, const int32_t* page_table, int32_t n_lpages, int32_t n_ppages,
                    int32_t n_kv, int32_t n_q, float* out, int32_t variant) {
    if (n_q < 0 || n_lpages < 0 || n_ppages < 0 || n_kv <= 0) return QSA_ERR_ARG;
    if (variant < QSA_ATTN_DEFAULT || variant > QSA_ATTN_TCGEN05_SM) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!q || !out || !page_table) return QSA_ERR_ARG;
    if (n_ppages > 0 && (!k_pool || !v_pool || !k_scale || !v_scale)) return QSA_ERR_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_pool) || !aligned16(v_pool)) return QSA_ERR_ARG;
    // index arithmetic of the kernels: rows of q/out and pool rows fit in 32-bit grid terms
    if ((long long)n_q * n_kv * qsa::kHeadsPerKv > (1LL << 31) / qsa::kHeadDim) return QSA_ERR_UNSUPPORTED;
    if ((long long)n_lpages * qsa::kPage > (1LL << 31)) return QSA_ERR_UNSUPPORTED;
    if ((n_q + qsa::kGroup - 1) / qsa::kGroup > (1 << 30) || n_kv > 65535) return QSA_ERR_UNSUPPORTED;
    return QSA_OK;
}

}  // namespace

extern "C" {

int qsa_attn_default_variant(void) { return QSA_ATTN_TCGEN05; }

const char* qsa_status_str(int status) {
    switch (status) {
        case QSA_OK: return "ok";
        case QSA_ERR_ARG: return "invalid argument";
        case QSA_ERR_UNSUPPORTED: return "unsupported shape or variant";
        case QSA_ERR_CAPACITY: return "workspace too small";
        case QSA_ERR_CUDA: return "CUDA launch failed";
        case QSA_ERR_DEVICE_CHECK: return "device-side check failed";
        default: return "unknown status";
    }
}

size_t qsa_union_workspace_bytes(int32_t n_q, int32_t union_stride) {
    if (n_q < 0 || union_stride <= 0) return 0;
    return union_layout(n_q, union_stride).total;
}

int qsa_union_build(const int32_t* sel, const int32_t* sel_count, int32_t n_q, int32_t sel_stride,
                    int32_t* union_cells, uint8_t* union_mask, int32_t* union_count, int32_t union_stride,
                    int32_t* dev_status, void* stream) {
    int rc = check_union_args(n_q, union_stride);
    if (rc != QSA_OK) return rc;
    if (sel_stride <= 0) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!sel || !sel_count || !union_cells || !union_mask || !union_count) return QSA_ERR_ARG;
    return cuda_status(qsa::launch_union_build(sel, sel_count, n_q, sel_stride, union_cells, union_mask, union_count,
                                               union_stride, dev_status, static_cast<cudaStream_t>(stream)));
}

int qsa_union_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                   const uint16_t* v_scale, const int32_t* page_table, int32_t n_lpages, int32_t n_ppages,
                   int32_t n_kv, const int32_t* union_cells, const uint8_t* union_mask,
                   const int32_t* union_count, int32_t union_stride, int32_t n_q, float sm_scale, float* out,
                   int32_t variant, int32_t* dev_status, void* stream) {
    int rc = check_union_args(n_q, union_stride);
    if (rc != QSA_OK) return rc;
    rc = check_attn_args(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, n_q, out,
                         variant);
    if (rc != QSA_OK) return rc;
    if (n_q == 0) return QSA_OK;
    if (!union_cells || !union_mask || !union_count) return QSA_ERR_ARG;
    const qsa::AttnArgs a{q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv,
                          union_cells, union_mask, union_count, union_stride, n_q, sm_scale, out, dev_status,
                          nullptr, nullptr, 0};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (variant == QSA_ATTN_DEFAULT) variant = qsa_attn_default_variant();
    if (variant == QSA_ATTN_TCGEN05_SM) return cuda_status(qsa::launch_attn_sm(a, s));
    return cuda_status(qsa::launch_attn_tc(a, s));
}

int qsa_prompt_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                    const uint16_t* v_scale, const int32_t* page_table, int32_t n_lpages, int32_t n_ppages,
                    int32_t n_kv, const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                    float sm_scale, float* out, void* workspace, size_t workspace_bytes, int32_t union_stride,
                    int32_t variant, int32_t* dev_status, void* stream) {
    int rc = check_union_args(n_q, union_stride);
    if (rc != QSA_OK) return rc;
    rc = check_attn_args(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, n_q, out,
                         variant);
    if (rc != QSA_OK) return rc;
    if (sel_stride <= 0) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!sel || !sel_count || !workspace) return QSA_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return QSA_ERR_ARG;
    const UnionLayout L = union_layout(n_q, union_stride);
    if (workspace_bytes < L.total) return QSA_ERR_CAPACITY;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* ucell = reinterpret_cast<int32_t*>(ws + L.cells);
    uint8_t* umask = ws + L.mask;
    int32_t* ucount = reinterpret_cast<int32_t*>(ws + L.count);
    rc = qsa_union_build(sel, sel_count, n_q, sel_stride, ucell, umask, ucount, union_stride, dev_status, stream);
    if (rc != QSA_OK) return rc;
    return qsa_union_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, ucell, umask,
                          ucount, union_stride, n_q, sm_scale, out, variant, dev_status, stream);
}

int qsa_fused_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                   const uint16_t* v_scale, const int32_t* page_table, int32_t n_lpages, int32_t n_ppages,
                   int32_t n_kv, const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                   float sm_scale, float* out, int32_t* dev_status, void* stream) {
    int rc = check_attn_args(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, n_q, out,
                             QSA_ATTN_DEFAULT);
    if (rc != QSA_OK) return rc;
    if (sel_stride <= 0) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!sel || !sel_count) return QSA_ERR_ARG;
    // the group's union (up to 8 x sel_stride entries) must fit the CTA's shared
    // memory next to the pipeline's: sm_103's per-block opt-in limit is 227 KB
    if (qsa::attn_fused_smem_bytes(sel_stride) > (size_t)227 * 1024) return QSA_ERR_UNSUPPORTED;
    // the fused grid is (KV head, group): the group count is its y extent
    if ((n_q + qsa::kGroup - 1) / qsa::kGroup > 65535) return QSA_ERR_UNSUPPORTED;
    const qsa::AttnArgs a{q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv,
                          nullptr, nullptr, nullptr, 0, n_q, sm_scale, out, dev_status,
                          sel, sel_count, sel_stride};
    return cuda_status(qsa::launch_attn_fused(a, static_cast<cudaStream_t>(stream)));
}

int qsa_select_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                    const uint16_t* v_scale, const int32_t* page_table, int32_t n_lpages, int32_t n_ppages,
                    int32_t n_kv, const int32_t* sel, const int32_t* sel_count, int32_t sel_stride, int32_t n_q,
                    float sm_scale, float* out, int32_t* dev_status, void* stream) {
    int rc = check_attn_args(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, n_q, out,
                             QSA_ATTN_DEFAULT);
    if (rc != QSA_OK) return rc;
    if (sel_stride <= 0) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!sel || !sel_count) return QSA_ERR_ARG;
    const qsa::SelArgs a{q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv,
                         sel, sel_count, sel_stride, n_q, sm_scale, out, dev_status, 0};
    return cuda_status(qsa::launch_select_attn(a, static_cast<cudaStream_t>(stream)));
}

int qsa_decode_attn(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool, const uint16_t* k_scale,
                    const uint16_t* v_scale, const int32_t* page_tables, int32_t pt_stride, int32_t n_lpages,
                    int32_t n_ppages, int32_t n_kv, const int32_t* sel, const int32_t* sel_count, int32_t sel_stride,
                    int32_t n_q, float sm_scale, float* out, int32_t* dev_status, void* stream) {
    int rc = check_attn_args(q, k_pool, v_pool, k_scale, v_scale, page_tables, n_lpages, n_ppages, n_kv, n_q, out,
                             QSA_ATTN_DEFAULT);
    if (rc != QSA_OK) return rc;
    if (sel_stride <= 0 || pt_stride < 0 || (pt_stride > 0 && pt_stride < n_lpages)) return QSA_ERR_ARG;
    if (n_q == 0) return QSA_OK;
    if (!sel || !sel_count) return QSA_ERR_ARG;
    const qsa::SelArgs a{q, k_pool, v_pool, k_scale, v_scale, page_tables, n_lpages, n_ppages, n_kv,
                         sel, sel_count, sel_stride, n_q, sm_scale, out, dev_status, pt_stride};
    return cuda_status(qsa::launch_select_attn(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
