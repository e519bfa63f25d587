// prompt_attn_static.cu -- qsa_prompt_attn_static (declared in include/qsa.h):
// the whole prompt-attention step with its union arrays in a fixed scratch that
// lives in this library's own static device memory, so the call allocates
// nothing and takes no workspace from the caller.
//
// Who needs it: a caller that cannot hand over device memory.  A plain C host
// with no device allocator of its own would otherwise have to call cudaMalloc /
// cudaFree around every step, and those synchronise the device (stalling the
// other streams of a serving loop); a caller running under an allocator it does
// not own (a framework's caching allocator it must not reach into) has no way
// to reserve the workspace at all.  Here the memory exists from module load on.
//
// The call validates, looks up the scratch's device address (once per device),
// and then runs the unchanged qsa_prompt_attn on it.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "qsa.h"

// Union arrays of one step (union_cells, union_mask, union_count, laid out as
// qsa_union_workspace_bytes describes).  Nothing here must start at zero: the
// union build writes every group's count and every entry below it before the
// attention kernel reads them, and nothing past a group's count is read.
static __device__ __align__(256) uint8_t qsa_static_union_scratch[QSA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch[kMaxDevices];   // device address per device ordinal, set once
std::mutex g_setup;

// Device address of the scratch on the current device.  The first call on a
// device resolves it with cudaGetSymbolAddress (which may load this module on
// that device); later calls read the cached pointer.
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QSA_ERR_UNSUPPORTED;
    void* p = g_scratch[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup);
        p = g_scratch[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            if (cudaGetSymbolAddress(&p, qsa_static_union_scratch) != cudaSuccess || p == nullptr) return QSA_ERR_CUDA;
            if ((reinterpret_cast<uintptr_t>(p) & 255u) != 0) return QSA_ERR_CUDA;
            g_scratch[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return QSA_OK;
}

}  // namespace

extern "C" int qsa_prompt_attn_static(const uint16_t* q, const int8_t* k_pool, const int8_t* v_pool,
                                      const uint16_t* k_scale, const uint16_t* v_scale, const int32_t* page_table,
                                      int32_t n_lpages, int32_t n_ppages, int32_t n_kv, const int32_t* sel,
                                      const int32_t* sel_count, int32_t sel_stride, int32_t n_q, float sm_scale,
                                      float* out, int32_t union_stride, int32_t variant, int32_t* dev_status,
                                      void* stream) {
    // host-only checks first, before anything touches CUDA: sizes and shape
    // arguments, then the scratch's capacity, then the pointers
    if (n_q < 0 || union_stride <= 0 || union_stride % 64 != 0) return QSA_ERR_ARG;
    if (n_lpages < 0 || n_ppages < 0 || n_kv <= 0 || sel_stride <= 0) return QSA_ERR_ARG;
    if (variant < QSA_ATTN_DEFAULT || variant > QSA_ATTN_TCGEN05_SM) return QSA_ERR_ARG;
    if (n_q == 0)
        return qsa_prompt_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, sel,
                               sel_count, sel_stride, n_q, sm_scale, out, nullptr, 0, union_stride, variant,
                               dev_status, stream);
    if (qsa_union_workspace_bytes(n_q, union_stride) > (size_t)QSA_STATIC_SCRATCH_BYTES) return QSA_ERR_CAPACITY;
    if (!q || !out || !page_table || !sel || !sel_count) return QSA_ERR_ARG;
    // the scratch used is the current device's: a stream of another device is refused
    if (stream != nullptr) {
        int dev = -1, sdev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
        if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return QSA_ERR_ARG;
        if (sdev != dev) return QSA_ERR_ARG;
    }
    void* scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != QSA_OK) return rc;
    return qsa_prompt_attn(q, k_pool, v_pool, k_scale, v_scale, page_table, n_lpages, n_ppages, n_kv, sel, sel_count,
                           sel_stride, n_q, sm_scale, out, scratch, (size_t)QSA_STATIC_SCRATCH_BYTES, union_stride,
                           variant, dev_status, stream);
}
