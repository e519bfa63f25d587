// union_build.cu -- first kernel: per group of 8 neighbouring queries, the sorted
// union of their selection lists with an 8-bit membership mask per cell.
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary (for every 8 neighbouring positions, the sorted
// union of their selected cells, each marked with the positions that chose it)
// and section "What changed" (one work-group per 8 positions over a local cell
// bitmap).  Section Extra Notes fixes the storage: int32 cell + separate mask byte.
//
// GB300 design: one 512-thread CTA per group, running the shared-memory build of
// union_core.cuh (a byte map per window of cells, marking, a page scan and an
// ordered compaction) with its output in the group's rows of the union arrays.
#include "union_core.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads)
union_build_kernel(const int32_t* __restrict__ sel, const int32_t* __restrict__ sel_count, int n_q,
                   int sel_stride, int32_t* __restrict__ ucell, uint8_t* __restrict__ umask,
                   int32_t* __restrict__ ucount, int ustride, int32_t* dev_status) {
    extern __shared__ uint4 smem_map[];                  // kUnionWindow bytes
    __shared__ uint8_t s_touched[kUnionPages];
    __shared__ uint16_t s_pages[kUnionPages];
    __shared__ int s_small[5 * kGroup];
    __shared__ int s_warp[kThreads / 32];
    const UnionScratch sc{smem_map, s_touched, s_pages, s_small, s_small + kGroup, s_small + 2 * kGroup,
                          s_small + 3 * kGroup, s_small + 4 * kGroup, s_warp};
    const int g = blockIdx.x;
    const size_t out_base = (size_t)g * ustride;
    int written = build_group_union<kThreads>(sel, sel_count, n_q, sel_stride, g * kGroup, ucell + out_base,
                                              umask + out_base, ustride, dev_status, sc);
    if (threadIdx.x == 0) {
        if (written > ustride) {
            report(dev_status, QSA_DEV_UNION_OVERFLOW);
            written = ustride;
        }
        ucount[g] = written;
    }
}

}  // namespace

cudaError_t launch_union_build(const int32_t* sel, const int32_t* sel_count, int n_q, int sel_stride,
                               int32_t* union_cells, uint8_t* union_mask, int32_t* union_count,
                               int union_stride, int32_t* dev_status, cudaStream_t stream) {
    // Per-call (and so per-device) opt-in to the 64 KB byte map.
    cudaError_t e = cudaFuncSetAttribute(union_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUnionWindow);
    if (e != cudaSuccess) return e;
    const int n_groups = (n_q + kGroup - 1) / kGroup;
    union_build_kernel<<<n_groups, kThreads, kUnionWindow, stream>>>(sel, sel_count, n_q, sel_stride, union_cells,
                                                                 union_mask, union_count, union_stride,
                                                                 dev_status);
    return cudaGetLastError();
}

}  // namespace qsa
