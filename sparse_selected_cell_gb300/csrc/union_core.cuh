// union_core.cuh -- the union of one group's selection lists, built by one CTA
// in shared memory: used by the union kernel (union_build.cu, results to global
// memory) and by the fused attention kernel (attn_sm.cu, results to shared
// memory, before its attention pipeline starts).
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary (for every 8 neighbouring positions, the sorted
// union of their selected cells, each marked with the positions that chose it)
// and section "What changed" (one work-group per 8 positions over a local cell
// bitmap).  Section Extra Notes fixes the storage: int32 cell + separate mask byte.
//
// The group's cell range is walked in windows of kUnionWindow cells held as a
// byte map in shared memory (byte = the 8-position mask); a context up to
// kUnionWindow cells is one window.  Each list is sorted, so its cells inside a
// window form one contiguous index range (found by binary search only when there
// are several windows).  Warps mark the lists (w % 8 = list), eight loads in
// flight per lane before their ORs of bit j into the cell's byte (OR is
// order-independent, so the result is deterministic).  The window is then
// compacted in cell order, visiting only the 64-cell pages that hold a marked
// cell (a page flag is set while marking; the flagged pages are listed in order
// by one block scan): each warp counts the entries of its contiguous run of
// listed pages, one shared-memory pass over the warp totals gives each warp its
// output offset, and each warp writes its pages' entries with warp-level prefix
// sums, two cells per lane.  Output is sorted by construction and bit-exact.
#pragma once
#include "qsa_common.cuh"

namespace qsa {

constexpr int kUnionWindow = 65536;                // cells (= bytes of shared memory) per window
constexpr int kUnionPages = kUnionWindow / kPage;  // 64-cell pages of a window

// Shared-memory scratch of one union build (every array owned by the CTA).
struct UnionScratch {
    uint4* map;        // kUnionWindow bytes: the window's byte map
    uint8_t* touched;  // [kUnionPages]: page p of the window holds a marked cell
    uint16_t* pages;   // [kUnionPages]: the touched pages, in increasing order
    int* cnt;          // [8]
    int* first;        // [8]
    int* last;         // [8]
    int* beg;          // [8]
    int* end;          // [8]
    int* warp;         // [kThreads / 32]
};

__device__ __forceinline__ int union_lower_bound(const int32_t* __restrict__ a, int n, long long x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if ((long long)__ldg(a + mid) < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Builds the union of queries q_begin .. q_begin + 7's lists (fewer for a ragged
// last group) into ucell / umask (global or shared memory), at most ustride
// entries; returns the union size (above ustride: the entries past it are not
// written).  Called by all kThreads threads of the CTA; it ends with the CTA
// synchronised.  A count outside [0, sel_stride] is clamped and reported.
template <int kThreads>
__device__ int build_group_union(const int32_t* __restrict__ sel, const int32_t* __restrict__ sel_count, int n_q,
                                 int sel_stride, int q_begin, int32_t* ucell, uint8_t* umask, int ustride,
                                 int32_t* dev_status, const UnionScratch& sc) {
    static_assert(kThreads % 32 == 0 && 2 * kThreads >= kUnionPages, "two page flags per thread");
    constexpr int kMarkUnroll = 8;                                   // list entries loaded per thread before marking
    constexpr int kMarkWarps = (kThreads / 32 / kGroup) * kGroup;    // warps that mark: whole sets of 8
    constexpr int kWindow = kUnionWindow;
    uint32_t* map32 = reinterpret_cast<uint32_t*>(sc.map);
    const uint16_t* map16 = reinterpret_cast<const uint16_t*>(sc.map);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nj = min(kGroup, n_q - q_begin);

    if (tid < kGroup) {
        int c = 0, first = INT32_MAX, last = INT32_MIN;
        if (tid < nj) {
            c = __ldg(sel_count + q_begin + tid);
            if (c < 0 || c > sel_stride) {
                report(dev_status, QSA_DEV_BAD_SEL_COUNT);
                c = c < 0 ? 0 : sel_stride;
            }
            if (c > 0) {
                const int32_t* lst = sel + (size_t)(q_begin + tid) * sel_stride;
                first = __ldg(lst);
                last = __ldg(lst + c - 1);
            }
        }
        sc.cnt[tid] = c;
        sc.first[tid] = first;
        sc.last[tid] = last;
    }
    __syncthreads();
    long long lo = INT32_MAX, hi = INT32_MIN;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        if (sc.cnt[j] > 0) {
            lo = min(lo, (long long)sc.first[j]);
            hi = max(hi, (long long)sc.last[j]);
        }
    }
    int written = 0;   // union entries produced so far (same value in every thread)
    for (long long w0 = lo & ~(long long)(kPage - 1); w0 <= hi; w0 += kWindow) {
        // 1. clear the byte map and the page flags of this window (the part it can use)
        const long long span = min((long long)kWindow, hi - w0 + 1);
        const int n_pg = (int)((span + kPage - 1) / kPage);   // pages the compaction may read
        const int n_pieces = n_pg * (kPage / 16);
        for (int p = tid; p < n_pieces; p += kThreads) sc.map[p] = make_uint4(0, 0, 0, 0);
        for (int p = tid; p < n_pg; p += kThreads) sc.touched[p] = 0;
        // 2. index range of each list inside [w0, w0 + kWindow)
        const bool one_window = hi - w0 < kWindow;
        if (tid < kGroup) {
            int b = 0, e = 0;
            if (sc.cnt[tid] > 0) {
                if (one_window) {
                    e = sc.cnt[tid];
                } else {
                    const int32_t* lst = sel + (size_t)(q_begin + tid) * sel_stride;
                    b = union_lower_bound(lst, sc.cnt[tid], w0);
                    e = union_lower_bound(lst, sc.cnt[tid], w0 + kWindow);
                }
            }
            sc.beg[tid] = b;
            sc.end[tid] = e;
        }
        __syncthreads();
        // 3. mark: bit j of the byte of every cell in list j, and the cell's page
        // flag.  Warps w and w + 8 take list w % 8, kMarkUnroll loads per lane in
        // flight before the ORs.  Cells outside the window (several windows) or
        // outside [0, n) cannot occur in one window: lo and hi bound every list.
        {
            const int j = warp & (kGroup - 1);
            if (j < nj && warp < kMarkWarps) {
                const int32_t* lst = sel + (size_t)(q_begin + j) * sel_stride;
                const int e = sc.end[j];
                constexpr int kStride = kMarkWarps / kGroup * 32;   // lanes on one list
                for (int t0 = sc.beg[j] + (warp / kGroup) * 32 + lane; t0 < e; t0 += kStride * kMarkUnroll) {
                    int cell[kMarkUnroll];
#pragma unroll
                    for (int u = 0; u < kMarkUnroll; ++u) {
                        const int t = t0 + u * kStride;
                        cell[u] = t < e ? __ldg(lst + t) : INT32_MIN;
                    }
#pragma unroll
                    for (int u = 0; u < kMarkUnroll; ++u) {
                        const long long off = (long long)cell[u] - w0;
                        if (cell[u] != INT32_MIN && off >= 0 && off < span) {
                            atomicOr(map32 + (off >> 2), 1u << (((int)off & 3) * 8 + j));
                            sc.touched[off >> 6] = 1;
                        }
                    }
                }
            }
        }
        __syncthreads();
        // 4. the touched pages in increasing order: thread t owns flags [2t, 2t+2)
        {
            int f[2], c = 0;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int p = 2 * tid + k;
                f[k] = p < n_pg ? sc.touched[p] : 0;
                c += f[k];
            }
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sc.warp[warp] = incl;
            __syncthreads();
            int base = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) base += w < warp ? sc.warp[w] : 0;
            int idx = base + incl - c;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (f[k]) sc.pages[idx++] = (uint16_t)(2 * tid + k);
        }
        int n_touched = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) n_touched += sc.warp[w];
        __syncthreads();
        // 5. compact the touched pages in cell order.  Warp w owns the contiguous
        // run of touched pages [w * per_warp, (w + 1) * per_warp); a page is one
        // step of the warp, lane i holding cells 2i and 2i+1.  The warps' entry
        // counts go through one block pass, then each warp writes its pages with
        // warp-level scans.
        const int per_warp = (n_touched + kThreads / 32 - 1) / (kThreads / 32);
        const int t_lo = min(n_touched, warp * per_warp), t_hi = min(n_touched, t_lo + per_warp);
        int cnt_w = 0;
        for (int t = t_lo; t < t_hi; ++t) {
            const uint32_t two = map16[sc.pages[t] * (kPage / 2) + lane];
            cnt_w += __popc(__ballot_sync(0xffffffffu, (two & 0xFFu) != 0)) +
                     __popc(__ballot_sync(0xffffffffu, (two >> 8) != 0));
        }
        if (lane == 0) sc.warp[warp] = cnt_w;
        __syncthreads();
        int run = written, total = 0;   // run: output index of this warp's first entry
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int x = sc.warp[w];
            run += w < warp ? x : 0;
            total += x;
        }
        for (int t = t_lo; t < t_hi; ++t) {
            const int pg = sc.pages[t];
            const uint32_t two = map16[pg * (kPage / 2) + lane];
            const uint32_t m0 = two & 0xFFu, m1 = two >> 8;
            const int n = (m0 != 0) + (m1 != 0);
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int idx = run + incl - n;
            const int cell0 = (int)(w0 + (long long)pg * kPage) + 2 * lane;
            if (m0) {
                if (idx < ustride) {
                    ucell[idx] = cell0;
                    umask[idx] = (uint8_t)m0;
                }
                ++idx;
            }
            if (m1 && idx < ustride) {
                ucell[idx] = cell0 + 1;
                umask[idx] = (uint8_t)m1;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        written += total;
        __syncthreads();      // the map, the page list and sc.warp are reused by the next window
    }
    return written;
}

}  // namespace qsa
