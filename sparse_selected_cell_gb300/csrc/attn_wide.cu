// attn_wide.cu -- union attention on the 5th-generation tensor cores, persistent
// and one CTA per SM: 128-cell chunks, the Q operand in Tensor Memory.
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary: one work-group per (8 positions, KV head) covers
// the 96 rows of 8 positions x 12 heads; the INT8 K/V of each chunk of the
// union is dequantised once; S = Q K^T and O += P V run on the matrix units with
// FP32 sums; in the online softmax a cell is -inf for every position that did
// not select it.  Section Extra Notes: non-resident pages are masked.
//
// The arithmetic is that of attn_tc.cu (exact BF16 K and V, the K scale times
// sm_scale * log2(e) on the FP32 score column, the V scale folded into P, a lazy
// exp2-domain rescale); what differs is the shape of the pipeline:
//   * One CTA per SM owns all 512 Tensor Memory columns: two 128-column S
//     buffers, the Q operand (64 columns: 128 lanes x 128 BF16), O (128).  With
//     Q in Tensor Memory the tensor core reads only K and V from shared memory,
//     and S = Q K^T runs 128 columns wide (M=128 N=128 K=16 issues at the full
//     rate, where N=64 costs the same time for half the work).
//   * The CTA is persistent: it works through the (group g, KV head h) items
//     blockIdx.x, blockIdx.x + gridDim.x, ... as one stream of chunks, so the
//     producer and loaders run on into the next item while the softmax ends the
//     current one.
// Warp roles (24 warps):
//   softmax   warps w < 16 with w % 4 != 3: lane quadrant w % 4 (rows
//             32 * (w % 4) + lane), column quarter w / 4 (S columns [32q, 32q+32)
//             of each chunk).  The four warps of a quadrant swap their quarter
//             maxima through shared memory (one mbarrier per quadrant and
//             chunk) and so share one running max; each keeps its own FP32 sum of
//             p, writes P over its own S columns and owns 32 of O's columns.
//             They write each item's Q rows into Tensor Memory, the first item's
//             at the start and the next item's once the last S of the current
//             one has completed.
//   warps 3, 22  producers (even and odd chunks of the CTA's stream; one warp's
//             chain of dependent loads per chunk is longer than a chunk takes):
//             union entries -> page table -> per-chunk tables (pool row, K/V
//             scales, one 32-bit selection word per query and quarter), an L2
//             prefetch of each chunk's K/V rows and of the next item's Q.
//   warps 7, 23  MMA issuers (one thread each): S(t) = Q K^T into S buffer t & 1;
//             O += P(t) V, an item's first P V waiting until the softmax has read
//             the previous item's O.
//   warps 11, 15, 16-21  loaders/converters, four for K and four for V: bulk
//             copies of the INT8 rows (8 KB per whole page, else 128 B per row)
//             into a shared-memory staging ring two chunks ahead, then conversion
//             to BF16 into 128-byte-swizzled operand tiles (two deep).
// Rows 96-127 (TMEM lanes 96-127) are padding: never written, never read back.
// Every wait is bounded in time (see attn_tc.cu).
#include "qsa_common.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace {

constexpr int kCW = 128;                       // union cells per chunk
constexpr int kQuarters = kCW / 32;            // softmax warps per lane quadrant
constexpr int kSoftW = 3 * kQuarters;          // 12
constexpr int kLoadW = 8;
constexpr int kLoadThreads = 32 * kLoadW;
constexpr int kWarpsW = 24;
constexpr int kThreadsW = 32 * kWarpsW;        // 768
constexpr int kWarpProd = 3, kWarpProd2 = 22, kWarpMmaW = 7, kWarpPvW = 23;
constexpr int kProducers = 2;                  // producer p writes the tables of chunks t = p (mod 2)
constexpr int kNSW = 6;                        // per-chunk table ring
constexpr int kNBW = 2;                        // BF16 K / V operand tiles
constexpr int kNStage = 2;                     // INT8 staging slots (bulk copies land here)
constexpr uint32_t kTmemColsW = 512;
constexpr uint32_t kColS = 0, kColQ = 256, kColO = 384;   // S buffer sb at kColS + 128 * sb
constexpr float kRescaleLog2W = 32.f;
constexpr uint64_t kWaitNsW = 1000000000ull;

struct TabW {
    int32_t row[kCW];               // pool row (page * n_kv + h) * 64 + cell % 64; -1 for a masked cell
    float ks[kCW];                  // K scale * sm_scale * log2(e); 0 for a masked cell
    float vs[kCW];                  // V scale; 0 for a masked cell
    uint32_t rowmask[kGroup][kQuarters];   // bit c of [j][q]: query j selected resident cell 32q + c
    int32_t page_row[4];            // [half]: first pool row when the 64 cells of the half are one
                                    // whole resident page (its 8 KB of K, of V, contiguous); else -1
};

constexpr uint32_t kTileW = kCW * kHeadDim * 2;   // 32 KB BF16 K or V tile (two 64-column halves)
constexpr uint32_t kHalfW = kTileW / 2;
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kNBW * kTileW;
constexpr uint32_t kStageBytes = 2 * kCW * kHeadDim;   // 32 KB: the chunk's INT8 K rows, then its V rows
constexpr uint32_t kOffStage = kOffV + kNBW * kTileW;
constexpr uint32_t kOffTab = kOffStage + kNStage * kStageBytes;
// quarter maxima by chunk parity [2][quarter][row], then the row sums [quarter][row]
constexpr uint32_t kOffX = kOffTab + kNSW * (uint32_t)sizeof(TabW);
constexpr uint32_t kXFloats = 3 * kQuarters * kRows;
constexpr uint32_t kOffBarsW = (kOffX + kXFloats * 4 + 7u) & ~7u;
enum { B_TAB_FULL = 0, B_TAB_EMPTY = kNSW, B_K_FULL = 2 * kNSW, B_K_EMPTY = B_K_FULL + kNBW,
       B_V_FULL = B_K_EMPTY + kNBW, B_V_EMPTY = B_V_FULL + kNBW, B_S_FULL = B_V_EMPTY + kNBW,
       B_P_READY = B_S_FULL + 2, B_PV_DONE = B_P_READY + 2, B_O_DONE = B_PV_DONE + 2, B_O_FREE, B_Q_READY,
       B_DRAIN, B_DRAIN_PV, B_QUAD, B_ST_FULL = B_QUAD + 3, B_ST_EMPTY = B_ST_FULL + 2 * kNStage,
       B_NUM = B_ST_EMPTY + 2 * kNStage };   // staging barriers [part (K, V)][slot]
constexpr uint32_t kOffMiscW = kOffBarsW + B_NUM * 8;     // tmem base, abort flag
constexpr uint32_t kSmemW = kOffMiscW + 16 + 1024;        // + alignment slack
static_assert(kSmemW <= 227 * 1024, "shared memory budget");
static_assert(sizeof(TabW) % 16 == 0, "table alignment");

struct CtxW {
    const AttnArgs* a;
    uint8_t* base;
    uint32_t base_u;
    uint32_t tmem;
    volatile int* abort_flag;
    int n_heads, n_items;
    float kmul;
    int g, h, nj, q_begin, U, n_chunks;   // the current item (each role keeps its own copy)
};

__device__ __forceinline__ uint32_t barw(const CtxW& c, int i) { return c.base_u + kOffBarsW + 8u * i; }
__device__ __forceinline__ TabW* tab(const CtxW& c, int s) { return reinterpret_cast<TabW*>(c.base + kOffTab) + s; }

__device__ __forceinline__ bool waitw(const CtxW& c, uint32_t addr, uint32_t parity) {
    if (tc::mbar_wait(addr, parity, c.abort_flag, kWaitNsW)) return true;
    report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
    return false;
}

// Item w = h * n_groups + g: at any time the CTAs work on neighbouring groups of
// one KV head, so the live part of the K/V pool is one head's pages (L2-resident).
// Every role walks the same item sequence and reads the same union count, so all
// agree on each item's chunk count.
__device__ __forceinline__ void set_item(CtxW& c, int w) {
    const AttnArgs& a = *c.a;
    const int n_groups = c.n_items / a.n_kv;
    c.h = w / n_groups;
    c.g = w - c.h * n_groups;
    c.q_begin = c.g * kGroup;
    c.nj = min(kGroup, a.n_q - c.q_begin);
    int U = __ldg(a.union_count + c.g);
    if (U < 0 || U > a.union_stride) {
        report(a.dev_status, QSA_DEV_BAD_UNION_COUNT);
        U = U < 0 ? 0 : a.union_stride;
    }
    c.U = U;
    c.n_chunks = (U + kCW - 1) / kCW;
}

// Next item after w that has chunks (n_items if none); leaves it in c.
__device__ __forceinline__ int next_item(CtxW& c, int w) {
    for (w += gridDim.x; w < c.n_items; w += gridDim.x) {
        set_item(c, w);
        if (c.n_chunks > 0) return w;
    }
    return c.n_items;
}

// Barrier among the four softmax warps of lane quadrant q (their n-th call):
// an mbarrier with one arrival per warp, so that the wait is bounded like every
// other wait (a warp that gave up never leaves its partners blocked).
__device__ __forceinline__ bool quad_sync(const CtxW& c, int q, uint32_t n) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(barw(c, B_QUAD + q));
    return waitw(c, barw(c, B_QUAD + q), n & 1);
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void prefetch_l2w(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

constexpr int kPer = kCW / 32;   // union entries per producer lane per chunk

struct EntW {
    int cell[kPer];
    int mask[kPer];   // bits 0-7: the group's queries that selected the cell; bit 8: entry present
};

// Chunk placement as in attn_tc.cu, with 128-cell chunks: `lead` is the index of
// the first page-aligned union cell among entries 1..63 (0 if none); chunk c
// holds union positions lead + 128c + slot, a position past the end wrapping to
// entry p - U when that is one of the `lead` entries before it.
__device__ __forceinline__ int union_lead_w(const CtxW& c, int lane) {
    const int32_t* ucell = c.a->union_cells + (size_t)c.g * c.a->union_stride;
    const uint32_t b0 =
        __ballot_sync(0xffffffffu, lane >= 1 && lane < c.U && (__ldg(ucell + lane) & (kPage - 1)) == 0);
    if (b0) return __ffs(b0) - 1;
    const uint32_t b1 = __ballot_sync(0xffffffffu, 32 + lane < c.U && (__ldg(ucell + 32 + lane) & (kPage - 1)) == 0);
    return b1 ? 31 + __ffs(b1) : 0;
}

__device__ __forceinline__ EntW load_ent(const CtxW& c, int lead, int chunk, int lane) {
    EntW e;
    const int32_t* ucell = c.a->union_cells + (size_t)c.g * c.a->union_stride;
    const uint8_t* umask = c.a->union_mask + (size_t)c.g * c.a->union_stride;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int p = lead + chunk * kCW + lane + 32 * k;
        const int u = p < c.U ? p : (p - c.U < lead ? p - c.U : -1);
        const bool present = chunk < c.n_chunks && u >= 0;
        e.cell[k] = present ? __ldg(ucell + u) : 0;
        e.mask[k] = present ? (int)__ldg(umask + u) | 0x100 : 0;
    }
    return e;
}

// Page-table loads for the present entries (-1: absent, bad cell, or not resident).
__device__ __forceinline__ void load_pg(const CtxW& c, const EntW& e, int (&pg)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        pg[k] = -1;
        if (!(e.mask[k] & 0x100)) continue;
        const int cell = e.cell[k];
        if (cell < 0 || (cell >> 6) >= c.a->n_lpages) {
            report(c.a->dev_status, QSA_DEV_BAD_CELL);
            continue;
        }
        pg[k] = __ldg(c.a->page_table + (cell >> 6));
    }
}

__device__ __forceinline__ void rows_of(const CtxW& c, const EntW& e, const int (&pg)[kPer], int (&row)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        row[k] = -1;
        if (pg[k] < 0) continue;
        if (pg[k] >= c.a->n_ppages) {
            report(c.a->dev_status, QSA_DEV_BAD_PAGE);
            continue;
        }
        row[k] = (pg[k] * c.a->n_kv + c.h) * kPage + (e.cell[k] & (kPage - 1));
    }
}

// K and V scale of each entry, packed (K low, V high half).
__device__ __forceinline__ void load_sc(const CtxW& c, const int (&row)[kPer], uint32_t (&sc)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        sc[k] = row[k] >= 0 ? (uint32_t)__ldg(c.a->k_scale + row[k]) | ((uint32_t)__ldg(c.a->v_scale + row[k]) << 16)
                            : 0u;
}

// The chunks i of one item with t0 + i = p (mod kProducers); table ring slots
// continue from t0.  Three of the producer's chunks of dependent loads stay in
// flight: entries of its chunk i+3s, page table of i+2s, scales of i+s (s =
// kProducers), while chunk i's table is written.
__device__ bool producer_item(const CtxW& c, int lane, int t0, int p) {
    constexpr int s = kProducers;
    const int lead = union_lead_w(c, lane);
    const int i0 = ((p - t0) % s + s) % s;
    EntW e0 = load_ent(c, lead, i0, lane), e1 = load_ent(c, lead, i0 + s, lane), e2 = load_ent(c, lead, i0 + 2 * s, lane);
    int pg0[kPer], pg1[kPer], r0[kPer];
    load_pg(c, e0, pg0);
    load_pg(c, e1, pg1);
    rows_of(c, e0, pg0, r0);
    uint32_t s0[kPer];
    load_sc(c, r0, s0);
    for (int i = i0; i < c.n_chunks; i += s) {
        const int t = t0 + i, ts = t % kNSW;
        const EntW e3 = load_ent(c, lead, i + 3 * s, lane);
        int pg2[kPer], r1[kPer];
        uint32_t s1[kPer];
        load_pg(c, e2, pg2);
        rows_of(c, e1, pg1, r1);
        load_sc(c, r1, s1);
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            if (r1[k] >= 0) {
                const size_t off = (size_t)r1[k] * kHeadDim;
                prefetch_l2w(c.a->k_pool + off);
                prefetch_l2w(c.a->v_pool + off);
            }
        if (!waitw(c, barw(c, B_TAB_EMPTY + ts), ((t / kNSW) & 1) ^ 1)) return false;
        TabW* T = tab(c, ts);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const bool ok = r0[k] >= 0;
            T->row[lane + 32 * k] = ok ? r0[k] : -1;
            T->ks[lane + 32 * k] = ok ? __half2float(__ushort_as_half((uint16_t)(s0[k] & 0xFFFFu))) * c.kmul : 0.f;
            T->vs[lane + 32 * k] = ok ? __half2float(__ushort_as_half((uint16_t)(s0[k] >> 16))) : 0.f;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // whole-page halves: one bulk copy each for K and V
            const int base = __shfl_sync(0xffffffffu, r0[2 * hh], 0);
            const bool mine = base >= 0 && (base & (kPage - 1)) == 0 && r0[2 * hh] == base + lane &&
                              r0[2 * hh + 1] == base + 32 + lane;
            const bool whole = __all_sync(0xffffffffu, mine);
            if (lane == 0) T->page_row[hh] = whole ? base : -1;
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j)
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const uint32_t b = __ballot_sync(0xffffffffu, r0[k] >= 0 && ((e0.mask[k] >> j) & 1));
                if (lane == j) T->rowmask[j][k] = b;
            }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(barw(c, B_TAB_FULL + ts));
        e0 = e1;
        e1 = e2;
        e2 = e3;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            pg1[k] = pg2[k];
            r0[k] = r1[k];
            s0[k] = s1[k];
        }
    }
    return true;
}

__device__ void producer_w(const CtxW& c0, int lane, int p) {
    CtxW c = c0;
    int t0 = 0;
    for (int w = next_item(c, (int)blockIdx.x - (int)gridDim.x); w < c.n_items; w = next_item(c, w)) {
        {   // the softmax writes the next item's Q rows when this one ends: pull them into L2
            CtxW cn = c;
            const int wn = next_item(cn, w);
            if (p == 0 && wn < cn.n_items) {
                const uint8_t* qrow = reinterpret_cast<const uint8_t*>(cn.a->q) +
                                      ((size_t)cn.q_begin * cn.n_heads + (size_t)cn.h * kHeadsPerKv) * (kHeadDim * 2);
                for (int e = lane; e < cn.nj * kHeadsPerKv * 2; e += 32) {
                    const int j = e / (2 * kHeadsPerKv), rem = e - j * 2 * kHeadsPerKv;
                    prefetch_l2w(qrow + (size_t)j * cn.n_heads * kHeadDim * 2 + (size_t)rem * 128);
                }
            }
        }
        if (!producer_item(c, lane, t0, p)) return;
        t0 += c.n_chunks;
    }
}

// ------------------------------------------------------------------ loaders / converters
// Two groups of four loader warps, one for K and one for V, each running ahead
// on its own: the K group is held back only by S (a K tile is free once S has
// read it), the V group only by P V.  A group copies its part of a chunk's INT8
// rows into a staging slot with bulk copies (the async proxy; completion counted
// in bytes on the slot's mbarrier) two chunks ahead, so no thread waits on a
// global load, then converts the staged rows to a BF16 operand tile.
constexpr int kGroupThreads = kLoadThreads / 2;          // 128 per part
constexpr int kRowsW = kCW * 8 / kGroupThreads;          // rows per thread per tile: 8

// Staging of part `pt` (0: K, 1: V) of chunk i into slot i % kNStage.  Group
// thread lt covers row lt.  A half-chunk that is one whole resident page is one
// 8 KB bulk copy (by the thread of its first row); otherwise each resident row is
// a 128-byte copy.  Each warp then arrives once on the slot's FULL barrier
// (after its lanes announced their bytes).
__device__ __forceinline__ bool issue_copies(const CtxW& c, int lt, int pt, int i) {
    const int st = i % kNStage;
    if (!waitw(c, barw(c, B_TAB_FULL + i % kNSW), (i / kNSW) & 1)) return false;
    const TabW* T = tab(c, i % kNSW);
    const int hh = lt / kPage;
    const int8_t* pool = pt == 0 ? c.a->k_pool : c.a->v_pool;
    const uint32_t part = c.base_u + kOffStage + st * kStageBytes + pt * (kCW * kHeadDim);
    const uint32_t full = barw(c, B_ST_FULL + pt * kNStage + st);
    const int pr = T->page_row[hh];
    if (pr >= 0) {
        if ((lt & (kPage - 1)) == 0) {
            tc::mbar_expect_tx(full, kPage * kHeadDim);
            tc::bulk_g2s(part + lt * kHeadDim, pool + (size_t)pr * kHeadDim, kPage * kHeadDim, full);
        }
    } else {
        const int r = T->row[lt];
        if (r >= 0) {
            tc::mbar_expect_tx(full, kHeadDim);
            tc::bulk_g2s(part + lt * kHeadDim, pool + (size_t)r * kHeadDim, kHeadDim, full);
        }
    }
    __syncwarp();
    if ((lt & 31) == 0) tc::mbar_arrive(full);
    return true;
}

// Which 16 bytes group thread lt handles in each of its rows: row
// row0(lt) + 16k, bytes [16i, 16i+16) with i = col16(lt).  A 16-byte shared
// access is served 8 lanes at a time; the 8 lanes of each such phase take two
// adjacent rows (an even and an odd one) and opposite 64-byte halves of them,
// so the staging reads (unswizzled 128-byte rows) hit 32 distinct banks, and the
// BF16 stores -- the even row's into the even 16-byte slots of its swizzled
// 128-byte row, the odd row's into the odd ones -- do too.
__device__ __forceinline__ int row0(int lt) { return 4 * (lt >> 5) + 2 * ((lt >> 4) & 1) + ((lt >> 2) & 1); }
__device__ __forceinline__ int col16(int lt) { return 4 * (((lt >> 3) & 1) ^ ((lt >> 2) & 1)) + (lt & 3); }

__device__ __forceinline__ void read_stage(const uint8_t* part, int lt, uint4 (&x)[kRowsW]) {
#pragma unroll
    for (int k = 0; k < kRowsW; ++k) {
        const int row = row0(lt) + (kGroupThreads / 8) * k;
        x[k] = *reinterpret_cast<const uint4*>(part + row * kHeadDim + 16 * col16(lt));
    }
}

// The 16 INT8 values of row row0 + 16k, columns 16i..16i+15, as BF16 into the
// 128-byte-swizzled tile (zeros for a masked cell): two 16-byte stores into
// half i >> 2.
__device__ __forceinline__ void store_row16(uint8_t* tile, int lt, int k, uint4 x, bool present) {
    const int i = col16(lt), row = row0(lt) + (kGroupThreads / 8) * k;
    if (!present) x = make_uint4(0, 0, 0, 0);
    uint4 lo, hi;
    int8x4_to_bf16(x.x, lo.x, lo.y);
    int8x4_to_bf16(x.y, lo.z, lo.w);
    int8x4_to_bf16(x.z, hi.x, hi.y);
    int8x4_to_bf16(x.w, hi.z, hi.w);
    uint8_t* half = tile + (i >> 2) * kHalfW + row * 128;
    const uint32_t c0 = 2u * (uint32_t)(i & 3);
    *reinterpret_cast<uint4*>(half + ((c0 ^ (row & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ (row & 7)) << 4)) = hi;
}

// Chunks of all of this CTA's items.
__device__ __forceinline__ int total_chunks(const CtxW& c0) {
    CtxW c = c0;
    int n = 0;
    for (int w = next_item(c, (int)blockIdx.x - (int)gridDim.x); w < c.n_items; w = next_item(c, w)) n += c.n_chunks;
    return n;
}

// Loader group `pt` (0: K, 1: V), thread lt of 128.
__device__ void loader_w(const CtxW& c, int pt, int lt) {
    const int n = total_chunks(c);
    if (n == 0) return;
    const int b_full = pt == 0 ? B_K_FULL : B_V_FULL, b_empty = pt == 0 ? B_K_EMPTY : B_V_EMPTY;
    uint8_t* tiles = c.base + (pt == 0 ? kOffK : kOffV);
    int issued = 0, consumed = 0;   // chunks whose copies were issued / have landed
    bool ok = true;
    for (; issued < n && issued < kNStage && ok; ++issued) ok = issue_copies(c, lt, pt, issued);
#pragma unroll 1
    for (int i = 0; i < n && ok; ++i) {
        const int st = i % kNStage, ts = i % kNSW, b = i % kNBW;
        if (!(ok = waitw(c, barw(c, B_ST_FULL + pt * kNStage + st), (i / kNStage) & 1))) break;
        consumed = i + 1;
        uint4 x[kRowsW];
        read_stage(c.base + kOffStage + st * kStageBytes + pt * (kCW * kHeadDim), lt, x);
        __syncwarp();
        if ((lt & 31) == 0) tc::mbar_arrive(barw(c, B_ST_EMPTY + pt * kNStage + st));   // done with the slot
        if (issued < n) {   // issued == i + kNStage: refill the slot once the group's warps have read it
            if (!(ok = waitw(c, barw(c, B_ST_EMPTY + pt * kNStage + st), (i / kNStage) & 1))) break;
            tc::fence_proxy_async();
            if (!(ok = issue_copies(c, lt, pt, issued))) break;
            ++issued;
        }
        const TabW* T = tab(c, ts);
        if (!(ok = waitw(c, barw(c, b_empty + b), ((i / kNBW) & 1) ^ 1))) break;
        uint8_t* tile = tiles + b * kTileW;
#pragma unroll
        for (int k = 0; k < kRowsW; ++k)
            store_row16(tile, lt, k, x[k], T->row[row0(lt) + (kGroupThreads / 8) * k] >= 0);
        tc::fence_proxy_async();
        __syncwarp();
        if ((lt & 31) == 0) {
            tc::mbar_arrive(barw(c, b_full + b));
            tc::mbar_arrive(barw(c, B_TAB_EMPTY + ts));
        }
    }
    // after a failed wait: copies still in flight land before the CTA exits (bounded)
    for (int j = consumed; !ok && j < issued; ++j)
        if (!tc::mbar_wait_drain(barw(c, B_ST_FULL + pt * kNStage + j % kNStage), (j / kNStage) & 1, kWaitNsW)) break;
}

// ------------------------------------------------------------------ MMA issuers
// Two issuing threads, so that neither kind of MMA waits behind the other's
// dependencies (an issuing thread blocks while the tensor core's queue is full):
//   warp 7 lane 0   S(t) = Q K^T into S buffer t & 1, once K(t) is converted and
//                   P(t-2) V -- the last reader of that buffer -- has completed;
//   warp 23 lane 0  O += P(t) V once P(t) and V(t) are ready.
// Completion of P V is signalled per S buffer (PV_DONE[t & 1]), so that a wait
// for P(t-2) V can never be satisfied by a later phase.

__device__ void mma_s(const CtxW& c0) {
    constexpr uint32_t idS = tc::idesc_bf16(128, kCW, false, false);   // A = Q (TMEM), B = K tile, K-major
    CtxW c = c0;
    int t0 = 0, kk = 0;
    bool ok = true;
    for (int w = next_item(c, (int)blockIdx.x - (int)gridDim.x); w < c.n_items && ok; w = next_item(c, w), ++kk) {
        for (int i = 0; i < c.n_chunks && ok; ++i) {
            const int t = t0 + i, b = t % kNBW;
            if (i == 0 && !(ok = waitw(c, barw(c, B_Q_READY), kk & 1))) break;   // the item's Q rows
            if (!(ok = waitw(c, barw(c, B_K_FULL + b), (t / kNBW) & 1))) break;
            if (t >= 2 && !(ok = waitw(c, barw(c, B_PV_DONE + (t & 1)), ((t - 2) >> 1) & 1))) break;
            tc::fence_after_sync();
            const uint32_t kt = c.base_u + kOffK + b * kTileW;
            const uint32_t tS = c.tmem + kColS + 128 * (t & 1);
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k) {
                const uint32_t koff = (k >> 2) * kHalfW + (k & 3) * 32;
                tc::mma_ts(tS, c.tmem + kColQ + 8 * k, tc::smem_desc(kt + koff, 16, 1024, 2), idS, k > 0 ? 1u : 0u);
            }
            tc::commit(barw(c, B_S_FULL + (t & 1)));
            tc::commit(barw(c, B_K_EMPTY + b));
        }
        t0 += c.n_chunks;
    }
    tc::commit(barw(c, B_DRAIN));
    if (!tc::mbar_wait_drain(barw(c, B_DRAIN), 0, kWaitNsW)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

__device__ void mma_pv(const CtxW& c0) {
    constexpr uint32_t idO = tc::idesc_bf16(128, kHeadDim, false, true);   // A = P (TMEM), B = V tile, MN-major
    CtxW c = c0;
    int t0 = 0, kk = 0;
    bool ok = true;
    for (int w = next_item(c, (int)blockIdx.x - (int)gridDim.x); w < c.n_items && ok; w = next_item(c, w), ++kk) {
        for (int i = 0; i < c.n_chunks && ok; ++i) {
            const int t = t0 + i, b = t % kNBW;
            const bool first = i == 0;
            if (!(ok = waitw(c, barw(c, B_P_READY + (t & 1)), (t >> 1) & 1))) break;
            if (!(ok = waitw(c, barw(c, B_V_FULL + b), (t / kNBW) & 1))) break;
            // an item's first P V overwrites O: the softmax must have read the previous item's O
            if (first && kk > 0 && !(ok = waitw(c, barw(c, B_O_FREE), (kk - 1) & 1))) break;
            tc::fence_after_sync();
            const uint32_t vt = c.base_u + kOffV + b * kTileW;
            const uint32_t tP = c.tmem + kColS + 128 * (t & 1);
            const uint32_t tO = c.tmem + kColO;
#pragma unroll
            for (int k = 0; k < kCW / 16; ++k)   // P of cells 16k..16k+15: columns 32(k>>1) + 8(k&1)
                tc::mma_ts(tO, tP + 8 * (k & 1) + 32 * (k >> 1), tc::smem_desc(vt + k * 2048, kHalfW, 1024, 2), idO,
                           (!first || k > 0) ? 1u : 0u);
            tc::commit(barw(c, B_PV_DONE + (t & 1)));
            tc::commit(barw(c, B_V_EMPTY + b));
            if (i == c.n_chunks - 1) tc::commit(barw(c, B_O_DONE));
        }
        t0 += c.n_chunks;
    }
    tc::commit(barw(c, B_DRAIN_PV));
    if (!tc::mbar_wait_drain(barw(c, B_DRAIN_PV), 0, kWaitNsW)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ softmax
// Scale + mask 16 score columns (see attn_tc.cu): v = s * ks where selected,
// -inf elsewhere; `uniform`: the warp's queries selected all of the slice or
// none of it, so the mask is a per-lane bias in the same FMA.
__device__ __forceinline__ void scale_mask16w(uint32_t* s, uint32_t sel, bool uniform, const float* ks, float& mx,
                                              float& my) {
    if (uniform) {
        const float bias = sel ? 0.f : -INFINITY;
        const float2 b2 = make_float2(bias, bias);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            const float4 kq = *reinterpret_cast<const float4*>(ks + 4 * c4);
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(s[4 * c4]), __uint_as_float(s[4 * c4 + 1])),
                                        make_float2(kq.x, kq.y), b2);
            const float2 b = __ffma2_rn(make_float2(__uint_as_float(s[4 * c4 + 2]), __uint_as_float(s[4 * c4 + 3])),
                                        make_float2(kq.z, kq.w), b2);
            s[4 * c4] = __float_as_uint(a.x);
            s[4 * c4 + 1] = __float_as_uint(a.y);
            s[4 * c4 + 2] = __float_as_uint(b.x);
            s[4 * c4 + 3] = __float_as_uint(b.y);
            mx = fmax3(mx, a.x, a.y);
            my = fmax3(my, b.x, b.y);
        }
        return;
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        const float4 kq = *reinterpret_cast<const float4*>(ks + 4 * c4);
        const float2 a = __fmul2_rn(make_float2(__uint_as_float(s[4 * c4]), __uint_as_float(s[4 * c4 + 1])),
                                    make_float2(kq.x, kq.y));
        const float2 b = __fmul2_rn(make_float2(__uint_as_float(s[4 * c4 + 2]), __uint_as_float(s[4 * c4 + 3])),
                                    make_float2(kq.z, kq.w));
        const float v0 = ((sel >> (4 * c4)) & 1u) ? a.x : -INFINITY;
        const float v1 = ((sel >> (4 * c4 + 1)) & 1u) ? a.y : -INFINITY;
        const float v2 = ((sel >> (4 * c4 + 2)) & 1u) ? b.x : -INFINITY;
        const float v3 = ((sel >> (4 * c4 + 3)) & 1u) ? b.y : -INFINITY;
        s[4 * c4] = __float_as_uint(v0);
        s[4 * c4 + 1] = __float_as_uint(v1);
        s[4 * c4 + 2] = __float_as_uint(v2);
        s[4 * c4 + 3] = __float_as_uint(v3);
        mx = fmax3(mx, v0, v1);
        my = fmax3(my, v2, v3);
    }
}

// p = 2^(v - m) for 16 columns, summed into la / lb; p * (V scale) out as 8
// packed BF16 pairs.
__device__ __forceinline__ void exp16w(const uint32_t* s, const float* vs, float2 nm, uint32_t* p, float2& la,
                                       float2& lb) {
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) {
        const float4 vq = *reinterpret_cast<const float4*>(vs + 4 * u4);
        const float2 x01 = __fadd2_rn(make_float2(__uint_as_float(s[4 * u4]), __uint_as_float(s[4 * u4 + 1])), nm);
        const float2 x23 = __fadd2_rn(make_float2(__uint_as_float(s[4 * u4 + 2]), __uint_as_float(s[4 * u4 + 3])), nm);
        const float2 e01 = make_float2(fast_exp2(x01.x), fast_exp2(x01.y));
        const float2 e23 = make_float2(fast_exp2(x23.x), fast_exp2(x23.y));
        la = __fadd2_rn(la, e01);
        lb = __fadd2_rn(lb, e23);
        const float2 w01 = __fmul2_rn(e01, make_float2(vq.x, vq.y));
        const float2 w23 = __fmul2_rn(e23, make_float2(vq.z, vq.w));
        p[2 * u4] = pack_bf16x2(w01.x, w01.y);
        p[2 * u4 + 1] = pack_bf16x2(w23.x, w23.y);
    }
}

__device__ __forceinline__ size_t row_offset(const CtxW& c, int r) {
    const int j = r / kHeadsPerKv, hq = r - j * kHeadsPerKv;
    return ((size_t)(c.q_begin + j) * c.n_heads + (size_t)c.h * kHeadsPerKv + hq) * kHeadDim;
}

// Q row r of the item in c, elements [32q, 32q+32) -> TMEM lane r, columns
// kColQ + 16q .. +16 (packed BF16 pairs; rows of absent ragged queries are zero);
// then arrive on Q_READY.
__device__ __forceinline__ void write_q_w(const CtxW& c, int q, int quad, int r, int lane) {
    const bool row_ok = r / kHeadsPerKv < c.nj;
    const uint4* src = reinterpret_cast<const uint4*>(c.a->q + row_offset(c, r) + 32 * q);
    uint32_t v[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 x = row_ok ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
        v[4 * k] = x.x;
        v[4 * k + 1] = x.y;
        v[4 * k + 2] = x.z;
        v[4 * k + 3] = x.w;
    }
    tc::tmem_st16(c.tmem + ((uint32_t)(32 * quad) << 16) + kColQ + 16 * q, v);
    tc::tmem_wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(barw(c, B_Q_READY));
}

// Zero this warp's 32 output columns of row r for every item without chunks
// between w (exclusive) and the next item that has some.
__device__ __forceinline__ void zero_empty_items(const CtxW& c0, int w, int q, int r) {
    CtxW c = c0;
    for (w += gridDim.x; w < c.n_items; w += gridDim.x) {
        set_item(c, w);
        if (c.n_chunks > 0) return;
        if (r / kHeadsPerKv < c.nj) {
            float4* out = reinterpret_cast<float4*>(c.a->out + row_offset(c, r) + 32 * q);
            for (int v = 0; v < 8; ++v) out[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

__device__ void softmax_w(const CtxW& c0, int q, int quad, int lane) {
    CtxW c = c0;
    const int r = 32 * quad + lane;
    const int j = r / kHeadsPerKv;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    float* xchg = reinterpret_cast<float*>(c.base + kOffX);
    const float thresh = kRescaleLog2W;
    zero_empty_items(c, (int)blockIdx.x - (int)gridDim.x, q, r);
    int w = next_item(c, (int)blockIdx.x - (int)gridDim.x);
    if (w < c.n_items) write_q_w(c, q, quad, r, lane);
    int t0 = 0, kk = 0;
    uint32_t nsync = 0;
    bool ok = true;
    while (w < c.n_items) {
        float m = -INFINITY, l = 0.f;
        for (int i = 0; i < c.n_chunks; ++i) {
            const int t = t0 + i, sb = t & 1, ts = t % kNSW;
            const uint32_t tS = c.tmem + lane_base + kColS + 128 * sb + 32 * q;
            if (!(ok = waitw(c, barw(c, B_TAB_FULL + ts), (t / kNSW) & 1))) break;
            const TabW* T = tab(c, ts);
            const uint32_t sel = T->rowmask[j][q];
            if (!(ok = waitw(c, barw(c, B_S_FULL + sb), (t >> 1) & 1))) break;
            tc::fence_after_sync();
            uint32_t sv[32];
            tc::tmem_ld32(tS, sv);
            const uint32_t sel_lo = sel & 0xFFFFu, sel_hi = sel >> 16;
            const bool act_lo = __any_sync(0xffffffffu, sel_lo != 0), act_hi = __any_sync(0xffffffffu, sel_hi != 0);
            const bool uni_lo = __all_sync(0xffffffffu, sel_lo == 0 || sel_lo == 0xFFFFu);
            const bool uni_hi = __all_sync(0xffffffffu, sel_hi == 0 || sel_hi == 0xFFFFu);
            const float* ksp = &T->ks[32 * q];
            tc::tmem_wait_ld();
            float mx = -INFINITY, my = -INFINITY;
            if (act_lo) scale_mask16w(&sv[0], sel_lo, uni_lo, ksp, mx, my);
            if (act_hi) scale_mask16w(&sv[16], sel_hi, uni_hi, ksp + 16, mx, my);
            // swap quarter maxima with the quadrant's other warps, so all four take the same step
            float* xb = xchg + (t & 1) * (kQuarters * kRows);
            xb[q * kRows + r] = fmaxf(mx, my);
            if (!(ok = quad_sync(c, quad, nsync++))) break;
            const float m_new =
                fmax3(fmax3(m, xb[r], xb[kRows + r]), xb[2 * kRows + r], xb[3 * kRows + r]);
            const bool need = (m != -INFINITY) && (m_new > m + thresh);
            const float m_use = (m == -INFINITY || need) ? m_new : m;
            const float alpha = need ? fast_exp2(m - m_new) : 1.f;
            const float m_sub = m_use == -INFINITY ? 0.f : m_use;
            uint32_t p[16];
            const float2 nm = make_float2(-m_sub, -m_sub);
            float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
            const float* vsp = &T->vs[32 * q];
            if (act_lo) {
                exp16w(&sv[0], vsp, nm, &p[0], la, lb);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) p[v] = 0u;
            }
            if (act_hi) {
                exp16w(&sv[16], vsp + 16, nm, &p[8], la, lb);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) p[8 + v] = 0u;
            }
            l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
            m = m_use;
            tc::tmem_st16(tS, p);
            if (__any_sync(0xffffffffu, need)) {
                // O must hold every earlier P V before it is rescaled: wait for PV(t-1);
                // this warp rescales its 32 of O's columns
                if (!(ok = waitw(c, barw(c, B_PV_DONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1))) break;
                tc::fence_after_sync();
#pragma unroll 1
                for (int h16 = 0; h16 < 2; ++h16) {
                    uint32_t o[16];
                    const uint32_t ta = c.tmem + lane_base + kColO + 32 * q + 16 * h16;
                    tc::tmem_ld16(ta, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 16; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
                    tc::tmem_st16(ta, o);
                }
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(barw(c, B_P_READY + sb));
                tc::mbar_arrive(barw(c, B_TAB_EMPTY + ts));
            }
        }
        if (!ok) break;
        float4* out = reinterpret_cast<float4*>(c.a->out + row_offset(c, r) + 32 * q);
        const bool row_ok = j < c.nj;
        t0 += c.n_chunks;
        // the item's last S has completed (its chunk was read above): the next
        // item's Q rows can replace this item's
        zero_empty_items(c, w, q, r);
        w = next_item(c, w);   // c holds the next item from here on
        if (w < c.n_items) write_q_w(c, q, quad, r, lane);
        // total weight of the row over the quadrant's four warps
        float* xl = xchg + 2 * kQuarters * kRows;
        xl[q * kRows + r] = l;
        if (!(ok = quad_sync(c, quad, nsync++))) break;
        const float l_tot = (xl[r] + xl[kRows + r]) + (xl[2 * kRows + r] + xl[3 * kRows + r]);
        if (!(ok = waitw(c, barw(c, B_O_DONE), kk & 1))) break;
        tc::fence_after_sync();
        uint32_t o[32];
        tc::tmem_ld32(c.tmem + lane_base + kColO + 32 * q, o);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(barw(c, B_O_FREE));   // O may be overwritten
        const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
        if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
                out[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                     __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
        ++kk;
    }
}

__global__ void __launch_bounds__(kThreadsW, 1) attn_wide_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u = smem_u32(smem_raw);
    const uint32_t base_u = (raw_u + 1023u) & ~1023u;
    CtxW c;
    c.a = &a;
    c.base = smem_raw + (base_u - raw_u);
    c.base_u = base_u;
    c.abort_flag = reinterpret_cast<volatile int*>(c.base + kOffMiscW + 4);
    c.n_heads = a.n_kv * kHeadsPerKv;
    c.n_items = ((a.n_q + kGroup - 1) / kGroup) * a.n_kv;
    c.kmul = a.sm_scale * kLog2e;
    c.g = c.h = c.nj = c.q_begin = c.U = c.n_chunks = 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(c.base + kOffMiscW);
    if (tid == 0) {
        for (int s = 0; s < kNSW; ++s) {
            tc::mbar_init(barw(c, B_TAB_FULL + s), 1);
            tc::mbar_init(barw(c, B_TAB_EMPTY + s), kLoadW + kSoftW);
        }
        for (int b = 0; b < kNBW; ++b) {
            tc::mbar_init(barw(c, B_K_FULL + b), kLoadW / 2);
            tc::mbar_init(barw(c, B_K_EMPTY + b), 1);
            tc::mbar_init(barw(c, B_V_FULL + b), kLoadW / 2);
            tc::mbar_init(barw(c, B_V_EMPTY + b), 1);
        }
        for (int sb = 0; sb < 2; ++sb) {
            tc::mbar_init(barw(c, B_S_FULL + sb), 1);
            tc::mbar_init(barw(c, B_P_READY + sb), kSoftW);
        }
        tc::mbar_init(barw(c, B_PV_DONE), 1);
        tc::mbar_init(barw(c, B_PV_DONE + 1), 1);
        tc::mbar_init(barw(c, B_DRAIN_PV), 1);
        tc::mbar_init(barw(c, B_O_DONE), 1);
        tc::mbar_init(barw(c, B_O_FREE), kSoftW);
        tc::mbar_init(barw(c, B_Q_READY), kSoftW);
        tc::mbar_init(barw(c, B_DRAIN), 1);
        for (int qd = 0; qd < 3; ++qd) tc::mbar_init(barw(c, B_QUAD + qd), kQuarters);
        for (int st = 0; st < 2 * kNStage; ++st) {
            tc::mbar_init(barw(c, B_ST_FULL + st), kLoadW / 2);
            tc::mbar_init(barw(c, B_ST_EMPTY + st), kLoadW / 2);
        }
        *c.abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kWarpMmaW) {
        tc::tmem_alloc(smem_u32(tmem_holder), kTmemColsW);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    c.tmem = *tmem_holder;

    if (warp == kWarpProd || warp == kWarpProd2) {
        producer_w(c, lane, warp == kWarpProd ? 0 : 1);
    } else if (warp == kWarpMmaW) {
        if (lane == 0) mma_s(c);
    } else if (warp == kWarpPvW) {
        if (lane == 0) mma_pv(c);
    } else if (warp < 16 && (warp & 3) != 3) {
        softmax_w(c, warp >> 2, warp & 3, lane);
    } else {
        const int li = warp == 11 ? 0 : warp == 15 ? 1 : warp - 14;   // warps 11, 15, 16-21
        loader_w(c, li >> 2, (li & 3) * 32 + lane);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMmaW) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemColsW);
    }
}

}  // namespace

cudaError_t launch_attn_wide(const AttnArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemW);
    if (e != cudaSuccess) return e;
    const long long items = (long long)((a.n_q + kGroup - 1) / kGroup) * a.n_kv;
    const int grid = (int)(items < sms ? items : sms);
    if (grid <= 0) return cudaSuccess;
    attn_wide_kernel<<<grid, kThreadsW, kSmemW, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
