// attn_sm.cu -- union attention with one CTA per SM: Q, an O per softmax set
// and three S/P buffers in Tensor Memory, two softmax warp sets on alternating
// chunks, each with its own running max, combined at the end; and
// the same kernel with the group's union built inside the CTA (the fused path,
// no union arrays in global memory and no first launch).
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary: one work-group per (8 positions, KV head) covers
// the 96 rows of 8 positions x 12 heads; the sorted union of the 8 positions'
// selections, each cell marked by the positions that chose it, is processed in
// 64-cell chunks whose INT8 K/V are dequantised once; S = Q K^T and O += P V run
// on the matrix units with FP32 sums; in the online softmax a cell is -inf for
// every position that did not select it.  Section What changed: the union
// kernel and the attention kernel run as a launch pair.  Section Extra Notes:
// non-resident pages are masked.
//
// One CTA per (group g, KV head h) on its own SM: 96 query-head rows (row r =
// j*12 + hq, TMEM lane r).  The CTA owns all 512 TMEM columns: Q [0,64) as FP16
// pairs (the A operand of S), set 0's O [64,192), set 1's O [192,320), and three
// S/P buffers of 64 columns from 320, so S can run up to two chunks ahead of the
// softmax.  Warp roles:
//   softmax, two sets of six: set s (warps 8s + {0,1,2,4,5,6}) takes the chunks
//              t with t % 2 == s.  Within a set, warps 8s+q and 8s+q+4 own the
//              32 rows of TMEM lane quadrant q and columns [0,32) / [32,64) of
//              the chunk and swap half-chunk maxima (a 64-thread named
//              barrier).  A warp reads its 32 S columns, scales each by its K
//              scale and masks cells its query did not select.  Each set keeps
//              its own running max m (it only moves when a weight would exceed
//              2^12: lazy rescale), its own O (P(t) V accumulates into the O of
//              the set that took chunk t) and per warp its FP32 sum of p, so
//              the sets never wait for each other.  A warp writes P = p * (V
//              scale) as FP16 over its own S columns.  At the end the four warps
//              of a quadrant take M = max(m_0, m_1), weigh each set's sums and O
//              by 2^(m_s - M), and each stores 32 of the output's columns.  Set 0
//              writes Q into TMEM first.
//   warps 3, 22 producers (even / odd chunks): union entries -> page table ->
//              per-chunk tables in a 16-deep ring (pool row of each cell, K scale
//              times sm_scale * log2(e), V scale divided by a power of two per
//              chunk, one 64-bit selection mask per query built with warp
//              ballots), three of its chunks of loads in flight each, and an L2
//              prefetch of each chunk's K/V rows.  After the last chunk each
//              writes one end-of-stream table.
//   warps 7, 23 MMA issuers (the whole warp runs the loop; one elected lane
//              issues): warp 7 S(t) = Q K^T (A = Q from TMEM, B = K tile, M=128
//              N=64 K=128) into S buffer t % 3, warp 23 O += P(t) V (A = P from
//              TMEM, B = V tile, M=128 N=128 K=64) into the O of chunk t's set, all
//              operands FP16.
//   warps 16-19 K loaders, warps 11, 15, 20, 21 V loaders: one 16-byte load per
//              row and thread of the chunk's INT8 rows, issued two chunks ahead
//              into registers, converted exactly to FP16 straight into operand
//              tiles in the 128-byte swizzled layouts the tensor core reads.
// Fused path: before the pipeline starts, the whole CTA builds the group's
//              union into shared memory with the union kernel's own build
//              (union_core.cuh: a byte map per window of cells, marking, a page
//              scan and an ordered compaction), the byte map in the K/V tile
//              area and its small arrays in the table ring, not yet in use; the
//              producers then read the union from there in place of the union
//              arrays.
// The chunk placement, the tables and every product are the same in both
// paths, so the fused path's output equals the launch pair's bit for bit.
// Precision.  K and V enter the products exactly; the K scale multiplies the
// score column in FP32.  P = e * vs' is rounded to FP16 once, where vs' = V
// scale * 2^-ev for the chunk's exponent ev (its largest |V scale| in [1, 2));
// the weight's exponent carries ev back (x = s * ks + ev), so any FP16 scale
// keeps P inside FP16's range, and the row sum adds each chunk's weights times
// 2^-ev.  Masking comes after all scaling.  Rows 96-127 of the M=128 tiles are
// padding (never read back).
// Every wait is bounded in time; a wait that runs out sets a CTA-wide abort
// flag and QSA_DEV_WAIT_TIMEOUT, every role then stops, the MMA issuers drain
// the MMAs they started, and the CTA frees its Tensor Memory and exits.
#include "qsa_common.cuh"
#include "tc_ptx.cuh"
#include "union_core.cuh"

namespace qsa {
namespace {

constexpr int kWarpProducer0 = 3, kWarpProducer1 = 22;   // even / odd chunks
constexpr int kWarpMmaS = 7, kWarpMmaPV = 23;             // S issuer, P V issuer
constexpr int kLoadThreads = 128;            // per loader group (K or V)
constexpr int kSetWarps = 6;                 // softmax warps per set
constexpr int kNS = 16;                      // per-chunk table ring
constexpr int kNSb = 3;                      // S/P buffers in TMEM
constexpr int kNK = 3;                       // K tiles
constexpr int kNV = 3;                       // V tiles
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColO = 64, kColS = 320;   // O of set s at kColO + 128 s; S buffer b at kColS + 64 b
// Lazy rescale threshold (exp2 domain): the running max only moves, and O is
// only rescaled, when a weight exceeds it by more than 2^12.  P = e * vs' then
// stays below 2^13, inside FP16, and FP16 / FP32 rounding is relative, so a
// stale max costs no accuracy.
constexpr float kRescaleLog2 = 12.f;
constexpr uint64_t kWaitNs = 1000000000ull;

constexpr int kWarps = 24;

__device__ __forceinline__ int k_loader_index(int warp) { return warp - 16; }   // warps 16-19
__device__ __forceinline__ int v_loader_index(int warp) {                      // warps 20, 21, 11, 15
    return warp >= 20 ? warp - 20 : (warp == 11 ? 2 : 3);
}

struct RawTab {
    int32_t row[kChunk];           // pool row (page * n_kv + h) * 64 + cell % 64; -1 for a masked cell
    float ks[kChunk];              // K scale * sm_scale * log2(e); 0 for a masked cell
    float vs[kChunk];              // V scale * 2^-ev; 0 for a masked cell
    uint64_t rowmask[8];           // bit c: query j of the group selected resident cell c
    float vshift;                  // ev
    float vinv;                    // 2^-ev
    int32_t end;                   // 1: no chunk here; the stream ended before it
    int32_t pad;
};

constexpr uint32_t kTileBytes = kChunk * kHeadDim * 2;   // 16 KB FP16 K or V tile (two 64-column halves)
constexpr uint32_t kOffKb = 0;
constexpr uint32_t kOffVb = kOffKb + kNK * kTileBytes;
constexpr uint32_t kOffRawTab = kOffVb + kNV * kTileBytes;
// Shared scalars per row: half-chunk maxima swapped within a set, by set and
// chunk parity [2][2][2][96]; each set's final running max [2][96]; the row sums
// at the end [4][96]; the Q row scale [96].
constexpr uint32_t kOffXchg = kOffRawTab + kNS * (uint32_t)sizeof(RawTab);
constexpr uint32_t kOffMslot = kOffXchg + 8 * kRows * 4;
constexpr uint32_t kOffLsum = kOffMslot + 2 * kRows * 4;
constexpr uint32_t kOffRs = kOffLsum + 4 * kRows * 4;
constexpr uint32_t kOffBars = (kOffRs + kRows * 4 + 7u) & ~7u;
// K_EMPTY[b]: S(t) with t % kNK == b has read K tile b.  S_FULL[b]: S(t), t % 3
// == b, is in S buffer b.  P_READY[b]: P(t) is in S buffer b (or, at t = the
// chunk count, the stream has ended).  V_EMPTY[b]: P(t) V with t % kNV == b
// has completed (V tile b free).  PV_DONE[b]: P(t) V with t % 3 == b has
// completed.  Before it rescales its set's O, the softmax warp of chunk t waits
// on it for P(t-2) V, the set's previous chunk (P V runs in chunk order, so
// every earlier P V into that O is complete too).  The slot cannot be a phase
// further on: P(t+1) V follows P(t) V, which needs this warp's P(t).  And its
// previous phase (P(t-5) V) is complete: the warp has seen S(t) complete, issued
// after P(t-3) V had completed.
enum { BAR_TAB_FULL = 0, BAR_TAB_EMPTY = kNS, BAR_K_FULL = 2 * kNS, BAR_K_EMPTY = BAR_K_FULL + kNK,
       BAR_V_FULL = BAR_K_EMPTY + kNK, BAR_V_EMPTY = BAR_V_FULL + kNV, BAR_S_FULL = BAR_V_EMPTY + kNV,
       BAR_P_READY = BAR_S_FULL + kNSb, BAR_PV_DONE = BAR_P_READY + kNSb, BAR_O_DONE = BAR_PV_DONE + kNSb,
       BAR_Q_READY, BAR_DRAIN_S, BAR_DRAIN_PV, NUM_BARS };
constexpr uint32_t kOffMisc = kOffBars + NUM_BARS * 8;      // tmem base, abort flag, chunk count
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;           // + alignment slack
// The fused path keeps its group's union after that: cells (int32) then masks (uint8).
constexpr uint32_t kOffUnion = (kSmemUsed + 15u) & ~15u;
// While the union is built (before any tile or table is used), the byte map of
// its window sits in the K/V tile area and its small arrays in the table ring.
static_assert(kNK * kTileBytes + kNV * kTileBytes >= (uint32_t)kUnionWindow, "byte map fits the tile area");
constexpr uint32_t kUnionSmallBytes = kUnionPages + 2 * kUnionPages + 5 * kGroup * 4 + kWarps * 4;
static_assert(kNS * sizeof(RawTab) >= kUnionSmallBytes, "union scratch fits the table ring");
__host__ __device__ constexpr uint32_t fused_union_capacity(int sel_stride) {
    return ((uint32_t)kGroup * (uint32_t)sel_stride + 15u) & ~15u;
}

struct Ctx {
    const AttnArgs* a;
    uint8_t* base;
    uint32_t base_u;
    uint32_t tmem;
    volatile int* abort_flag;
    volatile int* n_final;   // the chunk count
    const int32_t* ucell;    // the group's union: cells and masks (global memory, or shared on the fused path)
    const uint8_t* umask;
    int g, h, nj, q_begin, n_heads, U, n_chunks;
    float kmul;
};

__device__ __forceinline__ uint32_t bar(const Ctx& c, int i) { return c.base_u + kOffBars + 8u * i; }
__device__ __forceinline__ RawTab* raw_tab(const Ctx& c, int s) {
    return reinterpret_cast<RawTab*>(c.base + kOffRawTab) + s;
}
__device__ __forceinline__ float* smem_f(const Ctx& c, uint32_t off) { return reinterpret_cast<float*>(c.base + off); }

__device__ __forceinline__ bool wait_addr(const Ctx& c, uint32_t addr, uint32_t parity) {
    if (tc::mbar_wait(addr, parity, c.abort_flag, kWaitNs)) return true;
    report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
    return false;
}

// Named barriers (immediate ids): 1 + 3*set + quad for the two warps of a set
// that share lane quadrant quad (64 threads), 7 + quad for all four softmax
// warps of the quadrant (128 threads, once at the end).  A named barrier cannot
// time out, so after an abort a warp never waits on one: it checks the CTA's
// abort flag first and returns false, and a warp that leaves after a failed
// wait adds its share to both of its barriers with non-blocking arrives
// (leave_all).  Every warp passes its barriers in the same order as their
// other users, so a partner is then either released from the barrier it is
// waiting on or sees the flag at its next one.
template <int kCount>
__device__ __forceinline__ void named_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kCount) : "memory");
}
template <int kCount>
__device__ __forceinline__ void named_arrive(int id) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(kCount) : "memory");
}
__device__ __forceinline__ bool pair_sync(int set, int quad, bool aborted) {
    if (aborted) return false;
    named_sync<64>(1 + 3 * set + quad);
    return true;
}
__device__ __forceinline__ void leave_all(int set, int quad) {
    named_arrive<64>(1 + 3 * set + quad);
    named_arrive<128>(7 + quad);
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct Entries {
    int cell[2], mask[2];
    bool present[2];
    bool exists;   // the chunk exists (a chunk past the end does not)
};

// Chunk placement.  `lead` is the index of the first page-aligned union cell
// after entry 0 among entries 1..63 (0 if there is none).  Chunk c holds union
// positions p = lead + 64c + slot, slot = 0..63; a position past the end wraps
// to entry p - U when that is one of the `lead` entries before it, and is
// empty otherwise.  So every union entry sits in exactly one slot and the chunk
// count stays ceil(U / 64); when the union is a few loose cells (such as sink
// cells 0-2) followed by whole 64-cell pages, every chunk but the last is one
// whole page, and each query selects all of such a chunk or none of it.
__device__ __forceinline__ int union_lead(const Ctx& c, int lane, bool& ok) {
    const int U = c.U;
    const int32_t* first = c.ucell;
    ok = true;
    const uint32_t b0 = __ballot_sync(0xffffffffu, lane >= 1 && lane < U && (first[lane] & (kPage - 1)) == 0);
    if (b0) return __ffs(b0) - 1;
    const uint32_t b1 = __ballot_sync(0xffffffffu, 32 + lane < U && (first[32 + lane] & (kPage - 1)) == 0);
    return b1 ? 31 + __ffs(b1) : 0;
}

__device__ __forceinline__ Entries load_entries(const Ctx& c, int lead, int chunk, int lane, bool& ok) {
    Entries e;
    const int U = c.U;
    ok = true;
    e.exists = ok && (long long)chunk * kChunk < (long long)U;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int p = lead + chunk * kChunk + lane + 32 * k;
        const int u = p < U ? p : (p - U < lead ? p - U : -1);
        e.present[k] = e.exists && u >= 0;
        if (!e.present[k]) {
            e.cell[k] = 0;
            e.mask[k] = 0;
        } else {
            e.cell[k] = c.ucell[u];
            e.mask[k] = c.umask[u];
        }
    }
    return e;
}

// Page-table step: issues the loads only; the values are checked when used.
__device__ __forceinline__ void load_pages(const Ctx& c, const Entries& e, int (&page)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        page[k] = -1;
        if (!e.present[k]) continue;
        const int cell = e.cell[k];
        if (cell < 0 || (cell >> 6) >= c.a->n_lpages) {
            report(c.a->dev_status, QSA_DEV_BAD_CELL);
            continue;
        }
        page[k] = __ldg(c.a->page_table + (cell >> 6));    // < 0: not resident, masked
    }
}

// Pool row of each entry for the CTA's KV head (-1 = masked).
__device__ __forceinline__ void pool_rows(const Ctx& c, const Entries& e, const int (&page)[2], int (&row)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        row[k] = -1;
        if (page[k] < 0) continue;
        if (page[k] >= c.a->n_ppages) {
            report(c.a->dev_status, QSA_DEV_BAD_PAGE);
            continue;
        }
        row[k] = (page[k] * c.a->n_kv + c.h) * kPage + (e.cell[k] & (kPage - 1));
    }
}

struct Scales {
    uint16_t ks[2], vs[2];
};

__device__ __forceinline__ Scales load_scales(const Ctx& c, const int (&row)[2]) {
    Scales s;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool ok = row[k] >= 0;
        s.ks[k] = ok ? __ldg(c.a->k_scale + row[k]) : (uint16_t)0;
        s.vs[k] = ok ? __ldg(c.a->v_scale + row[k]) : (uint16_t)0;
    }
    return s;
}

// Producer p takes the chunks i = p, p + 2, ...  Each step of its loop is a
// chain of dependent loads (union entries -> page table -> scales), so two
// producers share the chunks, and each keeps three of its chunks in flight:
// entries of its chunk i+6, page table of i+4, scales of i+2, while chunk i's
// table is written.  At its first chunk past the end it writes an end-of-stream
// table instead (so the tables of chunks n and n+1 both say "end", one from
// each producer) and publishes the chunk count n.
__device__ void producer_role(const Ctx& c, int first, int lane) {
    constexpr int kStep = 2;
    bool ok = true;
    const int lead = union_lead(c, lane, ok);
    Entries e0, e1, e2;
    int pg0[2], pg1[2], r0[2];
    Scales s0;
    if (ok) {
        e0 = load_entries(c, lead, first, lane, ok);
        if (ok) e1 = load_entries(c, lead, first + kStep, lane, ok);
        if (ok) e2 = load_entries(c, lead, first + 2 * kStep, lane, ok);
    }
    if (!ok) return;
    load_pages(c, e0, pg0);
    load_pages(c, e1, pg1);
    pool_rows(c, e0, pg0, r0);
    s0 = load_scales(c, r0);
    for (int i = first;; i += kStep) {
        const int ts = i % kNS;
        const Entries e3 = load_entries(c, lead, i + 3 * kStep, lane, ok);
        if (!ok) break;
        int pg2[2], r1[2];
        load_pages(c, e2, pg2);
        pool_rows(c, e1, pg1, r1);
        const Scales s1 = load_scales(c, r1);
        // the loaders gather chunk i+2 several chunks from now: pull its rows into L2
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (r1[k] >= 0) {
                const size_t off = (size_t)r1[k] * kHeadDim;
                prefetch_l2(c.a->k_pool + off);
                prefetch_l2(c.a->v_pool + off);
            }
        // the chunk's V exponent: its largest |V scale| (FP16 magnitudes order
        // like their bit patterns), 0 when it has no resident cell
        uint32_t av = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (r0[k] >= 0) av = max(av, (uint32_t)(s0.vs[k] & 0x7FFFu));
        av = __reduce_max_sync(0xffffffffu, av);
        const int ev = av ? f32_exponent(__half2float(__ushort_as_half((uint16_t)av))) : 0;
        const float vdown = exp2i(-ev);
        if (!wait_addr(c, bar(c, BAR_TAB_EMPTY + ts), ((i / kNS) & 1) ^ 1)) break;
        RawTab* T = raw_tab(c, ts);
        if (!e0.exists) {   // the stream ended before chunk i: the chunk count is i or i - 1
            if (lane == 0) {
                T->end = 1;
                *c.n_final = (c.U + kChunk - 1) / kChunk;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(c, BAR_TAB_FULL + ts));
            break;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool okr = r0[k] >= 0;
            T->row[lane + 32 * k] = okr ? r0[k] : -1;
            T->ks[lane + 32 * k] = okr ? __half2float(__ushort_as_half(s0.ks[k])) * c.kmul : 0.f;
            T->vs[lane + 32 * k] = okr ? __half2float(__ushort_as_half(s0.vs[k])) * vdown : 0.f;
        }
        if (lane == 0) {
            T->vshift = (float)ev;
            T->vinv = vdown;
            T->end = 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t lo = __ballot_sync(0xffffffffu, r0[0] >= 0 && ((e0.mask[0] >> j) & 1));
            const uint32_t hi = __ballot_sync(0xffffffffu, r0[1] >= 0 && ((e0.mask[1] >> j) & 1));
            if (lane == j) T->rowmask[j] = (uint64_t)lo | ((uint64_t)hi << 32);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_TAB_FULL + ts));
        e0 = e1;
        e1 = e2;
        e2 = e3;
        s0 = s1;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            pg1[k] = pg2[k];
            r0[k] = r1[k];
        }
    }
}

// ------------------------------------------------------------------ loaders
// Thread ct of a loader group handles, in each of its rows row0(ct) + 16k
// (k = 0..3), the 16 bytes [16i, 16i+16) with i = col16(ct): one 16-byte load
// per row, converted to 16 FP16 values = two 16-byte stores into half i >> 2 of
// the tile.  A 16-byte shared store is served 8 lanes at a time; the 8 lanes of
// each such phase take an even and an odd row and opposite halves, so the even
// row fills the even 16-byte slots of its swizzled 128-byte row and the odd row
// the odd ones: every phase is one conflict-free wavefront.
constexpr int kRowsPerThread = kChunk * 8 / kLoadThreads;
__device__ __forceinline__ int row0(int ct) { return 4 * (ct >> 5) + 2 * ((ct >> 4) & 1) + ((ct >> 2) & 1); }
__device__ __forceinline__ int col16(int ct) { return 4 * (((ct >> 3) & 1) ^ ((ct >> 2) & 1)) + (ct & 3); }

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Waits for chunk i's table, reads the thread's pool rows and issues their loads
// from `pool`, and releases the table slot at once.  An end-of-stream table
// loads nothing and sets `n` to the chunk count.
__device__ __forceinline__ bool prefetch_rows(const Ctx& c, const int8_t* pool, int ct, int i,
                                              uint4 (&x)[kRowsPerThread], int& n) {
    if (i > n) return true;   // past the end-of-stream tables: there is nothing to read
    if (!wait_addr(c, bar(c, BAR_TAB_FULL + i % kNS), (i / kNS) & 1)) return false;
    const RawTab* T = raw_tab(c, i % kNS);
    int rows[kRowsPerThread];
    const bool end = T->end != 0;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) rows[k] = end ? -1 : T->row[row0(ct) + (kLoadThreads / 8) * k];
    if (end) n = min(n, *c.n_final);
    __syncwarp();
    if ((ct & 31) == 0) tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + i % kNS));
    const int i16 = col16(ct);
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k)
        x[k] = rows[k] >= 0 ? ldg_stream16(pool + (size_t)rows[k] * kHeadDim + 16 * i16) : make_uint4(0, 0, 0, 0);
    return true;
}

// Converts the thread's 16 bytes of row k to the exact FP16 integers (|int8| <=
// 128 fits FP16's significand) and stores them into the 128-byte-swizzled tile.
__device__ __forceinline__ void store_row(uint8_t* tile, int ct, int k, uint4 x) {
    const int i = col16(ct), row = row0(ct) + (kLoadThreads / 8) * k;
    uint8_t* rowp = tile + (i >> 2) * (kTileBytes / 2) + row * 128;
    const uint32_t c0 = 2u * (uint32_t)(i & 3);
    uint4 lo, hi;
    int8x4_to_f16(x.x, lo.x, lo.y);
    int8x4_to_f16(x.y, lo.z, lo.w);
    int8x4_to_f16(x.z, hi.x, hi.y);
    int8x4_to_f16(x.w, hi.z, hi.w);
    *reinterpret_cast<uint4*>(rowp + ((c0 ^ (row & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (row & 7)) << 4)) = hi;
}

// One loader group (K: tiles kOffKb, kNK deep, freed by S; V: tiles kOffVb, kNV
// deep, freed by P V).  Chunk i's rows are in registers while the loads of
// chunks i+1 and i+2 are in flight.  At the end the K group arrives once more on
// K_FULL: that is how the S issuer learns the stream has ended.  That arrival,
// like every other, first waits for the tile's previous use to complete (S(n-3)):
// the loader warps do not run in step, and an mbarrier only counts arrivals, so
// one warp's end arrival must not be counted with a slower warp's arrival for
// chunk n-3.
template <bool kIsV>
__device__ void loader_role(const Ctx& c, int ct) {
    constexpr int nb = kIsV ? kNV : kNK;
    const int8_t* pool = kIsV ? c.a->v_pool : c.a->k_pool;
    uint8_t* tiles = c.base + (kIsV ? kOffVb : kOffKb);
    const int bar_full = kIsV ? BAR_V_FULL : BAR_K_FULL, bar_empty = kIsV ? BAR_V_EMPTY : BAR_K_EMPTY;
    int n = INT32_MAX;   // the chunk count, once an end-of-stream table has been seen
    uint4 x[kRowsPerThread], x1[kRowsPerThread], xn[kRowsPerThread];
    if (!prefetch_rows(c, pool, ct, 0, x, n)) return;
    if (!prefetch_rows(c, pool, ct, 1, x1, n)) return;
#pragma unroll 1
    for (int i = 0;; ++i) {
        const int b = i % nb;
        if (i >= n) {
            if (!kIsV) {
                if (!wait_addr(c, bar(c, bar_empty + b), ((i / nb) & 1) ^ 1)) return;
                __syncwarp();
                if ((ct & 31) == 0) tc::mbar_arrive(bar(c, bar_full + b));
            }
            return;
        }
        if (!prefetch_rows(c, pool, ct, i + 2, xn, n)) return;
        if (!wait_addr(c, bar(c, bar_empty + b), ((i / nb) & 1) ^ 1)) return;   // tile b free again
        uint8_t* tile = tiles + b * kTileBytes;
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) store_row(tile, ct, k, x[k]);
        tc::fence_proxy_async();
        __syncwarp();
        if ((ct & 31) == 0) tc::mbar_arrive(bar(c, bar_full + b));
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) {
            x[k] = x1[k];
            x1[k] = xn[k];
        }
    }
}

// ------------------------------------------------------------------ MMA issuers
// Two warps issue (the whole warp runs the loop, one elected lane issues), so
// the waits of one stream do not hold up the other.  The S issuer: S(t) needs
// chunk t's K tile and S buffer t % 3 back, i.e. P(t-3) V complete (it read
// P(t-3) from that buffer).  The P V issuer: P(t) V needs P(t) and chunk t's V
// tile; tcgen05.mma from one thread executes in issue order, so the P V stream
// accumulates into O in chunk order.  Both learn the chunk count from the
// stream's end (an extra K_FULL arrival; P_READY of the chunk past the last).
constexpr uint32_t kF16 = ~((7u << 7) | (7u << 10));   // A and B format fields (bits 7-12) zero: FP16

__device__ void mma_s_role(const Ctx& c) {
    constexpr uint32_t idS = tc::idesc_bf16(128, kChunk, false, false) & kF16;   // A = Q (TMEM), B = K tile, K-major
    // Operand descriptors are built once; a K step or another buffer only moves the
    // 14-bit start-address field (address >> 4), which never carries out of it
    // (shared-memory addresses are below 256 KB).
    const uint64_t dk0 = tc::smem_desc(c.base_u + kOffKb, 16, 1024, 2);
    const uint32_t tQ = c.tmem + kColQ;
    bool ok = wait_addr(c, bar(c, BAR_Q_READY), 0);
    for (int t = 0; ok; ++t) {
        const int b = t % kNK, sb = t % kNSb;
        if (t >= kNSb && !(ok = wait_addr(c, bar(c, BAR_PV_DONE + sb), ((t - kNSb) / kNSb) & 1))) break;
        if (!(ok = wait_addr(c, bar(c, BAR_K_FULL + b), (t / kNK) & 1))) break;
        if (t >= *c.n_final) break;
        tc::fence_after_sync();
        const uint64_t dk = dk0 + (uint64_t)((b * kTileBytes) >> 4);
        const uint32_t tS = c.tmem + kColS + 64 * sb;
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {   // Q dims 16k..16k+15: TMEM columns 8k..8k+7
            const uint32_t koff = (k >> 2) * (kTileBytes / 2) + (k & 3) * 32;
            tc::mma_ts_elect(tS, tQ + 8 * k, dk + (koff >> 4), idS, k > 0 ? 1u : 0u);
        }
        tc::commit_elect(bar(c, BAR_S_FULL + sb));
        tc::commit_elect(bar(c, BAR_K_EMPTY + b));
    }
    // every MMA issued above must be complete before Tensor Memory is released
    tc::commit_elect(bar(c, BAR_DRAIN_S));
    if (!tc::mbar_wait_drain(bar(c, BAR_DRAIN_S), 0, kWaitNs)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

__device__ void mma_pv_role(const Ctx& c) {
    constexpr uint32_t idO = tc::idesc_bf16(128, kHeadDim, false, true) & kF16;  // A = P (TMEM), B = V tile, MN-major
    const uint64_t dv0 = tc::smem_desc(c.base_u + kOffVb, 8192, 1024, 2);
    for (int t = 0;; ++t) {
        const uint32_t tO = c.tmem + kColO + 128 * (t & 1);   // the O of the set that took chunk t
        const int b = t % kNV, sb = t % kNSb;
        if (!wait_addr(c, bar(c, BAR_P_READY + sb), (t / kNSb) & 1)) break;
        if (t >= *c.n_final) {   // after the last P V: O is final once these MMAs complete
            tc::commit_elect(bar(c, BAR_O_DONE));
            break;
        }
        if (!wait_addr(c, bar(c, BAR_V_FULL + b), (t / kNV) & 1)) break;
        tc::fence_after_sync();
        const uint64_t dv = dv0 + (uint64_t)((b * kTileBytes) >> 4);
        const uint32_t tP = c.tmem + kColS + 64 * sb;
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)   // P of cells 16k..16k+15: columns 8(k&1) + 32(k>>1)
            tc::mma_ts_elect(tO, tP + 8 * (k & 1) + 32 * (k >> 1), dv + ((k * 2048) >> 4), idO,
                             (t > 1 || k > 0) ? 1u : 0u);
        tc::commit_elect(bar(c, BAR_V_EMPTY + b));
        tc::commit_elect(bar(c, BAR_PV_DONE + sb));
    }
    tc::commit_elect(bar(c, BAR_DRAIN_PV));
    if (!tc::mbar_wait_drain(bar(c, BAR_DRAIN_PV), 0, kWaitNs)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ softmax
// Weights of 16 score columns in log2 units: x = s * ks + vsh where selected,
// -inf elsewhere (ks: the 16 columns' K scales times sm_scale * log2(e), in
// shared memory; vsh: the chunk's V exponent).  `uniform` (warp-uniform): every
// lane selected all of the slice or none of it, so the mask is a per-lane addend
// (vsh or -inf) of the same FMA.
__device__ __forceinline__ void scale_mask16(uint32_t* s, uint32_t sel, bool uniform, const float* ks, float vsh,
                                             float& mx, float& my) {
    if (uniform) {
        const float bias = sel ? vsh : -INFINITY;
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
    const float2 v2 = make_float2(vsh, vsh);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        const float4 kq = *reinterpret_cast<const float4*>(ks + 4 * c4);
        const float2 a = __ffma2_rn(make_float2(__uint_as_float(s[4 * c4]), __uint_as_float(s[4 * c4 + 1])),
                                    make_float2(kq.x, kq.y), v2);
        const float2 b = __ffma2_rn(make_float2(__uint_as_float(s[4 * c4 + 2]), __uint_as_float(s[4 * c4 + 3])),
                                    make_float2(kq.z, kq.w), v2);
        const float v0 = ((sel >> (4 * c4)) & 1u) ? a.x : -INFINITY;
        const float v1 = ((sel >> (4 * c4 + 1)) & 1u) ? a.y : -INFINITY;
        const float v2_ = ((sel >> (4 * c4 + 2)) & 1u) ? b.x : -INFINITY;
        const float v3 = ((sel >> (4 * c4 + 3)) & 1u) ? b.y : -INFINITY;
        s[4 * c4] = __float_as_uint(v0);
        s[4 * c4 + 1] = __float_as_uint(v1);
        s[4 * c4 + 2] = __float_as_uint(v2_);
        s[4 * c4 + 3] = __float_as_uint(v3);
        mx = fmax3(mx, v0, v1);
        my = fmax3(my, v2_, v3);
    }
}


// Weights e = 2^(x - m) for 16 columns: e is added to la / lb (the row's sum),
// and e * vs (vs: the 16 columns' scaled V scales in shared memory) goes out as
// 8 packed FP16 pairs -- the P that meets the exact V rows in P V.
__device__ __forceinline__ void exp16(const uint32_t* s, const float* vs, float2 nm, uint32_t* p, float2& la,
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
        p[2 * u4] = pack_f16x2(w01.x, w01.y);
        p[2 * u4 + 1] = pack_f16x2(w23.x, w23.y);
    }
}


// Softmax warp of set `set` (chunks t % 2 == set), half `hf` (0: columns [0,32)
// of each chunk, 1: [32,64)) over lane quadrant `quad` (rows 32*quad + lane).
__device__ void softmax_role(const Ctx& c, int set, int hf, int quad, int lane) {
    const AttnArgs& a = *c.a;
    const int r = 32 * quad + lane;
    const int j = r / kHeadsPerKv, hq = r - j * kHeadsPerKv;
    const bool row_ok = j < c.nj;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const size_t row_off = ((size_t)(c.q_begin + j) * c.n_heads + (size_t)c.h * kHeadsPerKv + hq) * kHeadDim;
    float* xchg = smem_f(c, kOffXchg);     // [set][parity][half][row]
    float* mslot = smem_f(c, kOffMslot);   // [set][row]: each set's final running max
    float* lsum = smem_f(c, kOffLsum);     // [set * 2 + half][row]
    float* rsv = smem_f(c, kOffRs);        // [row]
    // Set 0 writes Q row r, this warp's 64-element half, as FP16 pairs into TMEM
    // (lane r, columns kColQ + 32 hf ...): the A operand of S.  BF16 -> FP16 is
    // exact for |q| in [2^-17, 2^16); a row whose largest |q| is 2^14 or more, or
    // below 2^-10, is stored times 2^-e (e puts that largest value in [2^12,
    // 2^13)), and its scores are multiplied back by 2^e, both exact.
    if (set == 0) {
        uint4 x[8];
        float amax = 0.f;
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
            x[q16] = row_ok ? __ldg(reinterpret_cast<const uint4*>(a.q + row_off) + 8 * hf + q16) : make_uint4(0, 0, 0, 0);
            amax = fmax3(amax, fmax3(fabsf(bf16_lo(x[q16].x)), fabsf(bf16_hi(x[q16].x)), fabsf(bf16_lo(x[q16].y))),
                         fmax3(fabsf(bf16_hi(x[q16].y)), fabsf(bf16_lo(x[q16].z)), fabsf(bf16_hi(x[q16].z))));
            amax = fmax3(amax, fabsf(bf16_lo(x[q16].w)), fabsf(bf16_hi(x[q16].w)));
        }
        // the row's largest |q| over both halves (row-sum slots: not used before the end)
        lsum[hf * kRows + r] = amax;
        if (!pair_sync(0, quad, *c.abort_flag != 0)) {
            leave_all(0, quad);
            return;
        }
        amax = fmaxf(amax, lsum[(hf ^ 1) * kRows + r]);
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;   // floor(log2 amax)
        // |e| <= 114, so 2^e and 2^-e are normal floats
        const int e = (amax > 0.f && (ex >= 14 || ex < -10)) ? min(max(ex - 12, -114), 114) : 0;
        const float down = exp2i(-e);
        if (hf == 0) rsv[r] = exp2i(e);
        uint32_t qw[32];
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
            const uint32_t* bw = reinterpret_cast<const uint32_t*>(&x[q16]);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const __half2 f = __floats2half2_rn(bf16_lo(bw[v]) * down, bf16_hi(bw[v]) * down);
                qw[4 * q16 + v] = *reinterpret_cast<const uint32_t*>(&f);
            }
        }
        tc::tmem_st32(c.tmem + lane_base + kColQ + 32 * hf, qw);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_Q_READY));
    }
    // the row's Q scale (written by set 0 before its Q_READY arrive)
    if (!wait_addr(c, bar(c, BAR_Q_READY), 0)) {
        leave_all(set, quad);
        return;
    }
    const float rs = rsv[r];
    const bool qscaled = __any_sync(0xffffffffu, rs != 1.f);
    // Weights are kept in log2 units, x = q.k * ks + ev, and masked after all
    // scaling, so p = 2^(x - m) holds for any sm_scale (0 gives equal weights; no
    // -inf is ever multiplied).  Each set keeps its own running max m, its own
    // O and, per warp, the sum l of its half's weights relative to m; the two
    // sets are combined at the end.
    const float thresh = kRescaleLog2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = set;; t += 2) {
        const bool aborted = *c.abort_flag != 0;   // read after the previous pair barrier
        const int sb = t % kNSb, ts = t % kNS;
        const uint32_t tS = c.tmem + lane_base + kColS + 64 * sb;
        if (!(ok = wait_addr(c, bar(c, BAR_TAB_FULL + ts), (t / kNS) & 1))) break;   // the chunk's tables
        const RawTab* T = raw_tab(c, ts);
        if (T->end) {   // past the last chunk; the set at the chunk count tells the P V issuer
            // That arrival waits, like a chunk's own, for the buffer's previous P V
            // (chunk t-3) to complete: the warps do not run in step, and an mbarrier
            // only counts arrivals, so it must not be counted with a slower warp's
            // arrival for chunk t-3.
            const bool signal = t == *c.n_final;
            if (signal && t >= kNSb &&
                !(ok = wait_addr(c, bar(c, BAR_PV_DONE + sb), ((t - kNSb) / kNSb) & 1)))
                break;
            __syncwarp();
            if (lane == 0) {
                if (signal) tc::mbar_arrive(bar(c, BAR_P_READY + sb));
                tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));
            }
            break;
        }
        const uint32_t sel = (uint32_t)(T->rowmask[j] >> (32 * hf));
        const float vsh = T->vshift, vinv = T->vinv;
        if (!(ok = wait_addr(c, bar(c, BAR_S_FULL + sb), (t / kNSb) & 1))) break;
        tc::fence_after_sync();
        uint32_t sv[32];
        tc::tmem_ld32(tS + 32 * hf, sv);
        // A 16-column slice that none of the warp's queries selected is skipped (its P is zero).
        const uint32_t sel_lo = sel & 0xFFFFu, sel_hi = sel >> 16;
        const bool act_lo = __any_sync(0xffffffffu, sel_lo != 0), act_hi = __any_sync(0xffffffffu, sel_hi != 0);
        const bool uni_lo = __all_sync(0xffffffffu, sel_lo == 0 || sel_lo == 0xFFFFu);
        const bool uni_hi = __all_sync(0xffffffffu, sel_hi == 0 || sel_hi == 0xFFFFu);
        const float* ksp = &T->ks[32 * hf];
        tc::tmem_wait_ld();
        if (qscaled) {   // rows stored times 2^-e: restore their scores
#pragma unroll
            for (int v = 0; v < 32; ++v) sv[v] = __float_as_uint(__uint_as_float(sv[v]) * rs);
        }
        float mx = -INFINITY, my = -INFINITY;    // two chains for more ILP
        if (act_lo) scale_mask16(&sv[0], sel_lo, uni_lo, ksp, vsh, mx, my);
        if (act_hi) scale_mask16(&sv[16], sel_hi, uni_hi, ksp + 16, vsh, mx, my);
        // swap half-chunk maxima with the partner warp of the set
        float* xb = xchg + ((2 * set + ((t >> 1) & 1)) * 2) * kRows;
        xb[hf * kRows + r] = fmaxf(mx, my);
        if (!(ok = pair_sync(set, quad, aborted))) break;
        const float m_chunk = fmaxf(fmaxf(mx, my), xb[(hf ^ 1) * kRows + r]);
        const float m_new = fmaxf(m, m_chunk);
        const bool need = (m != -INFINITY) && (m_new > m + thresh);
        const float m_use = (m == -INFINITY || need) ? m_new : m;
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        const float m_sub = m_use == -INFINITY ? 0.f : m_use;
        uint32_t p[16];
        const float2 nm = make_float2(-m_sub, -m_sub);
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
        const float* vsp = &T->vs[32 * hf];
        if (act_lo) {
            exp16(&sv[0], vsp, nm, &p[0], la, lb);
        } else {
#pragma unroll
            for (int v = 0; v < 8; ++v) p[v] = 0u;
        }
        if (act_hi) {
            exp16(&sv[16], vsp + 16, nm, &p[8], la, lb);
        } else {
#pragma unroll
            for (int v = 0; v < 8; ++v) p[8 + v] = 0u;
        }
        l = l * alpha + ((la.x + la.y) + (lb.x + lb.y)) * vinv;
        m = m_use;
        tc::tmem_st16(tS + 32 * hf, p);
        if (__any_sync(0xffffffffu, need)) {
            // this set's O must hold every earlier P V of the set before it is
            // rescaled: wait for P(t-2) V; this warp rescales its half of the set's O
            if (!(ok = wait_addr(c, bar(c, BAR_PV_DONE + (t - 2) % kNSb), ((t - 2) / kNSb) & 1))) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int q8 = 0; q8 < 4; ++q8) {
                uint32_t o[16];
                const uint32_t ta = c.tmem + lane_base + kColO + 128 * set + 64 * hf + 16 * q8;
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
            tc::mbar_arrive(bar(c, BAR_P_READY + sb));
            tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));   // done with this chunk's table
        }
    }
    if (!ok) {
        leave_all(set, quad);
        return;
    }
    const int n = *c.n_final;
    // Output columns 32 * (2 hf + set) .. + 31 of row r.
    const int ocol = 32 * (2 * hf + set);
    float* out = a.out + row_off + ocol;
    if (n == 0) {
        if (row_ok)
            for (int v = 0; v < 8; ++v) reinterpret_cast<float4*>(out)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    // Combine the two sets: M = max(m_0, m_1); each set weighs 2^(m_s - M) (0 for a
    // set with no weight on this row, whose O is not read); the row's total weight is
    // the four warps' sums so weighted.
    if (hf == 0) mslot[set * kRows + r] = m;
    lsum[(2 * set + hf) * kRows + r] = l;
    if (*c.abort_flag != 0) {
        leave_all(set, quad);
        return;
    }
    named_sync<128>(7 + quad);
    const float m0 = mslot[r], m1 = mslot[kRows + r];
    const float mm = fmaxf(m0, m1);
    const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mm), w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mm);
    const float l_tot = w0 * (lsum[r] + lsum[kRows + r]) + w1 * (lsum[2 * kRows + r] + lsum[3 * kRows + r]);
    if (!wait_addr(c, bar(c, BAR_O_DONE), 0)) return;
    tc::fence_after_sync();
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    const float s0 = w0 * inv, s1 = w1 * inv;
    uint32_t o0[32], o1[32];
    tc::tmem_ld32(c.tmem + lane_base + kColO + ocol, o0);
    tc::tmem_ld32(c.tmem + lane_base + kColO + 128 + ocol, o1);
    tc::tmem_wait_ld();
    if (row_ok) {
#pragma unroll
        for (int v = 0; v < 32; ++v) {
            const float a0 = s0 != 0.f ? __uint_as_float(o0[v]) * s0 : 0.f;
            const float a1 = s1 != 0.f ? __uint_as_float(o1[v]) * s1 : 0.f;
            o0[v] = __float_as_uint(a0 + a1);
        }
#pragma unroll
        for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(out)[v] =
                make_float4(__uint_as_float(o0[4 * v]), __uint_as_float(o0[4 * v + 1]), __uint_as_float(o0[4 * v + 2]),
                            __uint_as_float(o0[4 * v + 3]));
    }
}

template <bool kFused>
__global__ void __launch_bounds__(32 * kWarps, 1) attn_sm_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u = smem_u32(smem_raw);
    const uint32_t base_u = (raw_u + 1023u) & ~1023u;
    Ctx c;
    c.a = &a;
    c.base = smem_raw + (base_u - raw_u);
    c.base_u = base_u;
    c.abort_flag = reinterpret_cast<volatile int*>(c.base + kOffMisc + 4);
    c.n_final = reinterpret_cast<volatile int*>(c.base + kOffMisc + 8);
    // fused path: the KV heads of a group are neighbours in the grid, so its lists are read while L2 holds them
    c.g = kFused ? blockIdx.y : blockIdx.x;
    c.h = kFused ? blockIdx.x : blockIdx.y;
    c.q_begin = c.g * kGroup;
    c.nj = min(kGroup, a.n_q - c.q_begin);
    c.n_heads = a.n_kv * kHeadsPerKv;
    c.kmul = a.sm_scale * kLog2e;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int U = 0;
    if (!kFused) {
        U = __ldg(a.union_count + c.g);
        if (U < 0 || U > a.union_stride) {
            if (tid == 0) report(a.dev_status, QSA_DEV_BAD_UNION_COUNT);
            U = U < 0 ? 0 : a.union_stride;
        }
        c.ucell = a.union_cells + (size_t)c.g * a.union_stride;
        c.umask = a.union_mask + (size_t)c.g * a.union_stride;
    }

    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(c.base + kOffMisc);
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(bar(c, BAR_TAB_FULL + s), 1);
            tc::mbar_init(bar(c, BAR_TAB_EMPTY + s), 4 + 4 + kSetWarps);   // K and V loaders + one softmax set
        }
        for (int b = 0; b < kNK; ++b) {
            tc::mbar_init(bar(c, BAR_K_FULL + b), 4);
            tc::mbar_init(bar(c, BAR_K_EMPTY + b), 1);
        }
        for (int b = 0; b < kNV; ++b) {
            tc::mbar_init(bar(c, BAR_V_FULL + b), 4);
            tc::mbar_init(bar(c, BAR_V_EMPTY + b), 1);
        }
        for (int b = 0; b < kNSb; ++b) {
            tc::mbar_init(bar(c, BAR_S_FULL + b), 1);
            tc::mbar_init(bar(c, BAR_P_READY + b), kSetWarps);
            tc::mbar_init(bar(c, BAR_PV_DONE + b), 1);
        }
        tc::mbar_init(bar(c, BAR_O_DONE), 1);
        tc::mbar_init(bar(c, BAR_Q_READY), kSetWarps);   // set 0's softmax warps
        tc::mbar_init(bar(c, BAR_DRAIN_S), 1);
        tc::mbar_init(bar(c, BAR_DRAIN_PV), 1);
        *c.abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kWarpMmaS) {
        tc::tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    c.tmem = *tmem_holder;
    if (kFused) {
        // The group's union, built by the whole CTA into shared memory before the
        // pipeline starts (the same build as the union kernel's, so the same
        // entries in the same order); its scratch is the tile area and the table
        // ring, not yet in use.
        const uint32_t cap = fused_union_capacity(a.sel_stride);
        int32_t* ucell = reinterpret_cast<int32_t*>(c.base + kOffUnion);
        uint8_t* umask = c.base + kOffUnion + 4 * cap;
        uint8_t* small = c.base + kOffRawTab;
        const UnionScratch sc{reinterpret_cast<uint4*>(c.base + kOffKb), small,
                              reinterpret_cast<uint16_t*>(small + kUnionPages),
                              reinterpret_cast<int*>(small + 3 * kUnionPages),
                              reinterpret_cast<int*>(small + 3 * kUnionPages) + kGroup,
                              reinterpret_cast<int*>(small + 3 * kUnionPages) + 2 * kGroup,
                              reinterpret_cast<int*>(small + 3 * kUnionPages) + 3 * kGroup,
                              reinterpret_cast<int*>(small + 3 * kUnionPages) + 4 * kGroup,
                              reinterpret_cast<int*>(small + 3 * kUnionPages) + 5 * kGroup};
        // every list holds at most sel_stride cells, so the union fits cap entries
        U = min(build_group_union<32 * kWarps>(a.sel, a.sel_count, a.n_q, a.sel_stride, c.q_begin, ucell, umask,
                                               (int)cap, a.dev_status, sc),
                (int)cap);
        c.ucell = ucell;
        c.umask = umask;
    }
    c.U = U;
    c.n_chunks = (U + kChunk - 1) / kChunk;
    if (tid == 0) *c.n_final = c.n_chunks;
    __syncthreads();

    if (warp == kWarpProducer0 || warp == kWarpProducer1) {
        producer_role(c, warp == kWarpProducer0 ? 0 : 1, lane);
    } else if (warp == kWarpMmaS) {
        mma_s_role(c);
    } else if (warp == kWarpMmaPV) {
        mma_pv_role(c);
    } else if (warp >= 16 && warp < 20) {
        loader_role<false>(c, 32 * k_loader_index(warp) + lane);
    } else if (warp == 20 || warp == 21 || warp == 11 || warp == 15) {
        loader_role<true>(c, 32 * v_loader_index(warp) + lane);
    } else {
        softmax_role(c, warp >> 3, (warp >> 2) & 1, warp & 3, lane);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMmaS) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemCols);
    }
}

template <bool kFused>
cudaError_t launch_sm(const AttnArgs& a, size_t smem, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(attn_sm_kernel<kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned n_groups = (unsigned)((a.n_q + kGroup - 1) / kGroup);
    const dim3 grid = kFused ? dim3((unsigned)a.n_kv, n_groups) : dim3(n_groups, (unsigned)a.n_kv);
    attn_sm_kernel<kFused><<<grid, 32 * kWarps, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t attn_fused_smem_bytes(int sel_stride) {
    return (size_t)kSmemBytes + 16 + (size_t)fused_union_capacity(sel_stride) * 5;
}

cudaError_t launch_attn_sm(const AttnArgs& a, cudaStream_t stream) { return launch_sm<false>(a, kSmemBytes, stream); }
cudaError_t launch_attn_fused(const AttnArgs& a, cudaStream_t stream) {
    return launch_sm<true>(a, attn_fused_smem_bytes(a.sel_stride), stream);
}

}  // namespace qsa
