// attn_tc.cu -- union attention on the 5th-generation tensor cores (tcgen05.mma,
// accumulators in Tensor Memory), warp-specialised and pipelined with mbarriers.
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary: one work-group per (8 positions, KV head) covers
// the 96 rows of 8 positions x 12 heads; the INT8 K/V of each 64-cell chunk of
// the union is dequantised once; S = Q K^T and O += P V run on the matrix units
// with FP32 sums; in the online softmax a cell is -inf for every position that
// did not select it.  Section Extra Notes: non-resident pages are masked.
//
// One CTA per (group g, KV head h): 96 query-head rows (row r = j*12 + hq, TMEM
// lane r) sharing the group's union.  Two CTAs share an SM.  Warp roles:
//   warps 0-2, 4-6  softmax.  Warps w and w+4 own the same 32 rows (TMEM lane
//              quadrant w); warp w takes columns [0,32) of every 64-cell chunk
//              and warp w+4 columns [32,64), so each row's online softmax is
//              split over two warps that swap their half-chunk maxima through
//              shared memory (one 64-thread named barrier per chunk) and so
//              always share one running max.  Per chunk a warp reads its 32 S
//              columns from TMEM, scales each by its K scale, masks cells its
//              query did not select (one 64-bit selection word per query),
//              computes p = 2^(v - m) in the exp2 domain (the table's K scale
//              carries sm_scale * log2(e); the running max m only moves when a
//              score exceeds it by more than 2^32 in p, and O is rescaled in
//              TMEM only then), writes P = p * (V scale)
//              as BF16 over its own S columns, and keeps its own FP32 sum of p.  At the
//              end the pair adds their sums and each stores half of O's columns.
//              They also write the Q rows, as FP16, into the shared-memory Q tile
//              first (a row outside FP16's comfortable range is stored times an
//              exact power of two that the scores undo).
//   warp 3     producer: union entries -> page table -> per-chunk tables in an
//              8-deep ring (pool row of each cell, K/V scales, one 64-bit
//              selection mask per query built with warp ballots), three chunks
//              of loads in flight, and an L2 prefetch of each chunk's K/V rows
//              well before the loaders gather them.  Also zeroes the Q tile's pad
//              rows.
//   warp 7     MMA issuer (one thread), per chunk t: S(t) = Q K^T (A = Q tile,
//              B = K tile, FP16, M=128 N=64 K=128) into S buffer t & 1, then
//              O += P(t-1) V (A = P from TMEM, B = V tile, BF16, M=128 N=128 K=64).
//              S is double-buffered, so S(t) runs while the softmax warps work
//              on chunk t-1.  (A tcgen05.mma with M=128, K=16 costs the same ~46
//              cycles for any N up to 64 and reaches full rate at N=128, so S is
//              issued 64 columns wide.)
//   warps 8-11 loaders/converters: one 16-byte load per row and thread of the
//              INT8 K rows (issued one chunk ahead into registers) and V rows
//              (issued before the chunk's K conversion), converted straight into
//              operand tiles in the 128-byte swizzled layouts the tensor core
//              reads -- K to FP16, V to BF16 -- double-buffered; a K tile is
//              refilled once S has read it, a V tile once P V has.  K and V stay
//              exact (|int8| <= 128 fits both formats): the K scale multiplies
//              the score column in FP32, so the logits carry no 16-bit rounding,
//              and the V scale multiplies p before P is rounded to BF16, so each
//              product term is rounded once.
// Rows 96-127 of the M=128 tiles are padding (Q rows zero, never stored).
// The MMA thread commits three barriers per chunk: S_FULL[b] (S buffer b full,
// and K tile b free), V_EMPTY[b] (P V done: V tile b free, and O may be
// rescaled) and, once, O_DONE.
// TMEM (256 columns): S/P buffers [0,64) and [64,128), O [128,256).  In S
// buffer b, P of columns [0,32) goes to [b*64, b*64+16) and P of columns
// [32,64) to [b*64+32, b*64+48): each softmax warp overwrites only S columns it
// has already read.
// Every wait is bounded in time; a wait that runs out sets a CTA-wide abort
// flag and QSA_DEV_WAIT_TIMEOUT, every role then stops, the MMA issuer drains
// the MMAs it started, and the CTA frees its Tensor Memory and exits.
#include "qsa_common.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace {

constexpr int kWarpProducer = 3;
constexpr int kWarpMma = 7;
constexpr int kWarpConv0 = 8;
constexpr int kConvWarps = 4;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kSoftWarps = 6;
constexpr int kThreadsTc = 32 * (kWarpConv0 + kConvWarps);   // 384
constexpr int kCtasPerSm = 2;
constexpr int kNS = 8;                     // per-chunk table ring
constexpr int kNB = 2;                     // BF16 operand buffers
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128;  // S buffer sb at kColS + 64 * sb
// Lazy rescale threshold (exp2 domain): the running max only moves, and O is
// only rescaled, when a score exceeds it by more than 2^32 in p.  P then stays
// below 2^32 (BF16 holds it), O and l below ~1e23 (FP32 holds them), and BF16 /
// FP32 rounding is relative, so a stale max costs no accuracy.
constexpr float kRescaleLog2 = 32.f;
constexpr uint64_t kWaitNs = 1000000000ull;

struct RawTab {
    int32_t row[kChunk];           // pool row (page * n_kv + h) * 64 + cell % 64; -1 for a masked cell
    float ks[kChunk];              // K scale * sm_scale * log2(e); 0 for a masked cell
    float vs[kChunk];              // V scale; 0 for a masked cell
    uint64_t rowmask[8];           // bit c: query j of the group selected resident cell c
};

constexpr uint32_t kTileBytes = kChunk * kHeadDim * 2;      // 16 KB BF16 K or V tile (two 64-column halves)
constexpr uint32_t kQTileBytes = 128 * kHeadDim * 2;        // 32 KB BF16 Q tile (two 64-column halves)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKb = kOffQ + kQTileBytes;
constexpr uint32_t kOffVb = kOffKb + kNB * kTileBytes;
constexpr uint32_t kOffRawTab = kOffVb + kNB * kTileBytes;
// half-chunk maxima swapped by the two softmax warps of a row, by chunk parity,
// and a third set of slots for the row sums at the end (a warp may still be
// reading its partner's last maximum when the partner writes its sum)
constexpr uint32_t kOffXchg = kOffRawTab + kNS * (uint32_t)sizeof(RawTab);
constexpr uint32_t kOffBars = (kOffXchg + 3 * 2 * kRows * 4 + 7u) & ~7u;
// K and V tiles are filled and freed separately (K is free once S is done, V
// once P V is done)
// With two K tiles and two S buffers, "K tile b is free" and "S buffer b is full"
// are one event (S(t) has completed, t % 2 == b): the loaders wait on S_FULL.  And
// "P(t) V has completed" is V_EMPTY[t % 2], which the softmax also waits on
// before a rescale of O.  So the MMA thread commits three barriers per chunk.
static_assert(kNB == 2, "K tile b and S buffer b share the S_FULL barrier");
enum { BAR_TAB_FULL = 0, BAR_TAB_EMPTY = kNS, BAR_K_FULL = 2 * kNS, BAR_V_FULL = BAR_K_FULL + kNB,
       BAR_V_EMPTY = BAR_V_FULL + kNB, BAR_S_FULL = BAR_V_EMPTY + kNB, BAR_P_READY = BAR_S_FULL + 2,
       BAR_O_DONE = BAR_P_READY + 2, BAR_Q_READY, BAR_DRAIN, NUM_BARS };
constexpr uint32_t kOffMisc = kOffBars + NUM_BARS * 8;      // tmem base, abort flag
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;           // + alignment slack
static_assert(kSmemBytes * kCtasPerSm <= 226 * 1024, "shared memory budget");

struct Ctx {
    const AttnArgs* a;
    uint8_t* base;
    uint32_t base_u;
    uint32_t tmem;
    volatile int* abort_flag;
    int g, h, nj, q_begin, n_heads, U, n_chunks;
    float kmul;
};

__device__ __forceinline__ uint32_t bar(const Ctx& c, int i) { return c.base_u + kOffBars + 8u * i; }
__device__ __forceinline__ RawTab* raw_tab(const Ctx& c, int s) {
    return reinterpret_cast<RawTab*>(c.base + kOffRawTab) + s;
}

__device__ __forceinline__ bool wait_addr(const Ctx& c, uint32_t addr, uint32_t parity) {
    if (tc::mbar_wait(addr, parity, c.abort_flag, kWaitNs)) return true;
    report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
    return false;
}

// Barrier among the 64 threads of the two softmax warps that own lane quadrant q
// (named barriers 1-3; immediate ids keep the kernel's barrier count at 4).  A
// named barrier cannot time out, so after an abort a warp never waits on one: it
// checks the CTA's abort flag first and returns false, and every softmax exit
// after a failed wait or a false pair_sync adds this warp's share with a
// non-blocking arrive (pair_leave).  Both warps pass the same barriers in the
// same order, so the partner is then either released from the barrier it is
// waiting on or sees the flag at its next one.  (`aborted` is the flag as read
// after this warp's previous pair barrier, which is all the argument needs.)
__device__ __forceinline__ bool pair_sync(int q, bool aborted) {
    if (aborted) return false;
    if (q == 0) asm volatile("bar.sync 1, 64;" ::: "memory");
    else if (q == 1) asm volatile("bar.sync 2, 64;" ::: "memory");
    else asm volatile("bar.sync 3, 64;" ::: "memory");
    return true;
}
__device__ __forceinline__ void pair_leave(int q) {
    if (q == 0) asm volatile("bar.arrive 1, 64;" ::: "memory");
    else if (q == 1) asm volatile("bar.arrive 2, 64;" ::: "memory");
    else asm volatile("bar.arrive 3, 64;" ::: "memory");
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct Entries {
    int cell[2], mask[2];
    bool present[2];
};

// Chunk placement.  `lead` is the index of the first page-aligned union cell
// after entry 0 among entries 1..63 (0 if there is none).  Chunk c holds union
// positions p = lead + 64c + slot, slot = 0..63; a position past the end wraps
// to entry p - U when that is one of the `lead` entries before it, and is
// empty otherwise.  So every union entry sits in exactly one slot and the chunk
// count stays ceil(U / 64); when the union is a few loose cells (such as sink
// cells 0-2) followed by whole 64-cell pages, every chunk but the last is one
// whole page, and each query selects all of such a chunk or none of it.
__device__ __forceinline__ int union_lead(const Ctx& c, int lane) {
    const int32_t* ucell = c.a->union_cells + (size_t)c.g * c.a->union_stride;
    const uint32_t b0 =
        __ballot_sync(0xffffffffu, lane >= 1 && lane < c.U && (__ldg(ucell + lane) & (kPage - 1)) == 0);
    if (b0) return __ffs(b0) - 1;
    const uint32_t b1 = __ballot_sync(0xffffffffu, 32 + lane < c.U && (__ldg(ucell + 32 + lane) & (kPage - 1)) == 0);
    return b1 ? 31 + __ffs(b1) : 0;
}

__device__ __forceinline__ Entries load_entries(const Ctx& c, int lead, int chunk, int lane) {
    Entries e;
    const int32_t* ucell = c.a->union_cells + (size_t)c.g * c.a->union_stride;
    const uint8_t* umask = c.a->union_mask + (size_t)c.g * c.a->union_stride;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int p = lead + chunk * kChunk + lane + 32 * k;
        const int u = p < c.U ? p : (p - c.U < lead ? p - c.U : -1);
        e.present[k] = chunk < c.n_chunks && u >= 0;
        e.cell[k] = e.present[k] ? __ldg(ucell + u) : 0;
        e.mask[k] = e.present[k] ? __ldg(umask + u) : 0;
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

// Three chunks of dependent loads stay in flight: entries of chunk i+3, page
// table of chunk i+2, scales of chunk i+1, while chunk i's table is written.
__device__ void producer_role(const Ctx& c, int lane) {
    {   // zero the Q tile's pad rows 96-127 once
        uint8_t* q = c.base + kOffQ;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int e = lane + 32 * k, row = 96 + (e >> 4), half = (e >> 3) & 1, q16 = e & 7;
            *reinterpret_cast<uint4*>(q + half * (kQTileBytes / 2) + row * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    tc::fence_proxy_async();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(c, BAR_Q_READY));
    if (c.n_chunks == 0) return;
    const int lead = union_lead(c, lane);
    Entries e0 = load_entries(c, lead, 0, lane), e1 = load_entries(c, lead, 1, lane),
            e2 = load_entries(c, lead, 2, lane);
    int pg0[2], pg1[2], r0[2];
    load_pages(c, e0, pg0);
    load_pages(c, e1, pg1);
    pool_rows(c, e0, pg0, r0);
    Scales s0 = load_scales(c, r0);
    for (int i = 0; i < c.n_chunks; ++i) {
        const int ts = i % kNS;
        const Entries e3 = load_entries(c, lead, i + 3, lane);
        int pg2[2], r1[2];
        load_pages(c, e2, pg2);
        pool_rows(c, e1, pg1, r1);
        const Scales s1 = load_scales(c, r1);
        // the loaders gather chunk i+1 several chunks from now: pull its rows into L2
#pragma unroll
        for (int k = 0; k < 2; ++k)
            if (r1[k] >= 0) {
                const size_t off = (size_t)r1[k] * kHeadDim;
                prefetch_l2(c.a->k_pool + off);
                prefetch_l2(c.a->v_pool + off);
            }
        if (!wait_addr(c, bar(c, BAR_TAB_EMPTY + ts), ((i / kNS) & 1) ^ 1)) break;
        RawTab* T = raw_tab(c, ts);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool ok = r0[k] >= 0;
            T->row[lane + 32 * k] = ok ? r0[k] : -1;
            T->ks[lane + 32 * k] = ok ? __half2float(__ushort_as_half(s0.ks[k])) * c.kmul : 0.f;
            T->vs[lane + 32 * k] = ok ? __half2float(__ushort_as_half(s0.vs[k])) : 0.f;
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

// ------------------------------------------------------------------ loaders / converters

// Thread ct of the loader group handles, in each of its rows row0(ct) + 16k
// (k = 0..3), the 16 bytes [16i, 16i+16) with i = col16(ct): one 16-byte load
// per row, converted to 16 BF16 / FP16 values = two 16-byte stores into half
// i >> 2 of the tile.  A 16-byte shared store is served 8 lanes at a time; the 8
// lanes of each such phase take an even and an odd row and opposite halves, so
// the even row fills the even 16-byte slots of its swizzled 128-byte row and the
// odd row the odd ones: every phase is one conflict-free wavefront.
constexpr int kRowsPerThread = kChunk * 8 / kConvThreads;
__device__ __forceinline__ int row0(int ct) { return 4 * (ct >> 5) + 2 * ((ct >> 4) & 1) + ((ct >> 2) & 1); }
__device__ __forceinline__ int col16(int ct) { return 4 * (((ct >> 3) & 1) ^ ((ct >> 2) & 1)) + (ct & 3); }

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Gathers the thread's 16 bytes of its rows (pool rows `rows`, -1 = masked).
__device__ __forceinline__ void load_rows(const int8_t* pool, const int (&rows)[kRowsPerThread], int ct,
                                          uint4 (&x)[kRowsPerThread]) {
    const int i = col16(ct);
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k)
        x[k] = rows[k] >= 0 ? ldg_stream16(pool + (size_t)rows[k] * kHeadDim + 16 * i) : make_uint4(0, 0, 0, 0);
}

// Wait for chunk i's table, read the thread's pool rows (kept for the V gather)
// and issue its K row loads (nothing past the last chunk).
__device__ __forceinline__ bool prefetch_k(const Ctx& c, int ct, int i, int (&rows)[kRowsPerThread],
                                           uint4 (&kx)[kRowsPerThread]) {
    if (i >= c.n_chunks) return true;
    if (!wait_addr(c, bar(c, BAR_TAB_FULL + i % kNS), (i / kNS) & 1)) return false;
    const RawTab* T = raw_tab(c, i % kNS);
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) rows[k] = T->row[row0(ct) + (kConvThreads / 8) * k];
    load_rows(c.a->k_pool, rows, ct, kx);
    return true;
}

// Converts the thread's 16 bytes of row k and stores them into the
// 128-byte-swizzled tile at `tile`: as FP16 for K (the operand of S, whose other
// operand Q is FP16 too; 3 integer/logic instructions per 4 values) and as BF16
// for V (whose partner P needs BF16's exponent range; 6 per 4 values).
template <bool kF16>
__device__ __forceinline__ void store_row(uint8_t* tile, int ct, int k, uint4 x) {
    const int i = col16(ct), row = row0(ct) + (kConvThreads / 8) * k;
    uint8_t* rowp = tile + (i >> 2) * (kTileBytes / 2) + row * 128;
    const uint32_t c0 = 2u * (uint32_t)(i & 3);
    uint4 lo, hi;
    if (kF16) {
        int8x4_to_f16(x.x, lo.x, lo.y);
        int8x4_to_f16(x.y, lo.z, lo.w);
        int8x4_to_f16(x.z, hi.x, hi.y);
        int8x4_to_f16(x.w, hi.z, hi.w);
    } else {
        int8x4_to_bf16(x.x, lo.x, lo.y);
        int8x4_to_bf16(x.y, lo.z, lo.w);
        int8x4_to_bf16(x.z, hi.x, hi.y);
        int8x4_to_bf16(x.w, hi.z, hi.w);
    }
    *reinterpret_cast<uint4*>(rowp + ((c0 ^ (row & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (row & 7)) << 4)) = hi;
}

// Chunk i: its K rows are in registers.  Issue its V loads, convert K into the
// K tile of buffer i % kNB, issue chunk i+1's K loads, then convert V.  The V
// tile is refilled only after P(i-2) V, the K tile after S(i-2).
__device__ __forceinline__ bool convert_chunk(const Ctx& c, int ct, int i, const int (&rows)[kRowsPerThread],
                                              const uint4 (&kx)[kRowsPerThread], int (&rn)[kRowsPerThread],
                                              uint4 (&kn)[kRowsPerThread]) {
    const int ts = i % kNS, b = i % kNB;
    const uint32_t par = ((i / kNB) & 1) ^ 1;
    uint8_t* kb = c.base + kOffKb + b * kTileBytes;
    uint8_t* vb = c.base + kOffVb + b * kTileBytes;
    uint4 vx[kRowsPerThread];
    load_rows(c.a->v_pool, rows, ct, vx);
    if (!wait_addr(c, bar(c, BAR_S_FULL + b), par)) return false;   // S(i-2) has read K tile b
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) store_row<true>(kb, ct, k, kx[k]);
    tc::fence_proxy_async();
    __syncwarp();
    if ((ct & 31) == 0) tc::mbar_arrive(bar(c, BAR_K_FULL + b));
    if (!prefetch_k(c, ct, i + 1, rn, kn)) return false;
    if (!wait_addr(c, bar(c, BAR_V_EMPTY + b), par)) return false;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) store_row<false>(vb, ct, k, vx[k]);
    tc::fence_proxy_async();
    __syncwarp();
    if ((ct & 31) == 0) {
        tc::mbar_arrive(bar(c, BAR_V_FULL + b));
        tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));
    }
    return true;
}

// One conversion body (kept out of line of any unrolling, to keep the kernel's
// code small); the next chunk's K rows move into place after each chunk.
__device__ void converter_role(const Ctx& c, int ct) {
    if (c.n_chunks == 0) return;
    uint4 kx[kRowsPerThread], kn[kRowsPerThread];
    int rows[kRowsPerThread], rn[kRowsPerThread];
    if (!prefetch_k(c, ct, 0, rows, kx)) return;
#pragma unroll 1
    for (int i = 0; i < c.n_chunks; ++i) {
        if (!convert_chunk(c, ct, i, rows, kx, rn, kn)) break;
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) {
            kx[k] = kn[k];
            rows[k] = rn[k];
        }
    }
}

// ------------------------------------------------------------------ MMA issuer
// Issue order: S(0), S(1), P(0) V, S(2), P(1) V, ..., S(n-1), P(n-2) V,
// P(n-1) V.  S(t) needs chunk t's K tile (and, for t = 0, the Q tile) and its S
// buffer back, i.e. P(t-2) V issued before it (tcgen05.mma executes in issue
// order, so P(t-2) is read before S(t) overwrites it); that makes the order
// above the only one possible.  P(t) V needs P(t) and chunk t's V tile.
__device__ void mma_role(const Ctx& c) {
    // A = Q tile, B = K tile, both FP16 (format fields, bits 7-12, zero), K-major
    constexpr uint32_t idS = tc::idesc_bf16(128, kChunk, false, false) & ~((7u << 7) | (7u << 10));
    constexpr uint32_t idO = tc::idesc_bf16(128, kHeadDim, false, true);   // B = V tile, MN-major
    const int n = c.n_chunks;
    // Operand descriptors are built once; a K step or another buffer only moves the
    // 14-bit start-address field (address >> 4), which never carries out of it
    // (shared-memory addresses are below 256 KB).
    const uint64_t dq0 = tc::smem_desc(c.base_u + kOffQ, 16, 1024, 2);
    const uint64_t dk0 = tc::smem_desc(c.base_u + kOffKb, 16, 1024, 2);
    const uint64_t dv0 = tc::smem_desc(c.base_u + kOffVb, 8192, 1024, 2);
    auto issue_s = [&](int t) -> bool {
        const int b = t % kNB;
        if (t == 0 && !wait_addr(c, bar(c, BAR_Q_READY), 0)) return false;
        if (!wait_addr(c, bar(c, BAR_K_FULL + b), (t / kNB) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dk = dk0 + (uint64_t)((b * kTileBytes) >> 4);
        const uint32_t tS = c.tmem + kColS + 64 * (t & 1);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t koff = (k >> 2) * (kTileBytes / 2) + (k & 3) * 32;
            const uint32_t qoff = (k >> 2) * (kQTileBytes / 2) + (k & 3) * 32;
            tc::mma_ss(tS, dq0 + (qoff >> 4), dk + (koff >> 4), idS, k > 0 ? 1u : 0u);
        }
        tc::commit(bar(c, BAR_S_FULL + (t & 1)));   // also: K tile b is free
        return true;
    };
    auto issue_pv = [&](int t) -> bool {
        const int b = t % kNB;
        if (!wait_addr(c, bar(c, BAR_P_READY + (t & 1)), (t >> 1) & 1)) return false;
        if (!wait_addr(c, bar(c, BAR_V_FULL + b), (t / kNB) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dv = dv0 + (uint64_t)((b * kTileBytes) >> 4);
        const uint32_t tP = c.tmem + kColS + 64 * (t & 1);
        const uint32_t tO = c.tmem + kColO;
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)   // P of cells 16k..16k+15: columns 8(k&1) + 32(k>>1)
            tc::mma_ts(tO, tP + 8 * (k & 1) + 32 * (k >> 1), dv + ((k * 2048) >> 4), idO, (t > 0 || k > 0) ? 1u : 0u);
        tc::commit(bar(c, BAR_V_EMPTY + b));   // also: P(t) V has completed
        if (t == n - 1) tc::commit(bar(c, BAR_O_DONE));
        return true;
    };
    bool ok = true;
    for (int t = 0; t <= n && ok && n > 0; ++t) {
        if (t < n) ok = issue_s(t);
        if (ok && t > 0) ok = issue_pv(t - 1);
    }
    // every MMA issued above must be complete before Tensor Memory is released
    tc::commit(bar(c, BAR_DRAIN));
    if (!tc::mbar_wait_drain(bar(c, BAR_DRAIN), 0, kWaitNs)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ softmax
// Scale + mask 16 score columns: v = s * ks where selected, -inf elsewhere
// (ks: the 16 columns' K scales in shared memory).  `uniform` (warp-uniform):
// every lane selected all of the slice or none of it, so the mask is a per-lane
// bias (0 or -inf) added in the same FMA.
__device__ __forceinline__ void scale_mask16(uint32_t* s, uint32_t sel, bool uniform, const float* ks, float& mx,
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

// Weights e = 2^(v - m) for 16 columns: e is added to la / lb (the row's
// sum), and e * (V scale) goes out as 8 packed BF16 pairs -- the P that meets
// the exact BF16 V rows in P V (vs: the 16 columns' V scales in shared memory).
__device__ __forceinline__ void exp16(const uint32_t* s, const float* vs, float2 nm, uint32_t* p,
                                      float2& la, float2& lb) {
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

// Softmax warp of half `hf` (0: columns [0,32) of each chunk, 1: [32,64)) over
// lane quadrant `quad` (rows 32*quad + lane).
__device__ void softmax_role(const Ctx& c, int hf, int quad, int lane) {
    const AttnArgs& a = *c.a;
    const int r = 32 * quad + lane;
    const int j = r / kHeadsPerKv, hq = r - j * kHeadsPerKv;
    const bool row_ok = j < c.nj;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const size_t row_off = ((size_t)(c.q_begin + j) * c.n_heads + (size_t)c.h * kHeadsPerKv + hq) * kHeadDim;
    float* xchg = reinterpret_cast<float*>(c.base + kOffXchg);   // [parity][half][row]; slots 2: row sums
    // Q row r, this warp's 64-element half -> FP16 in the swizzled K-major Q tile.
    // BF16 -> FP16 is exact for |q| in [2^-17, 2^16); a row whose largest |q| is
    // 2^14 or more, or below 2^-10, is stored times 2^-e (e puts that largest value
    // in [2^12, 2^13)), and its scores are multiplied back by 2^e, both exact.
    float rs = 1.f;
    bool qscaled = false;
    {
        uint4 x[8];
        float amax = 0.f;
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
            x[q16] = row_ok ? __ldg(reinterpret_cast<const uint4*>(a.q + row_off) + 8 * hf + q16) : make_uint4(0, 0, 0, 0);
            amax = fmax3(amax, fmax3(fabsf(bf16_lo(x[q16].x)), fabsf(bf16_hi(x[q16].x)), fabsf(bf16_lo(x[q16].y))),
                         fmax3(fabsf(bf16_hi(x[q16].y)), fabsf(bf16_lo(x[q16].z)), fabsf(bf16_hi(x[q16].z))));
            amax = fmax3(amax, fabsf(bf16_lo(x[q16].w)), fabsf(bf16_hi(x[q16].w)));
        }
        // the row's largest |q| over both halves (row-sum slots: not used again before the end)
        float* xl = xchg + 4 * kRows;
        xl[hf * kRows + r] = amax;
        if (!pair_sync(quad, *c.abort_flag != 0)) {
            pair_leave(quad);
            return;
        }
        amax = fmaxf(amax, xl[(hf ^ 1) * kRows + r]);
        if (!pair_sync(quad, *c.abort_flag != 0)) {   // both have read before either writes a row sum there
            pair_leave(quad);
            return;
        }
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;   // floor(log2 amax)
        // |e| <= 114, so 2^e and 2^-e are normal floats
        const int e = (amax > 0.f && (ex >= 14 || ex < -10)) ? min(max(ex - 12, -114), 114) : 0;
        qscaled = __any_sync(0xffffffffu, e != 0);
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
        rs = __uint_as_float((uint32_t)(127 + e) << 23);                  // 2^e
        uint8_t* qt = c.base + kOffQ + hf * (kQTileBytes / 2);
#pragma unroll
        for (int q16 = 0; q16 < 8; ++q16) {
            uint4 h;
            uint32_t* hw = reinterpret_cast<uint32_t*>(&h);
            const uint32_t* bw = reinterpret_cast<const uint32_t*>(&x[q16]);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const __half2 f = __floats2half2_rn(bf16_lo(bw[v]) * down, bf16_hi(bw[v]) * down);
                hw[v] = *reinterpret_cast<const uint32_t*>(&f);
            }
            *reinterpret_cast<uint4*>(qt + r * 128 + ((q16 ^ (r & 7)) << 4)) = h;
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_Q_READY));
    }
    // Scores are kept in log2 units, v = q.k * (K scale) * sm_scale * log2(e), and
    // masked after all scaling, so p = 2^(v - m) holds for any sm_scale (0 gives
    // equal weights; no -inf is ever multiplied).
    const float thresh = kRescaleLog2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < c.n_chunks; ++t) {
        const bool aborted = *c.abort_flag != 0;   // read after the previous pair barrier
        const int sb = t & 1, ts = t % kNS;
        const uint32_t tS = c.tmem + lane_base + kColS + 64 * sb;
        if (!(ok = wait_addr(c, bar(c, BAR_TAB_FULL + ts), (t / kNS) & 1))) break;   // the chunk's tables
        const RawTab* T = raw_tab(c, ts);
        const uint32_t sel = (uint32_t)(T->rowmask[j] >> (32 * hf));
        if (!(ok = wait_addr(c, bar(c, BAR_S_FULL + sb), (t >> 1) & 1))) break;
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
        if (act_lo) scale_mask16(&sv[0], sel_lo, uni_lo, ksp, mx, my);
        if (act_hi) scale_mask16(&sv[16], sel_hi, uni_hi, ksp + 16, mx, my);
        // swap half-chunk maxima with the partner warp, so both take the same step
        float* xb = xchg + (t & 1) * (2 * kRows);
        xb[hf * kRows + r] = fmaxf(mx, my);
        if (!(ok = pair_sync(quad, aborted))) break;
        const float m_new = fmax3(m, fmaxf(mx, my), xb[(hf ^ 1) * kRows + r]);
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
        l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
        m = m_use;
        tc::tmem_st16(tS + 32 * hf, p);
        if (__any_sync(0xffffffffu, need)) {
            // O must hold every earlier P V before it is rescaled: wait for PV(t-1);
            // this warp rescales its half of O's columns
            if (!(ok = wait_addr(c, bar(c, BAR_V_EMPTY + (t - 1) % kNB), ((t - 1) / kNB) & 1))) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int q8 = 0; q8 < 4; ++q8) {
                uint32_t o[16];
                const uint32_t ta = c.tmem + lane_base + kColO + 64 * hf + 16 * q8;
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
    float* out = a.out + row_off + 64 * hf;
    if (c.n_chunks == 0) {
        if (row_ok)
            for (int v = 0; v < 16; ++v) reinterpret_cast<float4*>(out)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (!ok) {
        pair_leave(quad);
        return;
    }
    // total weight of the row: this warp's sum plus the partner's
    float* xl = xchg + 4 * kRows;
    xl[hf * kRows + r] = l;
    if (!pair_sync(quad, *c.abort_flag != 0)) {
        pair_leave(quad);
        return;
    }
    const float l_tot = l + xl[(hf ^ 1) * kRows + r];
    if (!wait_addr(c, bar(c, BAR_O_DONE), 0)) return;
    tc::fence_after_sync();
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll 1
    for (int q4 = 0; q4 < 2; ++q4) {
        uint32_t o[32];
        tc::tmem_ld32(c.tmem + lane_base + kColO + 64 * hf + 32 * q4, o);
        tc::tmem_wait_ld();
        if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
                reinterpret_cast<float4*>(out + 32 * q4)[v] =
                    make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
        }
    }
}

__global__ void __launch_bounds__(kThreadsTc, kCtasPerSm) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u = smem_u32(smem_raw);
    const uint32_t base_u = (raw_u + 1023u) & ~1023u;
    Ctx c;
    c.a = &a;
    c.base = smem_raw + (base_u - raw_u);
    c.base_u = base_u;
    c.abort_flag = reinterpret_cast<volatile int*>(c.base + kOffMisc + 4);
    c.g = blockIdx.x;
    c.h = blockIdx.y;
    c.q_begin = c.g * kGroup;
    c.nj = min(kGroup, a.n_q - c.q_begin);
    c.n_heads = a.n_kv * kHeadsPerKv;
    c.kmul = a.sm_scale * kLog2e;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int U = __ldg(a.union_count + c.g);
    if (U < 0 || U > a.union_stride) {
        if (tid == 0) report(a.dev_status, QSA_DEV_BAD_UNION_COUNT);
        U = U < 0 ? 0 : a.union_stride;
    }
    c.U = U;
    c.n_chunks = (U + kChunk - 1) / kChunk;

    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(c.base + kOffMisc);
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(bar(c, BAR_TAB_FULL + s), 1);
            tc::mbar_init(bar(c, BAR_TAB_EMPTY + s), kConvWarps + kSoftWarps);   // loaders + softmax warps
        }
        for (int b = 0; b < kNB; ++b) {
            tc::mbar_init(bar(c, BAR_K_FULL + b), kConvWarps);
            tc::mbar_init(bar(c, BAR_V_FULL + b), kConvWarps);
            tc::mbar_init(bar(c, BAR_V_EMPTY + b), 1);
        }
        for (int sb = 0; sb < 2; ++sb) {
            tc::mbar_init(bar(c, BAR_S_FULL + sb), 1);
            tc::mbar_init(bar(c, BAR_P_READY + sb), kSoftWarps);
        }
        tc::mbar_init(bar(c, BAR_O_DONE), 1);
        tc::mbar_init(bar(c, BAR_Q_READY), kSoftWarps + 1);   // softmax warps + the producer (pad rows)
        tc::mbar_init(bar(c, BAR_DRAIN), 1);
        *c.abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    c.tmem = *tmem_holder;

    if (warp == kWarpProducer) {
        producer_role(c, lane);
    } else if (warp == kWarpMma) {
        if (lane == 0) mma_role(c);
    } else if (warp >= kWarpConv0) {
        converter_role(c, tid - kWarpConv0 * 32);
    } else {
        softmax_role(c, warp >> 2, warp & 3, lane);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((a.n_q + kGroup - 1) / kGroup, a.n_kv);
    attn_tc_kernel<<<grid, kThreadsTc, kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
