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
// A CTA takes one group g and kTiles KV heads ("tiles" of 96 query-head rows
// sharing the group's union); with one tile per CTA, two CTAs share an SM.
// Warp roles (one tile: 9 warps; two tiles: 16 warps, one CTA per SM):
//   warps 0-2 (4-6)  softmax for tile 0 (1): thread r owns row r = j*12 + hq
//              (TMEM lane r).  Writes its Q row into the tile's shared-memory Q
//              tile once; per chunk reads S (64 columns) from TMEM, scales each
//              column by its K scale, masks cells its query did not select (one
//              32-bit selection word per query and half chunk), runs the online
//              softmax in the exp2 domain (sm_scale * log2(e) applied inside the
//              exponent; the running max only moves when it grows by more than
//              2^8, and O is rescaled in TMEM only then), writes P as BF16 into
//              the S columns, and finally divides O by the FP32 sum of the
//              weights and stores it.
//   warp 3     producer: union entries -> page table -> per-chunk tables in an
//              8-deep ring shared by both tiles (pool row of each cell, scales of
//              both KV heads, one 64-bit selection mask per query built with warp
//              ballots), three chunks of loads in flight.  Also zeroes the Q
//              tiles' pad rows.
//   warp 8 (7) MMA issuer (one thread) for the CTA's tiles, per chunk t:
//              S(t) = Q K^T (A = Q tile, B = K tile, M=128 N=64 K=128) into S
//              buffer t & 1, then O += P(t-1) V (A = P from TMEM, B = V tile,
//              M=128 N=128 K=64).  S is double-buffered, so S(t) runs while the
//              softmax warps work on chunk t-1.  (A tcgen05.mma with M=128, K=16
//              costs the same ~46 cycles for any N up to 64 and reaches full rate
//              at N=128, so S is issued 64 columns wide; Q stays in shared memory
//              so that TMEM has room for two S buffers.)
//   warps 4-7 (8-15)  loaders/converters for tile 0 (and 1): 16-byte loads of
//              the INT8 K rows (issued one chunk ahead into registers) and V rows
//              (issued before the chunk's K conversion),
//              converted to BF16 straight into operand tiles in the 128-byte
//              swizzled layouts the tensor core reads, double-buffered; a K tile
//              is refilled once S has read it, a V tile once P V has.  K stays
//              exact (|int8| <= 128 fits BF16) and its FP16 scale multiplies the
//              score column in FP32, so the logits carry no BF16 rounding; V is
//              multiplied by its scale in FP32 and rounded to BF16 once.
// Rows 96-127 of the M=128 tiles are padding (Q rows zero, never stored).
// TMEM columns of tile u start at 256u: S/P buffers [0,64) and [64,128) (P
// overwrites the first 32 columns of its S), O [128,256).
// Every wait is bounded in time; a wait that runs out sets a CTA-wide abort
// flag and QSA_DEV_WAIT_TIMEOUT, every role then stops, the MMA issuer drains
// the MMAs it started, and the CTA frees its Tensor Memory and exits.
#include "qsa_common.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace {

constexpr int kTiles = 1;                  // KV heads per CTA (the layout below also supports 2)
constexpr int kWarpProducer = 3;
constexpr int kConvWarps = 4;              // per tile
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kWarpMma = kTiles == 1 ? 8 : 7;
constexpr int kWarpConv0 = kTiles == 1 ? 4 : 8;
constexpr int kThreadsTc = kTiles == 1 ? 288 : 512;
constexpr int kCtasPerSm = kTiles == 1 ? 2 : 1;
constexpr int kNS = 8;                     // per-chunk table ring
constexpr int kNB = 2;                     // BF16 operand buffers per tile
constexpr uint32_t kTmemCols = 256 * kTiles;
constexpr uint32_t kTileCols = 256;        // TMEM columns per tile
constexpr uint32_t kColS = 0, kColO = 128;  // S buffer sb at kColS + 64 * sb
// Lazy rescale threshold (exp2 domain): the running max only moves, and O is
// only rescaled, when a score exceeds it by more than 2^32 in p.  P then stays
// below 2^32 (BF16 holds it), O and l below ~1e23 (FP32 holds them), and BF16 /
// FP32 rounding is relative, so a stale max costs no accuracy.
constexpr float kRescaleLog2 = 32.f;
constexpr uint64_t kWaitNs = 1000000000ull;

struct RawTab {
    int32_t row[kTiles][kChunk];   // pool row (page * n_kv + h) * 64 + cell % 64; -1 for a masked cell
    float ks[kTiles][kChunk];      // K scale; 0 for a masked cell
    float vs[kTiles][kChunk];      // V scale; 0 for a masked cell
    uint64_t rowmask[8];           // bit c: query j of the group selected resident cell c
};

constexpr uint32_t kTileBytes = kChunk * kHeadDim * 2;      // 16 KB BF16 K or V tile (two 64-column halves)
constexpr uint32_t kQTileBytes = 128 * kHeadDim * 2;        // 32 KB BF16 Q tile (two 64-column halves)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKb = kOffQ + kTiles * kQTileBytes;
constexpr uint32_t kOffVb = kOffKb + kTiles * kNB * kTileBytes;
constexpr uint32_t kOffRawTab = kOffVb + kTiles * kNB * kTileBytes;
constexpr uint32_t kOffBars = (kOffRawTab + kNS * (uint32_t)sizeof(RawTab) + 7u) & ~7u;
// per-tile barrier block: K and V tiles are filled and freed separately (K is
// free once S is done, V once P V is done)
enum { TB_K_FULL = 0, TB_K_EMPTY = kNB, TB_V_FULL = 2 * kNB, TB_V_EMPTY = 3 * kNB, TB_S_FULL = 4 * kNB,
       TB_P_READY = 4 * kNB + 2, TB_PV_DONE = 4 * kNB + 4, TB_O_DONE, TB_Q_READY, TB_COUNT };
enum { BAR_TAB_FULL = 0, BAR_TAB_EMPTY = kNS, BAR_TILE0 = 2 * kNS, BAR_DRAIN = BAR_TILE0 + kTiles * TB_COUNT, NUM_BARS };
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
    int g, h0, n_tiles, nj, q_begin, n_heads, U, n_chunks;
    float kmul;
};

__device__ __forceinline__ uint32_t bar(const Ctx& c, int i) { return c.base_u + kOffBars + 8u * i; }
__device__ __forceinline__ uint32_t tbar(const Ctx& c, int u, int i) { return bar(c, BAR_TILE0 + u * TB_COUNT + i); }
__device__ __forceinline__ RawTab* raw_tab(const Ctx& c, int s) {
    return reinterpret_cast<RawTab*>(c.base + kOffRawTab) + s;
}

__device__ __forceinline__ bool wait_addr(const Ctx& c, uint32_t addr, uint32_t parity) {
    if (tc::mbar_wait(addr, parity, c.abort_flag, kWaitNs)) return true;
    report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct Entries {
    int cell[2], mask[2];
    bool present[2];
};

__device__ __forceinline__ Entries load_entries(const Ctx& c, int chunk, int lane) {
    Entries e;
    const int32_t* ucell = c.a->union_cells + (size_t)c.g * c.a->union_stride;
    const uint8_t* umask = c.a->union_mask + (size_t)c.g * c.a->union_stride;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int u = chunk * kChunk + lane + 32 * k;
        e.present[k] = chunk < c.n_chunks && u < c.U;
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

// Pool row of each entry for the CTA's first KV head (-1 = masked); the second
// head's row is 64 further on (same page, next head).
__device__ __forceinline__ void pool_rows(const Ctx& c, const Entries& e, const int (&page)[2], int (&row)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        row[k] = -1;
        if (page[k] < 0) continue;
        if (page[k] >= c.a->n_ppages) {
            report(c.a->dev_status, QSA_DEV_BAD_PAGE);
            continue;
        }
        row[k] = (page[k] * c.a->n_kv + c.h0) * kPage + (e.cell[k] & (kPage - 1));
    }
}

struct Scales {
    uint16_t ks[kTiles][2], vs[kTiles][2];
};

__device__ __forceinline__ Scales load_scales(const Ctx& c, const int (&row)[2]) {
    Scales s;
#pragma unroll
    for (int u = 0; u < kTiles; ++u)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool ok = row[k] >= 0 && u < c.n_tiles;
            s.ks[u][k] = ok ? __ldg(c.a->k_scale + row[k] + u * kPage) : (uint16_t)0;
            s.vs[u][k] = ok ? __ldg(c.a->v_scale + row[k] + u * kPage) : (uint16_t)0;
        }
    return s;
}

// Three chunks of dependent loads stay in flight: entries of chunk i+3, page
// table of chunk i+2, scales of chunk i+1, while chunk i's table is written.
__device__ void producer_role(const Ctx& c, int lane) {
    for (int u = 0; u < c.n_tiles; ++u) {   // zero each Q tile's pad rows 96-127 once
        uint8_t* q = c.base + kOffQ + u * kQTileBytes;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int e = lane + 32 * k, row = 96 + (e >> 4), half = (e >> 3) & 1, q16 = e & 7;
            *reinterpret_cast<uint4*>(q + half * (kQTileBytes / 2) + row * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    tc::fence_proxy_async();
    __syncwarp();
    if (lane == 0)
        for (int u = 0; u < c.n_tiles; ++u) tc::mbar_arrive(tbar(c, u, TB_Q_READY));
    if (c.n_chunks == 0) return;
    Entries e0 = load_entries(c, 0, lane), e1 = load_entries(c, 1, lane), e2 = load_entries(c, 2, lane);
    int pg0[2], pg1[2], r0[2];
    load_pages(c, e0, pg0);
    load_pages(c, e1, pg1);
    pool_rows(c, e0, pg0, r0);
    Scales s0 = load_scales(c, r0);
    for (int i = 0; i < c.n_chunks; ++i) {
        const int ts = i % kNS;
        const Entries e3 = load_entries(c, i + 3, lane);
        int pg2[2], r1[2];
        load_pages(c, e2, pg2);
        pool_rows(c, e1, pg1, r1);
        const Scales s1 = load_scales(c, r1);
        // the loaders gather chunk i+1 several chunks from now: pull its rows into L2
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int u = 0; u < kTiles; ++u)
                if (r1[k] >= 0 && u < c.n_tiles) {
                    const size_t off = (size_t)(r1[k] + u * kPage) * kHeadDim;
                    prefetch_l2(c.a->k_pool + off);
                    prefetch_l2(c.a->v_pool + off);
                }
        if (!wait_addr(c, bar(c, BAR_TAB_EMPTY + ts), ((i / kNS) & 1) ^ 1)) break;
        RawTab* T = raw_tab(c, ts);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool ok = r0[k] >= 0;
#pragma unroll
            for (int u = 0; u < kTiles; ++u) {
                T->row[u][lane + 32 * k] = ok ? r0[k] + u * kPage : -1;
                T->ks[u][lane + 32 * k] = ok ? __half2float(__ushort_as_half(s0.ks[u][k])) : 0.f;
                T->vs[u][lane + 32 * k] = ok ? __half2float(__ushort_as_half(s0.vs[u][k])) : 0.f;
            }
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
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Thread ct of a tile's loader group owns rows (ct >> 3) + 16k, k = 0..3,
// 16-byte segment ct & 7, of both K and V.
constexpr int kRowsPerThread = kChunk * 8 / kConvThreads;
__device__ __forceinline__ void load_rows(const Ctx& c, const int8_t* pool, const RawTab* T, int u, int ct,
                                          uint4 (&x)[kRowsPerThread]) {
    const int seg = ct & 7;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const int r = T->row[u][(ct >> 3) + (kConvThreads / 8) * k];
        x[k] = r >= 0 ? ldg_stream(pool + (size_t)r * kHeadDim + seg * 16) : make_uint4(0, 0, 0, 0);
    }
}

// Wait for chunk i's table and issue its K row loads (nothing past the last chunk).
__device__ __forceinline__ bool prefetch_k(const Ctx& c, int u, int ct, int i, uint4 (&kx)[kRowsPerThread]) {
    if (i >= c.n_chunks) return true;
    if (!wait_addr(c, bar(c, BAR_TAB_FULL + i % kNS), (i / kNS) & 1)) return false;
    load_rows(c, c.a->k_pool, raw_tab(c, i % kNS), u, ct, kx);
    return true;
}

__device__ __forceinline__ void tile_offsets(int ct, int k, uint32_t& o_a, uint32_t& o_b, bool& odd_first) {
    // Segments 0-3 fill the first 64 columns, 4-7 the second (8 KB apart, same
    // banks); the upper four store their odd 16-byte chunk first, so each
    // quarter-warp store covers eight distinct bank groups.
    const int seg = ct & 7, row = (ct >> 3) + (kConvThreads / 8) * k;
    odd_first = (seg & 4) != 0;
    const uint32_t q = (uint32_t)(seg & 3) * 2, x = (uint32_t)(row & 7);
    const uint32_t tile = (uint32_t)(seg >> 2) * (kTileBytes / 2) + (uint32_t)row * 128;
    const uint32_t o_lo = tile + ((q ^ x) << 4), o_hi = tile + (((q + 1) ^ x) << 4);
    o_a = odd_first ? o_hi : o_lo;
    o_b = odd_first ? o_lo : o_hi;
}

// Chunk i: its K rows are in registers.  Issue its V loads, convert K into the
// K tile of buffer i % kNB, issue chunk i+1's K loads, then convert V.  The V
// tile is refilled only after P(i-2) V, the K tile after S(i-2).
__device__ __forceinline__ bool convert_chunk(const Ctx& c, int u, int ct, int i, const uint4 (&kx)[kRowsPerThread],
                                              uint4 (&kn)[kRowsPerThread]) {
    const int ts = i % kNS, b = i % kNB;
    const uint32_t par = ((i / kNB) & 1) ^ 1;
    const RawTab* T = raw_tab(c, ts);
    uint8_t* kb = c.base + kOffKb + (u * kNB + b) * kTileBytes;
    uint8_t* vb = c.base + kOffVb + (u * kNB + b) * kTileBytes;
    uint4 vx[kRowsPerThread];
    load_rows(c, c.a->v_pool, T, u, ct, vx);
    if (!wait_addr(c, tbar(c, u, TB_K_EMPTY + b), par)) return false;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        uint32_t o_a, o_b;
        bool odd_first;
        tile_offsets(ct, k, o_a, o_b, odd_first);
        uint4 lo, hi;
        int8x16_to_bf16(kx[k], lo, hi);
        *reinterpret_cast<uint4*>(kb + o_a) = odd_first ? hi : lo;
        *reinterpret_cast<uint4*>(kb + o_b) = odd_first ? lo : hi;
    }
    tc::fence_proxy_async();
    __syncwarp();
    if ((ct & 31) == 0) tc::mbar_arrive(tbar(c, u, TB_K_FULL + b));
    if (!prefetch_k(c, u, ct, i + 1, kn)) return false;
    if (!wait_addr(c, tbar(c, u, TB_V_EMPTY + b), par)) return false;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        uint32_t o_a, o_b;
        bool odd_first;
        tile_offsets(ct, k, o_a, o_b, odd_first);
        uint4 lo, hi;
        dequant16(vx[k], T->vs[u][(ct >> 3) + (kConvThreads / 8) * k], lo, hi);
        *reinterpret_cast<uint4*>(vb + o_a) = odd_first ? hi : lo;
        *reinterpret_cast<uint4*>(vb + o_b) = odd_first ? lo : hi;
    }
    tc::fence_proxy_async();
    __syncwarp();
    if ((ct & 31) == 0) {
        tc::mbar_arrive(tbar(c, u, TB_V_FULL + b));
        tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));
    }
    return true;
}

// One conversion body (kept out of line of any unrolling, to keep the kernel's
// code small); the next chunk's K rows move into place after each chunk.
__device__ void converter_role(const Ctx& c, int u, int ct) {
    if (c.n_chunks == 0) return;
    uint4 kx[kRowsPerThread], kn[kRowsPerThread];
    if (!prefetch_k(c, u, ct, 0, kx)) return;
#pragma unroll 1
    for (int i = 0; i < c.n_chunks; ++i) {
        if (!convert_chunk(c, u, ct, i, kx, kn)) break;
#pragma unroll
        for (int k = 0; k < kRowsPerThread; ++k) kx[k] = kn[k];
    }
}

// ------------------------------------------------------------------ MMA issuer
// Issue order per tile: S(0), S(1), P(0) V, S(2), P(1) V, ..., S(n-1), P(n-2) V,
// P(n-1) V.  S(t) needs chunk t's K tile (and, for t = 0, the Q tile) and its S
// buffer back, i.e. P(t-2) V issued before it (tcgen05.mma executes in issue
// order, so P(t-2) is read before S(t) overwrites it); that makes the order
// above the only one possible.  P(t) V needs P(t) and chunk t's V tile.
__device__ void mma_role(const Ctx& c) {
    constexpr uint32_t idS = tc::idesc_bf16(128, kChunk, false, false);    // A = Q tile, B = K tile, K-major
    constexpr uint32_t idO = tc::idesc_bf16(128, kHeadDim, false, true);   // B = V tile, MN-major
    const int n = c.n_chunks;
    auto issue_s = [&](int u, int t) -> bool {
        const int b = t % kNB;
        if (t == 0 && !wait_addr(c, tbar(c, u, TB_Q_READY), 0)) return false;
        if (!wait_addr(c, tbar(c, u, TB_K_FULL + b), (t / kNB) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t q_u = c.base_u + kOffQ + u * kQTileBytes;
        const uint32_t kt = c.base_u + kOffKb + (u * kNB + b) * kTileBytes;
        const uint32_t tS = c.tmem + u * kTileCols + kColS + 64 * (t & 1);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t koff = (k >> 2) * (kTileBytes / 2) + (k & 3) * 32;
            const uint32_t qoff = (k >> 2) * (kQTileBytes / 2) + (k & 3) * 32;
            tc::mma_ss(tS, tc::smem_desc(q_u + qoff, 16, 1024, 2), tc::smem_desc(kt + koff, 16, 1024, 2), idS,
                       k > 0 ? 1u : 0u);
        }
        tc::commit(tbar(c, u, TB_S_FULL + (t & 1)));
        tc::commit(tbar(c, u, TB_K_EMPTY + b));
        return true;
    };
    auto issue_pv = [&](int u, int t) -> bool {
        const int b = t % kNB;
        if (!wait_addr(c, tbar(c, u, TB_P_READY + (t & 1)), (t >> 1) & 1)) return false;
        if (!wait_addr(c, tbar(c, u, TB_V_FULL + b), (t / kNB) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vt = c.base_u + kOffVb + (u * kNB + b) * kTileBytes;
        const uint32_t tP = c.tmem + u * kTileCols + kColS + 64 * (t & 1);
        const uint32_t tO = c.tmem + u * kTileCols + kColO;
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)
            tc::mma_ts(tO, tP + 8 * k, tc::smem_desc(vt + k * 2048, 8192, 1024, 2), idO, (t > 0 || k > 0) ? 1u : 0u);
        tc::commit(tbar(c, u, TB_PV_DONE));
        tc::commit(tbar(c, u, TB_V_EMPTY + b));
        if (t == n - 1) tc::commit(tbar(c, u, TB_O_DONE));
        return true;
    };
    bool ok = true;
    for (int t = 0; t <= n && ok && n > 0; ++t) {
        for (int u = 0; u < c.n_tiles && ok && t < n; ++u) ok = issue_s(u, t);
        for (int u = 0; u < c.n_tiles && ok && t > 0; ++u) ok = issue_pv(u, t - 1);
    }
    // every MMA issued above must be complete before Tensor Memory is released
    tc::commit(bar(c, BAR_DRAIN));
    if (!tc::mbar_wait_drain(bar(c, BAR_DRAIN), 0, kWaitNs)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ softmax
// Scale + mask 16 score columns: v = s * ks where selected, -inf elsewhere.
__device__ __forceinline__ void scale_mask16(uint32_t* s, uint32_t sel, const float4 (&kq)[4], float& mx, float& my) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        const float2 a = __fmul2_rn(make_float2(__uint_as_float(s[4 * c4]), __uint_as_float(s[4 * c4 + 1])),
                                    make_float2(kq[c4].x, kq[c4].y));
        const float2 b = __fmul2_rn(make_float2(__uint_as_float(s[4 * c4 + 2]), __uint_as_float(s[4 * c4 + 3])),
                                    make_float2(kq[c4].z, kq[c4].w));
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

// 2^(C*v - C*m) for 16 columns -> 8 packed BF16 pairs, adding the weights to la / lb.
__device__ __forceinline__ void exp16(const uint32_t* s, float2 C2, float2 nCm, uint32_t* p, float2& la, float2& lb) {
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) {
        const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(s[4 * u4]), __uint_as_float(s[4 * u4 + 1])), C2, nCm);
        const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(s[4 * u4 + 2]), __uint_as_float(s[4 * u4 + 3])), C2, nCm);
        const float2 e01 = make_float2(fast_exp2(x01.x), fast_exp2(x01.y));
        const float2 e23 = make_float2(fast_exp2(x23.x), fast_exp2(x23.y));
        la = __fadd2_rn(la, e01);
        lb = __fadd2_rn(lb, e23);
        p[2 * u4] = pack_bf16x2(e01.x, e01.y);
        p[2 * u4 + 1] = pack_bf16x2(e23.x, e23.y);
    }
}

__device__ void softmax_role(const Ctx& c, int u, int quad, int lane) {
    const AttnArgs& a = *c.a;
    const int r = 32 * quad + lane;
    const int j = r / kHeadsPerKv, hq = r - j * kHeadsPerKv;
    const bool row_ok = j < c.nj;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const uint32_t tcol = c.tmem + u * kTileCols;
    const size_t row_off =
        ((size_t)(c.q_begin + j) * c.n_heads + (size_t)(c.h0 + u) * kHeadsPerKv + hq) * kHeadDim;
    {   // Q row r -> the tile's 128-byte swizzled K-major Q tile (row r, two 64-column halves)
        uint8_t* qt = c.base + kOffQ + u * kQTileBytes;
#pragma unroll 4
        for (int cc = 0; cc < 16; ++cc) {
            uint4 x = make_uint4(0, 0, 0, 0);
            if (row_ok) x = __ldg(reinterpret_cast<const uint4*>(a.q + row_off) + cc);
            const int half = cc >> 3, q16 = cc & 7;
            *reinterpret_cast<uint4*>(qt + half * (kQTileBytes / 2) + r * 128 + ((q16 ^ (r & 7)) << 4)) = x;
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tbar(c, u, TB_Q_READY));
    }
    // Scores are kept in units of q.k * (K scale); the constant sm_scale * log2(e)
    // is applied inside the exponent: p = 2^(C * (v - m)).
    const float C = c.kmul;
    const float thresh = kRescaleLog2 / C;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < c.n_chunks; ++t) {
        const int sb = t & 1, ts = t % kNS;
        const uint32_t tS = tcol + lane_base + kColS + 64 * sb;
        if (!(ok = wait_addr(c, bar(c, BAR_TAB_FULL + ts), (t / kNS) & 1))) break;   // the chunk's tables
        const RawTab* T = raw_tab(c, ts);
        const uint64_t selj = T->rowmask[j];
        if (!(ok = wait_addr(c, tbar(c, u, TB_S_FULL + sb), (t >> 1) & 1))) break;
        tc::fence_after_sync();
        // The 64 columns go in two halves of 32, each with its own online-softmax
        // step; P of half h lands in columns [16h, 16h + 16).  A 16-column slice
        // that none of the warp's queries selected is skipped (its P is zero).
        float alpha_tot = 1.f;
        bool any_need = false;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {     // not unrolled: keeps one half's registers live at a time
            uint32_t sv[32];
            tc::tmem_ld32(tS + 32 * h, sv);
            const uint32_t sel_lo = (uint32_t)(selj >> (32 * h)) & 0xFFFFu, sel_hi = (uint32_t)(selj >> (32 * h + 16)) & 0xFFFFu;
            const bool act_lo = __any_sync(0xffffffffu, sel_lo != 0), act_hi = __any_sync(0xffffffffu, sel_hi != 0);
            float4 kq[4];
            if (act_lo) {
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) kq[c4] = *reinterpret_cast<const float4*>(&T->ks[u][32 * h + 4 * c4]);
            }
            tc::tmem_wait_ld();
            float mx = -INFINITY, my = -INFINITY;    // two chains for more ILP
            if (act_lo) scale_mask16(&sv[0], sel_lo, kq, mx, my);
            if (act_hi) {
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) kq[c4] = *reinterpret_cast<const float4*>(&T->ks[u][32 * h + 16 + 4 * c4]);
                scale_mask16(&sv[16], sel_hi, kq, mx, my);
            }
            const float m_new = fmax3(m, mx, my);
            const bool need = (m != -INFINITY) && (m_new > m + thresh);
            const float m_use = (m == -INFINITY || need) ? m_new : m;
            const float alpha = need ? fast_exp2(C * (m - m_new)) : 1.f;
            const float m_sub = m_use == -INFINITY ? 0.f : m_use;
            uint32_t p[16];
            const float2 C2 = make_float2(C, C), nCm = make_float2(-C * m_sub, -C * m_sub);
            float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
            if (act_lo) {
                exp16(&sv[0], C2, nCm, &p[0], la, lb);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) p[v] = 0u;
            }
            if (act_hi) {
                exp16(&sv[16], C2, nCm, &p[8], la, lb);
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) p[8 + v] = 0u;
            }
            l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
            m = m_use;
            alpha_tot *= alpha;
            tc::tmem_st16(tS + 16 * h, p);
            tc::tmem_wait_st();
            if (h == 1 && __any_sync(0xffffffffu, need)) {
                // the first half's P was taken against the old max: bring it to the new one
                uint32_t q16[16];
                tc::tmem_ld16(tS, q16);
                tc::tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 16; ++v) q16[v] = pack_bf16x2(bf16_lo(q16[v]) * alpha, bf16_hi(q16[v]) * alpha);
                tc::tmem_st16(tS, q16);
                tc::tmem_wait_st();
            }
            any_need |= need;
        }
        if (__any_sync(0xffffffffu, any_need)) {
            // O must hold every earlier P V before it is rescaled: wait for PV(t-1)
            if (!(ok = wait_addr(c, tbar(c, u, TB_PV_DONE), (t - 1) & 1))) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int q8 = 0; q8 < 8; ++q8) {
                uint32_t o[16];
                tc::tmem_ld16(tcol + lane_base + kColO + 16 * q8, o);
                tc::tmem_wait_ld();
#pragma unroll
                for (int v = 0; v < 16; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha_tot);
                tc::tmem_st16(tcol + lane_base + kColO + 16 * q8, o);
            }
            tc::tmem_wait_st();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
            tc::mbar_arrive(tbar(c, u, TB_P_READY + sb));
            tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));   // done with this chunk's table
        }
    }
    float* out = a.out + row_off;
    if (c.n_chunks == 0) {
        if (row_ok)
            for (int v = 0; v < 32; ++v) reinterpret_cast<float4*>(out)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (!ok || !wait_addr(c, tbar(c, u, TB_O_DONE), 0)) return;
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t o[32];
        tc::tmem_ld32(tcol + lane_base + kColO + 32 * q4, o);
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
    c.h0 = kTiles * blockIdx.y;
    c.n_tiles = min(kTiles, a.n_kv - c.h0);
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
            tc::mbar_init(bar(c, BAR_TAB_EMPTY + s), (kConvWarps + 3) * c.n_tiles);   // loaders + softmax warps
        }
        for (int u = 0; u < kTiles; ++u) {
            for (int b = 0; b < kNB; ++b) {
                tc::mbar_init(tbar(c, u, TB_K_FULL + b), kConvWarps);
                tc::mbar_init(tbar(c, u, TB_K_EMPTY + b), 1);
                tc::mbar_init(tbar(c, u, TB_V_FULL + b), kConvWarps);
                tc::mbar_init(tbar(c, u, TB_V_EMPTY + b), 1);
            }
            for (int sb = 0; sb < 2; ++sb) {
                tc::mbar_init(tbar(c, u, TB_S_FULL + sb), 1);
                tc::mbar_init(tbar(c, u, TB_P_READY + sb), 3);
            }
            tc::mbar_init(tbar(c, u, TB_PV_DONE), 1);
            tc::mbar_init(tbar(c, u, TB_O_DONE), 1);
            tc::mbar_init(tbar(c, u, TB_Q_READY), 4);   // three softmax warps + the producer (pad rows)
        }
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
        const int u = (warp - kWarpConv0) / kConvWarps;
        if (u < c.n_tiles) converter_role(c, u, tid - kWarpConv0 * 32 - u * kConvThreads);
    } else {
        const int u = warp >> 2;
        if (u < c.n_tiles) softmax_role(c, u, warp & 3, lane);
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
    const dim3 grid((a.n_q + kGroup - 1) / kGroup, (a.n_kv + kTiles - 1) / kTiles);
    attn_tc_kernel<<<grid, kThreadsTc, kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
