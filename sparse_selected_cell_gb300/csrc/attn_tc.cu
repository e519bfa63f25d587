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
// One CTA per (group g, KV head h); 9 warps, two CTAs per SM:
//   warps 0-2  softmax: thread r owns query-head row r = j*12 + hq (TMEM lane r).
//              Loads its Q row into TMEM once; per chunk reads S from TMEM,
//              scales each column by K scale * sm_scale * log2(e), masks cells
//              its query did not select, runs the online softmax in the exp2
//              domain (the running max only moves when it grows by more than
//              2^8, and O is rescaled in TMEM only then), writes P as BF16 into
//              the S columns, and finally normalises O and stores it.
//   warp 3     producer: union entries -> page table -> per-chunk tables in a
//              4-deep ring (pool row of each cell, scales, one 64-bit selection
//              mask per query built with warp ballots), three chunks of loads in
//              flight.  Also zeroes the TMEM pad rows.
//   warps 4-7  loaders/converters: 16-byte loads of the INT8 K and V rows
//              (issued one chunk ahead into registers), dequantised straight into
//              BF16 operand tiles in the 128-byte swizzled layouts the tensor core
//              reads (K exact, V times its scale), double-buffered.
//   warp 8     MMA issuer (one thread): S = Q K^T (A = Q from TMEM, B = K tile,
//              M=128 N=64 K=128) and O += P V (A = P from TMEM, B = V tile,
//              M=128 N=128 K=64), completion tracked with tcgen05.commit.
// Rows 96-127 of the M=128 tiles are padding (Q rows zero, never stored).
// TMEM columns: Q [0,64) as packed BF16 pairs, S/P [64,128), O [128,256).
// Every wait is bounded in time; a wait that runs out sets a CTA-wide abort
// flag and QSA_DEV_WAIT_TIMEOUT, every role then stops, the MMA issuer drains
// the MMAs it started, and the CTA frees its Tensor Memory and exits.
#include "qsa_common.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace {

constexpr int kThreadsTc = 288;
constexpr int kWarpProducer = 3;
constexpr int kWarpConv0 = 4;
constexpr int kWarpMma = 8;
constexpr int kNS = 4;                 // per-chunk table ring
constexpr int kNB = 2;                 // BF16 operand buffers
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColQ = 0, kColS = 64, kColO = 128;
constexpr float kRescaleLog2 = 8.f;    // lazy rescale threshold (exp2 domain)
constexpr uint64_t kWaitNs = 1000000000ull;

struct RawTab {
    int32_t row[kChunk];    // pool row (page * n_kv + h) * 64 + cell % 64; -1 for a masked cell
    float ks[kChunk];       // K scale * sm_scale * log2(e); 0 for a masked cell
    float vs[kChunk];       // V scale; 0 for a masked cell
    uint64_t rowmask[8];    // bit c: query j of the group selected resident cell c
};
struct BfTab {
    float ks[kChunk];
    uint64_t rowmask[8];
};

constexpr uint32_t kTileBytes = kChunk * kHeadDim * 2;         // 16 KB BF16 tile (two 64-column halves)
constexpr uint32_t kOffKb = 0;
constexpr uint32_t kOffVb = kOffKb + kNB * kTileBytes;
constexpr uint32_t kOffRawTab = kOffVb + kNB * kTileBytes;
constexpr uint32_t kOffBfTab = kOffRawTab + kNS * (uint32_t)sizeof(RawTab);
constexpr uint32_t kOffBars = (kOffBfTab + kNB * (uint32_t)sizeof(BfTab) + 7u) & ~7u;
enum {
    BAR_TAB_FULL = 0,
    BAR_TAB_EMPTY = BAR_TAB_FULL + kNS,
    BAR_BF_FULL = BAR_TAB_EMPTY + kNS,
    BAR_BF_EMPTY = BAR_BF_FULL + kNB,
    BAR_S_FULL = BAR_BF_EMPTY + kNB,
    BAR_P_READY,
    BAR_O_DONE,
    BAR_Q_READY,
    BAR_DRAIN,
    NUM_BARS
};
constexpr uint32_t kOffMisc = kOffBars + NUM_BARS * 8;           // tmem base, abort flag, zero flag
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;                // + alignment slack

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
__device__ __forceinline__ BfTab* bf_tab(const Ctx& c, int b) { return reinterpret_cast<BfTab*>(c.base + kOffBfTab) + b; }

__device__ __forceinline__ bool wait_bar(const Ctx& c, int i, uint32_t parity) {
    if (tc::mbar_wait(bar(c, i), parity, c.abort_flag, kWaitNs)) return true;
    report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------ producer
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

// Pool row of each entry (-1 = masked), from the entries and their page-table values.
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

__device__ __forceinline__ void load_scales(const Ctx& c, const int (&row)[2], uint16_t (&ks)[2], uint16_t (&vs)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        ks[k] = row[k] >= 0 ? __ldg(c.a->k_scale + row[k]) : (uint16_t)0;
        vs[k] = row[k] >= 0 ? __ldg(c.a->v_scale + row[k]) : (uint16_t)0;
    }
}

// Three chunks of dependent loads stay in flight: entries of chunk i+3, page
// table of chunk i+2, scales of chunk i+1, while chunk i's table is written.
__device__ void producer_role(const Ctx& c, int lane) {
    {   // zero the Q pad rows (TMEM lanes 96-127) once
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0u;
        const uint32_t t = c.tmem + (96u << 16) + kColQ;
        tc::tmem_st32(t, z);
        tc::tmem_st32(t + 32, z);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_Q_READY));
    }
    if (c.n_chunks == 0) return;
    Entries e0 = load_entries(c, 0, lane), e1 = load_entries(c, 1, lane), e2 = load_entries(c, 2, lane);
    int pg0[2], pg1[2], r0[2];
    load_pages(c, e0, pg0);
    load_pages(c, e1, pg1);
    pool_rows(c, e0, pg0, r0);
    uint16_t ks0[2], vs0[2];
    load_scales(c, r0, ks0, vs0);
    for (int i = 0; i < c.n_chunks; ++i) {
        const int ts = i % kNS;
        const Entries e3 = load_entries(c, i + 3, lane);
        int pg2[2], r1[2];
        load_pages(c, e2, pg2);
        pool_rows(c, e1, pg1, r1);
        uint16_t ks1[2], vs1[2];
        load_scales(c, r1, ks1, vs1);
        if (!wait_bar(c, BAR_TAB_EMPTY + ts, ((i / kNS) & 1) ^ 1)) break;
        RawTab* T = raw_tab(c, ts);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool ok = r0[k] >= 0;
            T->row[lane + 32 * k] = r0[k];
            T->ks[lane + 32 * k] = ok ? __half2float(__ushort_as_half(ks0[k])) * c.kmul : 0.f;
            T->vs[lane + 32 * k] = ok ? __half2float(__ushort_as_half(vs0[k])) : 0.f;
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
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            pg1[k] = pg2[k];
            r0[k] = r1[k];
            ks0[k] = ks1[k];
            vs0[k] = vs1[k];
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

// Thread ct owns rows (ct >> 3) + 16k, k = 0..3, 16-byte segment ct & 7, of both K and V.
__device__ __forceinline__ void load_rows(const Ctx& c, const RawTab* T, int ct, uint4 (&kx)[4], uint4 (&vx)[4]) {
    const int seg = ct & 7;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = T->row[(ct >> 3) + 16 * k];
        kx[k] = make_uint4(0, 0, 0, 0);
        vx[k] = make_uint4(0, 0, 0, 0);
        if (r >= 0) {
            const size_t off = (size_t)r * kHeadDim + seg * 16;
            kx[k] = ldg_stream(c.a->k_pool + off);
            vx[k] = ldg_stream(c.a->v_pool + off);
        }
    }
}

__device__ void converter_role(const Ctx& c, int ct) {
    const int lane = ct & 31;
    if (c.n_chunks == 0) return;
    uint4 ck[4], cv[4];
    if (!wait_bar(c, BAR_TAB_FULL + 0, 0)) return;
    load_rows(c, raw_tab(c, 0), ct, ck, cv);
    const int seg = ct & 7;
    for (int i = 0; i < c.n_chunks; ++i) {
        const int ts = i % kNS, b = i % kNB;
        uint4 nk[4], nv[4];
        if (i + 1 < c.n_chunks) {     // next chunk's rows in flight while this one is converted
            if (!wait_bar(c, BAR_TAB_FULL + (i + 1) % kNS, ((i + 1) / kNS) & 1)) break;
            load_rows(c, raw_tab(c, (i + 1) % kNS), ct, nk, nv);
        }
        if (!wait_bar(c, BAR_BF_EMPTY + b, ((i / kNB) & 1) ^ 1)) break;
        const RawTab* T = raw_tab(c, ts);
        uint8_t* kb = c.base + kOffKb + b * kTileBytes;
        uint8_t* vb = c.base + kOffVb + b * kTileBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int row = (ct >> 3) + 16 * k;
            const uint32_t q = (uint32_t)(seg & 3) * 2, x = (uint32_t)(row & 7);
            const uint32_t tile = (uint32_t)(seg >> 2) * (kTileBytes / 2) + (uint32_t)row * 128;
            const uint32_t o_lo = tile + ((q ^ x) << 4), o_hi = tile + (((q + 1) ^ x) << 4);
            uint4 lo, hi;
            int8x16_to_bf16(ck[k], lo, hi);
            *reinterpret_cast<uint4*>(kb + o_lo) = lo;
            *reinterpret_cast<uint4*>(kb + o_hi) = hi;
            dequant16(cv[k], T->vs[row], lo, hi);
            *reinterpret_cast<uint4*>(vb + o_lo) = lo;
            *reinterpret_cast<uint4*>(vb + o_hi) = hi;
        }
        BfTab* B = bf_tab(c, b);
        if (ct < kChunk) B->ks[ct] = T->ks[ct];
        if (ct < 8) B->rowmask[ct] = T->rowmask[ct];
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            tc::mbar_arrive(bar(c, BAR_TAB_EMPTY + ts));
            tc::mbar_arrive(bar(c, BAR_BF_FULL + b));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ck[k] = nk[k];
            cv[k] = nv[k];
        }
    }
}

// ------------------------------------------------------------------ MMA issuer
__device__ void mma_role(const Ctx& c) {
    constexpr uint32_t idS = tc::idesc_bf16(128, kChunk, false, false);    // B = K tile, K-major
    constexpr uint32_t idO = tc::idesc_bf16(128, kHeadDim, false, true);   // B = V tile, MN-major
    const uint32_t kb_u = c.base_u + kOffKb, vb_u = c.base_u + kOffVb;
    const uint32_t tS = c.tmem + kColS, tQ = c.tmem + kColQ, tO = c.tmem + kColO;
    auto issue_pv = [&](int i) {
        const int bp = i % kNB;
#pragma unroll
        for (int k = 0; k < kChunk / 16; ++k)
            tc::mma_ts(tO, tS + 8 * k, tc::smem_desc(vb_u + bp * kTileBytes + k * 2048, 8192, 1024, 2), idO,
                       (i > 0 || k > 0) ? 1u : 0u);
        tc::commit(bar(c, BAR_BF_EMPTY + bp));
    };
    bool ok = c.n_chunks > 0 && wait_bar(c, BAR_Q_READY, 0);
    if (ok) {
        tc::fence_after_sync();
        for (int i = 0; i < c.n_chunks && ok; ++i) {
            const int b = i % kNB;
            if (!(ok = wait_bar(c, BAR_BF_FULL + b, (i / kNB) & 1))) break;
            tc::fence_after_sync();
            if (i > 0) {
                if (!(ok = wait_bar(c, BAR_P_READY, (i - 1) & 1))) break;
                tc::fence_after_sync();
                issue_pv(i - 1);
            }
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k)
                tc::mma_ts(tS, tQ + 8 * k,
                           tc::smem_desc(kb_u + b * kTileBytes + (k >> 2) * (kTileBytes / 2) + (k & 3) * 32, 16, 1024, 2),
                           idS, k > 0 ? 1u : 0u);
            tc::commit(bar(c, BAR_S_FULL));
        }
        if (ok && (ok = wait_bar(c, BAR_P_READY, (c.n_chunks - 1) & 1))) {
            tc::fence_after_sync();
            issue_pv(c.n_chunks - 1);
            tc::commit(bar(c, BAR_O_DONE));
        }
    }
    // every MMA issued above must be complete before Tensor Memory is released
    tc::commit(bar(c, BAR_DRAIN));
    if (!tc::mbar_wait_drain(bar(c, BAR_DRAIN), 0, kWaitNs)) report(c.a->dev_status, QSA_DEV_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ softmax
__device__ void softmax_role(const Ctx& c, int r, int warp, int lane) {
    const AttnArgs& a = *c.a;
    const int j = r / kHeadsPerKv, hq = r - j * kHeadsPerKv;
    const bool row_ok = j < c.nj;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const size_t row_off = ((size_t)(c.q_begin + j) * c.n_heads + (size_t)c.h * kHeadsPerKv + hq) * kHeadDim;
    {   // Q row -> TMEM columns [0, 64) as packed BF16 pairs
        uint32_t qv[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                uint4 x = make_uint4(0, 0, 0, 0);
                if (row_ok) x = __ldg(reinterpret_cast<const uint4*>(a.q + row_off) + half * 8 + v);
                qv[4 * v] = x.x; qv[4 * v + 1] = x.y; qv[4 * v + 2] = x.z; qv[4 * v + 3] = x.w;
            }
            tc::tmem_st32(c.tmem + lane_base + kColQ + 32 * half, qv);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_Q_READY));
    }
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < c.n_chunks; ++i) {
        const int b = i % kNB;
        if (!(ok = wait_bar(c, BAR_S_FULL, i & 1))) break;
        tc::fence_after_sync();
        uint32_t s[64];
        tc::tmem_ld32(c.tmem + lane_base + kColS, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tc::tmem_ld32(c.tmem + lane_base + kColS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tc::tmem_wait_ld();
        if (!(ok = wait_bar(c, BAR_BF_FULL + b, (i / kNB) & 1))) break;   // acquire the chunk's tables
        const BfTab* T = bf_tab(c, b);
        const uint64_t mk = T->rowmask[j];
        float mx = -INFINITY;
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
            const float4 kq = *reinterpret_cast<const float4*>(&T->ks[4 * c4]);
            const float kk[4] = {kq.x, kq.y, kq.z, kq.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int col = 4 * c4 + t;
                const float v = ((mk >> col) & 1ull) ? __uint_as_float(s[col]) * kk[t] : -INFINITY;
                s[col] = __float_as_uint(v);
                mx = fmaxf(mx, v);
            }
        }
        const float m_new = fmaxf(m, mx);
        const bool need = (m != -INFINITY) && (m_new > m + kRescaleLog2);
        const float m_use = (m == -INFINITY || need) ? m_new : m;
        const float alpha = need ? fast_exp2(m - m_new) : 1.f;
        const float m_sub = m_use == -INFINITY ? 0.f : m_use;
        uint32_t p[32];
        float lsum = 0.f;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            p[t] = pack_bf16x2(fast_exp2(__uint_as_float(s[2 * t]) - m_sub),
                               fast_exp2(__uint_as_float(s[2 * t + 1]) - m_sub));
            lsum += bf16_lo(p[t]) + bf16_hi(p[t]);
        }
        l = l * alpha + lsum;
        m = m_use;
        tc::tmem_st32(c.tmem + lane_base + kColS, p);
        if (__any_sync(0xffffffffu, need)) {   // O is stable: the previous P V finished before S was ready
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t o[32];
                tc::tmem_ld32(c.tmem + lane_base + kColO + 32 * q4, o);
                tc::tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                tc::tmem_st32(c.tmem + lane_base + kColO + 32 * q4, o);
            }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(c, BAR_P_READY));
    }
    float* out = a.out + row_off;
    if (c.n_chunks == 0) {
        if (row_ok)
            for (int v = 0; v < 32; ++v) reinterpret_cast<float4*>(out)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (!ok || !wait_bar(c, BAR_O_DONE, 0)) return;
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t o[32];
        tc::tmem_ld32(c.tmem + lane_base + kColO + 32 * q4, o);
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

__global__ void __launch_bounds__(kThreadsTc, 2) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
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
            tc::mbar_init(bar(c, BAR_TAB_EMPTY + s), 4);
        }
        for (int b = 0; b < kNB; ++b) {
            tc::mbar_init(bar(c, BAR_BF_FULL + b), 4);
            tc::mbar_init(bar(c, BAR_BF_EMPTY + b), 1);
        }
        tc::mbar_init(bar(c, BAR_S_FULL), 1);
        tc::mbar_init(bar(c, BAR_P_READY), 3);
        tc::mbar_init(bar(c, BAR_O_DONE), 1);
        tc::mbar_init(bar(c, BAR_Q_READY), 4);
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

    if (warp < kWarpProducer) {
        softmax_role(c, tid, warp, lane);
    } else if (warp == kWarpProducer) {
        producer_role(c, lane);
    } else if (warp < kWarpMma) {
        converter_role(c, tid - kWarpConv0 * 32);
    } else if (lane == 0) {
        mma_role(c);
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
