// select_attn.cu -- per-position selected-cell attention without unions: every
// query position gathers its own selected cells (the baseline the union path
// replaces).
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary: the engine's default prompt path runs the decode
// kernel, every position gathering its own ~2,051 selected K/V cells; section
// Extra Notes times it against the union kernel at several union ratios.  The
// result is the same per-position softmax the union path computes; here it runs
// on the warp-level tensor path so that the comparison is between data-movement
// strategies, not between FP32 and tensor cores.  The same kernel serves decode
// over a batch of sequences (qsa_decode_attn): query i is sequence i's current
// position, with its own page table at page_table + i * pt_stride.
//
// One CTA of four warps per (query position i, KV head h): the warps each take a
// quarter of the position's list and merge their partial softmax states at the
// end (flash-decoding style: decode batches have few (query, KV head) items,
// and four CTAs' worth of warps per item fill the GPU in many waves).  The 12
// query heads are rows 0-11 of one m16 tile (rows 12-15 padding); the CTA keeps
// Q once in shared memory, and each warp reads its A fragments with ldmatrix.
// A warp walks its part of the list in steps of 16 cells:
//   * lanes 2c and 2c+1 resolve cell c -> page -> pool row in a register
//     pipeline (while step t is computed: the cells of step t+3 and the
//     page-table entries of step t+2 are loaded, and step t+1's K and V rows
//     are copied with 16-byte cp.async into a 2-deep INT8 stage ring, 16-byte
//     chunks XOR-swizzled by cell).  The two lanes copy the two halves of each
//     32-byte sector in the same instruction (with one lane per row, the halves
//     came from two instructions); the rows' K/V scales are loaded with the
//     copies and stored a step later, so no step waits on them;
//   * S = Q K^T with mma.sync m16n8k16 on FP16 operands (Q converted from BF16
//     once per CTA, exactly: rows far from FP16's range take a power-of-two
//     scaling, as in the union kernel): each lane's K operand is one 32-bit word
//     of the INT8 row (the head dimension is permuted inside every 16-wide k
//     step, for Q and K alike), converted exactly in registers (|int8| <= 128
//     fits FP16); the K scale (times sm_scale and log2 e) multiplies each score
//     column in FP32, unselected / masked cells are -inf, the online softmax
//     runs in the exp2 domain with the same lazy rescale as the union kernel
//     (the row-max shuffles and the rescale behind one warp vote), and
//     P = p * (V scale) enters O += P V as BF16; V also
//     goes from the INT8 stage straight into the B fragments (ldmatrix.trans of
//     byte pairs, the output columns permuted so that a lane's accumulators
//     cover four consecutive dims), so the kernel writes no operand tile.
#include <type_traits>

#include "qsa_common.cuh"

namespace qsa {
namespace {

constexpr int kSelWarps = 4;
constexpr int kSelThreads = 32 * kSelWarps;
constexpr int kStep = 16;                  // cells per step
constexpr int kStages = 2;                 // INT8 stage ring: copies run kStages - 1 steps ahead
constexpr float kSelRescaleLog2 = 32.f;    // lazy rescale threshold (exp2 domain), as in attn_tc.cu

// The (query, KV head)'s 12 query-head rows as FP16 (rows 12-15 zero), shared by
// the CTA's four warps: 256-byte rows, 16-byte chunks XOR-swizzled by (row & 7),
// each 16-wide k step in the permuted order the S fragments use (see below).
struct __align__(16) QTile {
    uint16_t q[16][kHeadDim];
    float rs[16];   // 2^e of each row's power-of-two scaling (1 for most rows)
};

struct __align__(16) WarpSmem {
    int8_t raw[kStages][2][kStep][kHeadDim];   // [stage][K|V][cell][d], 16-byte chunk c at stage_chunk(c, cell); 8 KB
    // scales of cells 2j, 2j+1 as one 16-byte entry {K, K, V, V} (K scale * sm_scale *
    // log2(e)); 0 for a masked cell
    float4 kvs[kStages][kStep / 2];
    uint32_t valid[kStages];                // bit 2c: cell c of the step is selected and resident
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// Position of 16-byte chunk c of a cell's 128-byte row in the INT8 stage: c XOR
// f(cell), f(cell) = 4 (cell & 1) + ((cell >> 1) & 3).  f takes 8 different
// values over 8 consecutive cells, so an ldmatrix over 8 cells at one chunk hits
// 8 bank groups; and two neighbouring cells differ in bit 2 of f, so the 16-byte
// K reads of two cells (chunks 0-3 or 4-7 of each) fill all 8 bank groups.
__device__ __forceinline__ uint32_t stage_chunk(int c, int cell) {
    return (uint32_t)(c ^ (((cell & 1) << 2) | ((cell >> 1) & 3)));
}

// Four INT8 values in a word -> BF16 pairs (bytes 0, 2) and (bytes 1, 3),
// exactly, in the way of int8x4_to_bf16.
__device__ __forceinline__ void int8x4_to_bf16_even_odd(uint32_t w, uint32_t& out02, uint32_t& out13) {
    const uint32_t l02 = __byte_perm(w, 0x4343u, 0x5240);   // [b0, 0x43, b2, 0x43]
    const uint32_t l13 = __byte_perm(w, 0x4343u, 0x5341);   // [b1, 0x43, b3, 0x43]
    out02 = bf16x2_sub(l02 & 0xFF7FFF7Fu, l02 & 0xFF80FF80u);
    out13 = bf16x2_sub(l13 & 0xFF7FFF7Fu, l13 & 0xFF80FF80u);
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kSelThreads, 4) select_attn_kernel(const SelArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    WarpSmem& s = reinterpret_cast<WarpSmem*>(smem_raw)[warp];
    QTile& qt = *reinterpret_cast<QTile*>(smem_raw + kSelWarps * sizeof(WarpSmem));
    // h-major: consecutive positions share cells
    const long long item = (long long)blockIdx.x;
    if (item >= (long long)a.n_q * a.n_kv) return;   // the CTA's warps share one item: all or none leave
    const int h = (int)(item / a.n_q), i = (int)(item - (long long)h * a.n_q);
    const int n_heads = a.n_kv * kHeadsPerKv;
    const float kmul = a.sm_scale * kLog2e;

    int cnt = __ldg(a.sel_count + i);
    if (cnt < 0 || cnt > a.sel_stride) {
        if (lane == 0 && warp == 0) report(a.dev_status, QSA_DEV_BAD_SEL_COUNT);
        cnt = cnt < 0 ? 0 : a.sel_stride;
    }
    // this warp's part of the list: whole 16-cell steps [first, first + n_steps)
    const int all_steps = (cnt + kStep - 1) / kStep;
    const int per_warp = (all_steps + kSelWarps - 1) / kSelWarps;
    const int first = min(all_steps, warp * per_warp);
    const int n_steps = min(all_steps, first + per_warp) - first;
    const int32_t* lst = a.sel + (size_t)i * a.sel_stride + first * kStep;
    cnt -= first * kStep;
    const int32_t* ptab = a.page_table + (size_t)i * a.pt_stride;   // this query's page table

    // ---- cell -> page -> row pipeline: lanes 2c and 2c + 1 both resolve cell c of a
    // step and copy its K and V rows, the even lane the first 16 bytes of every
    // 32-byte sector, the odd lane the second, so that each sector is requested
    // once, by one instruction; the even lane loads the K scale, the odd the V scale
    const int slot = lane >> 1, kv = lane & 1;
    auto load_cell = [&](int step) -> int {
        const int u = step * kStep + slot;
        return (step < n_steps && u < cnt) ? __ldg(lst + u) : -1;
    };
    // physical page (< 0 = masked: absent, bad or not resident); the entry is
    // checked against the pool when it is used, a step after its load
    auto resolve = [&](int cell) -> int {
        if (cell < 0) return -1;
        if ((cell >> 6) >= a.n_lpages) {
            report(a.dev_status, QSA_DEV_BAD_CELL);
            return -1;
        }
        return __ldg(ptab + (cell >> 6));
    };
    // Row copies of a step into stage st, and the load of the lane's scale (its
    // FP16 bits, 0 for a masked cell), which put_scale stores one step later, so
    // the load's latency is not waited for in the step that issues it.
    auto issue = [&](int cell, int page, int st) -> uint16_t {
        uint16_t sb = 0;
        if (page >= a.n_ppages) {
            report(a.dev_status, QSA_DEV_BAD_PAGE);
            page = -1;
        }
        const bool ok = page >= 0;
        if (ok) {
            const size_t row = ((size_t)page * a.n_kv + h) * kPage + (cell & (kPage - 1));
            const int8_t* ksrc = a.k_pool + row * kHeadDim + 16 * kv;
            const int8_t* vsrc = a.v_pool + row * kHeadDim + 16 * kv;
            const uint32_t kdst = smem_u32(&s.raw[st][0][slot][0]), vdst = smem_u32(&s.raw[st][1][slot][0]);
#pragma unroll
            for (int sec = 0; sec < 4; ++sec) {
                const uint32_t off = stage_chunk(2 * sec + kv, slot) << 4;
                cp_async16(kdst + off, ksrc + 32 * sec);
                cp_async16(vdst + off, vsrc + 32 * sec);
            }
            sb = __ldg((kv ? a.v_scale : a.k_scale) + row);
        }
        const uint32_t vm = __ballot_sync(0xffffffffu, ok && kv == 0);
        if (lane == 0) s.valid[st] = vm;
        return sb;
    };
    // A masked cell's scale is 0 (its score is -inf anyway; P is 0).
    auto put_scale = [&](uint16_t sb, int st) {
        const float sc = __half2float(__ushort_as_half(sb));
        reinterpret_cast<float*>(&s.kvs[st][slot >> 1])[2 * kv + (slot & 1)] = kv ? sc : sc * kmul;
    };

    // prologue: copies of steps 0 .. kStages-2 in flight (their scales stored
    // now); then the register pipeline holds the cells of step kStages-1
    // (resolved) and kStages
#pragma unroll 1
    for (int k = 0; k < kStages - 1; ++k) {
        const int c = load_cell(k);
        put_scale(issue(c, resolve(c), k), k);
        cp_async_commit();
    }
    int c1 = load_cell(kStages - 1), c2 = load_cell(kStages);
    int p1 = resolve(c1);
    uint16_t sb_next = 0;   // scale of step + kStages - 2 (loaded one step ago), stored at the next step's top

    // ---- Q (A operand of S, FP16), rows 0-11: the KV head's 12 query heads.  The
    // head dimension is permuted, for Q and K alike (a dot product does not
    // depend on the order of its terms): in k step kk = 4hk + k' (hk, k' < 4 ...),
    // the logical entries 2t, 2t+1, 2t+8, 2t+9 -- what lane (g, t) holds of an
    // m16n8k16 fragment -- are dims 64hk + 16t + 4k' .. +3.  So a lane's K operands
    // of four k steps are one 16-byte piece of the INT8 row (bytes 64hk + 16t ..
    // +15).  Thread t of the CTA stores row t >> 3, k step t & 7.
    // BF16 -> FP16 is exact for |q| in [2^-17, 2^16); a row whose largest |q| is
    // 2^14 or more, or below 2^-10, is stored times 2^-e (e puts that largest value
    // in [2^12, 2^13)), and its scores are multiplied back by 2^e, both exact: the
    // union kernel's rule, so both paths see the same FP16 Q.
    bool qscaled;
    {
        const int row = threadIdx.x >> 3, kk = threadIdx.x & 7;
        const bool live = row < kHeadsPerKv;
        const uint16_t* qsrc = a.q + ((size_t)i * n_heads + h * kHeadsPerKv + (live ? row : 0)) * kHeadDim +
                             64 * (kk >> 2) + 4 * (kk & 3);
        // logical pair (2t, 2t+1) is dims +16t, +16t+1; pair (2t+8, 2t+9) dims +16t+2, +16t+3
        uint32_t lg[8];
        float amax = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint2 x = live ? __ldg(reinterpret_cast<const uint2*>(qsrc + 16 * t)) : make_uint2(0u, 0u);
            lg[t] = x.x;
            lg[4 + t] = x.y;
            amax = fmax3(amax, fmaxf(fabsf(bf16_lo(x.x)), fabsf(bf16_hi(x.x))),
                         fmaxf(fabsf(bf16_lo(x.y)), fabsf(bf16_hi(x.y))));
        }
        // the row's 8 threads are 8 consecutive lanes
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;   // floor(log2 amax)
        // |e| <= 114, so 2^e and 2^-e are normal floats
        const int e = (amax > 0.f && (ex >= 14 || ex < -10)) ? min(max(ex - 12, -114), 114) : 0;
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
#pragma unroll
        for (int v = 0; v < 8; ++v) lg[v] = pack_f16x2(bf16_lo(lg[v]) * down, bf16_hi(lg[v]) * down);
        if (kk == 0) qt.rs[row] = __uint_as_float((uint32_t)(127 + e) << 23);
        qscaled = e != 0;
        uint8_t* qrow = reinterpret_cast<uint8_t*>(&qt.q[row][0]);
        *reinterpret_cast<uint4*>(qrow + (((2 * kk) ^ (row & 7)) << 4)) = make_uint4(lg[0], lg[1], lg[2], lg[3]);
        *reinterpret_cast<uint4*>(qrow + (((2 * kk + 1) ^ (row & 7)) << 4)) = make_uint4(lg[4], lg[5], lg[6], lg[7]);
    }
    qscaled = __syncthreads_or(qscaled) != 0;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int r0 = g4, r1 = g4 + 8;
    // ldmatrix x4 row addresses of the Q tile: lane l reads row (l & 7) + 8 ((l >> 3) & 1),
    // logical chunk 2 kk + (l >> 4)
    const int qr = (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t q_base = smem_u32(&qt.q[qr][0]);

    float o[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // ldmatrix row of lane l in the V stage: cell (l & 7) + 8 ((l >> 3) & 1), 16-byte chunk 2q + (l >> 4)
    const int vcell = (lane & 7) + 8 * ((lane >> 3) & 1);

    // The step loop, compiled twice: with and without the rows' power-of-two
    // score scaling, chosen once per CTA (no per-step test).
    auto walk = [&](auto scaled) {
#pragma unroll 1
        for (int step = 0; step < n_steps; ++step) {
            const int st = step % kStages;
            // pipeline: cells of step+kStages+1, page of step+kStages, copies of
            // step+kStages-1 (into the stage step-1 used), while step's copies land
            const int c3 = load_cell(step + kStages + 1);
            const int p2 = resolve(c2);
            // scales of step + kStages - 2 (its copies were issued one step ago; step 1's
            // were stored in the prologue), then step + kStages - 1's copies and scale load
            if (step > 0) put_scale(sb_next, (step + kStages - 2) % kStages);
            sb_next = issue(c1, p1, (step + kStages - 1) % kStages);
            cp_async_commit();
            cp_async_wait<kStages - 1>();
            __syncwarp();

            // S = Q K^T: 16 rows x 16 cells, K straight from the INT8 stage: lane (g, t)
            // of n tile nt reads, for k steps 4hk .. 4hk + 3, bytes 64hk + 16t .. +15 of
            // cell 8nt + g (one 16-byte load; one 32-bit word per k step) and converts
            // each word exactly to two FP16 pairs.  Even and odd k steps accumulate
            // separately (two shorter dependency chains).
            float sc[2][4];
            {
                // lane (g, t): the 16-byte pieces t and 4 + t of cells g and 8 + g (k steps 0-3, 4-7)
                uint4 kw[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int cell = nt * 8 + g4;
                    const uint8_t* krow = reinterpret_cast<const uint8_t*>(&s.raw[st][0][cell][0]);
                    kw[nt][0] = *reinterpret_cast<const uint4*>(krow + (stage_chunk(t4, cell) << 4));
                    kw[nt][1] = *reinterpret_cast<const uint4*>(krow + (stage_chunk(4 + t4, cell) << 4));
                }
                float acc[2][2][4] = {};   // [n tile][k step parity]: two shorter dependency chains each
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t qa[4];
                    ldsm_x4(q_base + (((2 * kk + (lane >> 4)) ^ (qr & 7)) << 4), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const uint4 v4 = kw[nt][kk >> 2];
                        const uint32_t w = (kk & 3) == 0 ? v4.x : (kk & 3) == 1 ? v4.y : (kk & 3) == 2 ? v4.z : v4.w;
                        uint32_t b0, b1;
                        int8x4_to_f16(w, b0, b1);
                        mma_f16(acc[nt][kk & 1], qa, b0, b1);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int v = 0; v < 4; ++v) sc[nt][v] = acc[nt][0][v] + acc[nt][1][v];
                if constexpr (decltype(scaled)::value) {   // rows stored times 2^-e: scores times 2^e (exact)
                    const float rs0 = qt.rs[r0], rs1 = qt.rs[r1];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        sc[nt][0] *= rs0;
                        sc[nt][1] *= rs0;
                        sc[nt][2] *= rs1;
                        sc[nt][3] *= rs1;
                    }
                }
            }
            // column scale (log2 domain), masked cells -inf
            const uint32_t vm = s.valid[st];
            float mx0 = -INFINITY, mx1 = -INFINITY;
            float2 vcs[2];   // V scales of the lane's columns, for P below
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int c = nt * 8 + 2 * t4;
                const float4 kv4 = s.kvs[st][c >> 1];
                const float2 kc = make_float2(kv4.x, kv4.y);
                vcs[nt] = make_float2(kv4.z, kv4.w);
                const bool okA = (vm >> (2 * c)) & 1u, okB = (vm >> (2 * c + 2)) & 1u;
                sc[nt][0] = okA ? sc[nt][0] * kc.x : -INFINITY;
                sc[nt][1] = okB ? sc[nt][1] * kc.y : -INFINITY;
                sc[nt][2] = okA ? sc[nt][2] * kc.x : -INFINITY;
                sc[nt][3] = okB ? sc[nt][3] * kc.y : -INFINITY;
                mx0 = fmax3(mx0, sc[nt][0], sc[nt][1]);
                mx1 = fmax3(mx1, sc[nt][2], sc[nt][3]);
            }
            // lazy rescale: the running max only moves when a score exceeds it by 2^32 in p
            // (a row's first valid score does too: -inf + 32 is -inf).  A lane's own scores
            // decide whether its row can move, so one warp vote skips the row-max shuffles
            // and the rescale in every step where no row moves, with the same result.
            float al0 = 1.f, al1 = 1.f;
            if (__any_sync(0xffffffffu, mx0 > m0 + kSelRescaleLog2 || mx1 > m1 + kSelRescaleLog2)) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const bool need0 = m0 != -INFINITY && mn0 > m0 + kSelRescaleLog2;
                const bool need1 = m1 != -INFINITY && mn1 > m1 + kSelRescaleLog2;
                if (need0) al0 = fast_exp2(m0 - mn0);
                if (need1) al1 = fast_exp2(m1 - mn1);
                if (m0 == -INFINITY || need0) m0 = mn0;
                if (m1 == -INFINITY || need1) m1 = mn1;
#pragma unroll
                for (int dt = 0; dt < 16; ++dt) {   // al = 1 leaves a row as it is
                    o[dt][0] *= al0;
                    o[dt][1] *= al0;
                    o[dt][2] *= al1;
                    o[dt][3] *= al1;
                }
            }
            const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
            float ps0 = 0.f, ps1 = 0.f;
            uint32_t af[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 vc = vcs[nt];
                const float e0 = fast_exp2(sc[nt][0] - mu0), e1 = fast_exp2(sc[nt][1] - mu0);
                const float e2 = fast_exp2(sc[nt][2] - mu1), e3 = fast_exp2(sc[nt][3] - mu1);
                ps0 += e0 + e1;
                ps1 += e2 + e3;
                af[2 * nt] = pack_bf16x2(e0 * vc.x, e1 * vc.y);       // row r0: A fragment a0 / a2
                af[2 * nt + 1] = pack_bf16x2(e2 * vc.x, e3 * vc.y);   // row r1: a1 / a3
            }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
            // O += P V: the 16 cells are one k16 step, V straight from the INT8 stage.
            // ldmatrix.trans on byte pairs: for the 32 dims 32q .. 32q+31, lane (g, t)
            // gets, of cells 2t, 2t+1 (and 2t+8, 2t+9), the pairs of dims 32q + 2g, +1
            // and 32q + 16 + 2g, +1.  Bytes 0 and 2 of a word are the two cells' values
            // of the even dim, bytes 1 and 3 of the odd one: the B operands of two n
            // tiles whose column g is dim 32q + 2g (tile "even") and 32q + 2g + 1
            // ("odd").  So O tile 4q + 2h + e holds dims 32q + 16h + 2n + e at column n,
            // and a lane's accumulators of rows g and g + 8 cover dims 32q + 16h + 4t
            // .. +3.
            {
                const uint32_t vrow = smem_u32(&s.raw[st][1][vcell][0]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t r[4];
                    ldsm_x4_t(vrow + (stage_chunk(2 * q + (lane >> 4), vcell) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t e0, d0, e1, d1;
                        int8x4_to_bf16_even_odd(r[2 * hh], e0, d0);       // cells 2t, 2t+1
                        int8x4_to_bf16_even_odd(r[2 * hh + 1], e1, d1);   // cells 2t+8, 2t+9
                        mma_bf16(o[4 * q + 2 * hh], af, e0, e1);
                        mma_bf16(o[4 * q + 2 * hh + 1], af, d0, d1);
                    }
                }
            }
            __syncwarp();   // the stage is refilled next step
            c1 = c2;
            c2 = c3;
            p1 = p2;
        }
    };
    if (qscaled) walk(std::true_type{});
    else walk(std::false_type{});
    cp_async_wait<0>();   // nothing left in flight when the warp exits

    // ---- O / l for rows 0-11
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    {
        // Merge the four warps' partial states.  Warp w's O and l are relative to
        // its own running max m_w; the row's result is sum_w 2^(m_w - M) O_w over
        // sum_w 2^(m_w - M) l_w with M = max_w m_w (a warp with no valid cell has
        // m_w = -inf and weight 0).  The stage buffers are free now.
        __syncthreads();
        float* po = reinterpret_cast<float*>(smem_raw);                  // [warp][16 rows][128]
        float* pm = po + kSelWarps * 16 * kHeadDim;                      // [warp][16 rows]
        float* pl = pm + kSelWarps * 16;                                 // [warp][16 rows]
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d = 32 * q + 16 * hh + 4 * t4, e = 4 * q + 2 * hh;
                *reinterpret_cast<float4*>(po + (warp * 16 + r0) * kHeadDim + d) =
                    make_float4(o[e][0], o[e + 1][0], o[e][1], o[e + 1][1]);
                *reinterpret_cast<float4*>(po + (warp * 16 + r1) * kHeadDim + d) =
                    make_float4(o[e][2], o[e + 1][2], o[e][3], o[e + 1][3]);
            }
        if (t4 == 0) {
            pm[warp * 16 + r0] = m0;
            pm[warp * 16 + r1] = m1;
            pl[warp * 16 + r0] = l0;
            pl[warp * 16 + r1] = l1;
        }
        __syncthreads();
        // thread t: rows 0-11, 4 consecutive dims each step
        for (int e = threadIdx.x; e < kHeadsPerKv * (kHeadDim / 4); e += kSelThreads) {
            const int row = e / (kHeadDim / 4), d = 4 * (e - row * (kHeadDim / 4));
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kSelWarps; ++w) M = fmaxf(M, pm[w * 16 + row]);
            float L = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kSelWarps; ++w) {
                const float mw = pm[w * 16 + row];
                const float wt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                L += wt * pl[w * 16 + row];
                const float4 ow = *reinterpret_cast<const float4*>(po + (w * 16 + row) * kHeadDim + d);
                acc.x += wt * ow.x;
                acc.y += wt * ow.y;
                acc.z += wt * ow.z;
                acc.w += wt * ow.w;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            float* dst = a.out + ((size_t)i * n_heads + h * kHeadsPerKv + row) * kHeadDim + d;
            *reinterpret_cast<float4*>(dst) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
    }
}

}  // namespace

cudaError_t launch_select_attn(const SelArgs& a, cudaStream_t stream) {
    const int smem = (int)(kSelWarps * sizeof(WarpSmem) + sizeof(QTile));
    cudaError_t e = cudaFuncSetAttribute(select_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long items = (long long)a.n_q * a.n_kv;
    const unsigned grid = (unsigned)items;
    select_attn_kernel<<<grid, kSelThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
