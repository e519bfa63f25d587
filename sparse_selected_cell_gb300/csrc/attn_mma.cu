// attn_mma.cu -- union attention on the warp-level tensor path (mma.sync
// m16n8k16, BF16 in, FP32 accumulate).  Kept as the legacy-path comparison for
// the tcgen05 kernel in attn_tc.cu; same contract, same results up to rounding.
//
// Source: "sycl: prompt attention over 8-query selection unions on XMX" (Strata
// PR #2808), section Summary: one work-group per (8 positions, KV head) covers
// 96 rows (8 positions x 12 heads); the INT8 K/V of each 64-cell chunk of the
// union is dequantised once; S = Q K^T and O += P V with FP32 sums; in the
// online softmax a cell is -inf for the positions that did not select it.
//
// Layout per CTA (group g, KV head h): 6 warps x 16 rows.  Row r = j*12 + hq
// (j = query within the group, hq = query head within the KV head).  Per chunk:
//   * warps 0-1 (one thread per union entry) walk a 3-deep register pipeline:
//     union entry -> page table -> scales, and issue 16-byte cp.async copies of
//     the K and V rows into a double-buffered INT8 stage;
//   * all threads dequantise the stage to BF16 into XOR-swizzled shared memory:
//     K exactly (int8 values are BF16-exact), V times its FP16 scale;
//   * each warp computes S = Q K^T from register-resident Q fragments, scales
//     each score column by its K scale * sm_scale * log2(e) in FP32, masks,
//     runs the online softmax in the exp2 domain and accumulates O += P V.
// Keeping K exact leaves the logits free of BF16 rounding, which matters when
// the softmax is peaked (large |q . k|).
#include "qsa_common.cuh"

namespace qsa {
namespace {

constexpr int kWarps = 6;
constexpr int kThreads = kWarps * 32;

struct __align__(16) SmemMma {
    int8_t raw[2][2][kChunk][kHeadDim];         // [stage][K|V][cell][d]  32 KB
    uint16_t kb[kChunk][kHeadDim];              // bf16 K', 256-B rows, 16-B chunks XOR (cell & 7)
    uint16_t vb[kChunk][kHeadDim];              // bf16 V'
    float ks[2][kChunk];                        // K scale * sm_scale * log2(e); 0 = invalid cell
    float vs[2][kChunk];                        // V scale; 0 = invalid cell
    uint8_t mask[2][kChunk];                    // membership byte; 0 = invalid cell
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `chunk` (0..15) of bf16 row `cell`
__device__ __forceinline__ uint32_t swz(int cell, int chunk) {
    return (uint32_t)(cell * 256 + ((chunk ^ (cell & 7)) << 4));
}

// One union entry's walk towards its K/V rows (thread t < 64 owns entry chunk*64 + t).
struct Entry {
    bool present;  // a union entry exists for this slot
    int cell;
    int mask;
    int page;      // physical page after the page-table step; -1 = masked
};

__global__ void __launch_bounds__(kThreads, 2)
attn_mma_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SmemMma& s = *reinterpret_cast<SmemMma*>(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.x, h = blockIdx.y;
    const int n_heads = a.n_kv * kHeadsPerKv;
    const int q_begin = g * kGroup;
    const int nj = min(kGroup, a.n_q - q_begin);

    int U = __ldg(a.union_count + g);
    if (U < 0 || U > a.union_stride) {
        if (tid == 0) report(a.dev_status, QSA_DEV_BAD_UNION_COUNT);
        U = U < 0 ? 0 : a.union_stride;
    }
    const int n_chunks = (U + kChunk - 1) / kChunk;
    const int32_t* ucell = a.union_cells + (size_t)g * a.union_stride;
    const uint8_t* umask = a.union_mask + (size_t)g * a.union_stride;
    const float kmul = a.sm_scale * kLog2e;

    // ---- union-entry pipeline (threads 0..63) ----
    auto load_entry = [&](int chunk) {
        Entry e{false, 0, 0, -1};
        const int u = chunk * kChunk + tid;
        if (tid < kChunk && chunk < n_chunks && u < U) {
            e.present = true;
            e.cell = __ldg(ucell + u);
            e.mask = __ldg(umask + u);
        }
        return e;
    };
    auto resolve = [&](Entry& e) {     // page-table step
        e.page = -1;
        if (!e.present) return;
        if (e.cell < 0) { report(a.dev_status, QSA_DEV_BAD_CELL); return; }
        const int lp = e.cell >> 6;
        if (lp >= a.n_lpages) { report(a.dev_status, QSA_DEV_BAD_CELL); return; }
        int pp = __ldg(a.page_table + lp);
        if (pp >= a.n_ppages) { report(a.dev_status, QSA_DEV_BAD_PAGE); pp = -1; }
        e.page = pp;
    };
    auto row_of = [&](const Entry& e) -> size_t {
        return ((size_t)e.page * a.n_kv + h) * kPage + (e.cell & (kPage - 1));
    };
    auto issue_copy = [&](const Entry& e, int stage) {
        if (tid >= kChunk || e.page < 0) return;
        const size_t r = row_of(e) * kHeadDim;
        const uint32_t dk = smem_u32(&s.raw[stage][0][tid][0]);
        const uint32_t dv = smem_u32(&s.raw[stage][1][tid][0]);
#pragma unroll
        for (int seg = 0; seg < 8; ++seg) {
            cp_async16(dk + seg * 16, a.k_pool + r + seg * 16);
            cp_async16(dv + seg * 16, a.v_pool + r + seg * 16);
        }
    };
    auto write_table = [&](const Entry& e, int stage, float ksv, float vsv) {
        if (tid >= kChunk) return;
        const bool ok = e.page >= 0;
        s.ks[stage][tid] = ok ? ksv * kmul : 0.f;
        s.vs[stage][tid] = ok ? vsv : 0.f;
        s.mask[stage][tid] = ok ? (uint8_t)e.mask : 0;
    };
    auto load_scales = [&](const Entry& e, float& ksv, float& vsv) {
        ksv = 0.f; vsv = 0.f;
        if (tid < kChunk && e.page >= 0) {
            const size_t r = row_of(e);
            ksv = __half2float(__ushort_as_half(__ldg(a.k_scale + r)));
            vsv = __half2float(__ushort_as_half(__ldg(a.v_scale + r)));
        }
    };

    Entry e1, e2, e3;
    float ks1, vs1;
    {
        Entry e0 = load_entry(0);
        e1 = load_entry(1);
        e2 = load_entry(2);
        resolve(e0);
        resolve(e1);
        float ks0, vs0;
        load_scales(e0, ks0, vs0);
        issue_copy(e0, 0);
        write_table(e0, 0, ks0, vs0);
    }
    cp_async_commit();

    // ---- Q fragments (A operand, 16 rows x 128 per warp) ----
    const int g4 = lane >> 2, t4 = lane & 3;
    const int r0 = warp * 16 + g4, r1 = r0 + 8;
    const int j0 = r0 / kHeadsPerKv, j1 = r1 / kHeadsPerKv;
    const bool v0 = j0 < nj, v1 = j1 < nj;
    const uint16_t* q0p = a.q + ((size_t)(q_begin + j0) * n_heads + h * kHeadsPerKv + r0 % kHeadsPerKv) * kHeadDim;
    const uint16_t* q1p = a.q + ((size_t)(q_begin + j1) * n_heads + h * kHeadsPerKv + r1 % kHeadsPerKv) * kHeadDim;
    uint32_t qa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int d = kk * 16 + 2 * t4;
        qa[kk][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q0p + d)) : 0u;
        qa[kk][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q1p + d)) : 0u;
        qa[kk][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(q0p + d + 8)) : 0u;
        qa[kk][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(q1p + d + 8)) : 0u;
    }

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const uint32_t kb_base = smem_u32(&s.kb[0][0]);
    const uint32_t vb_base = smem_u32(&s.vb[0][0]);

    for (int i = 0; i < n_chunks; ++i) {
        const int st = i & 1;
        // advance the entry pipeline: chunk i+3 entries, chunk i+2 page, chunk i+1 copies + scales
        e3 = load_entry(i + 3);
        resolve(e2);
        issue_copy(e1, st ^ 1);
        load_scales(e1, ks1, vs1);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();

        // dequantise chunk i: 1024 pieces of 16 int8 -> 16 bf16
        for (int u = tid; u < 2 * kChunk * 8; u += kThreads) {
            const int kv = u >> 9, cell = (u >> 3) & 63, seg = u & 7;
            const uint4 raw = *reinterpret_cast<const uint4*>(&s.raw[st][kv][cell][seg * 16]);
            uint4 lo, hi;
            if (kv) dequant16(raw, s.vs[st][cell], lo, hi);
            else int8x16_to_bf16(raw, lo, hi);
            uint8_t* base = reinterpret_cast<uint8_t*>(kv ? &s.vb[0][0] : &s.kb[0][0]);
            *reinterpret_cast<uint4*>(base + swz(cell, 2 * seg)) = lo;
            *reinterpret_cast<uint4*>(base + swz(cell, 2 * seg + 1)) = hi;
        }
        __syncthreads();

        // S = Q K'^T  (16 rows x 64 cells per warp)
        float sc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            const int cell = nt * 8 + (lane & 7);
#pragma unroll
            for (int kk2 = 0; kk2 < 4; ++kk2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb_base + swz(cell, 4 * kk2 + (lane >> 3)), b0, b1, b2, b3);
                mma_bf16(sc[nt], qa[2 * kk2], b0, b1);
                mma_bf16(sc[nt], qa[2 * kk2 + 1], b2, b3);
            }
        }
        // column scale, then mask: cell c is -inf for rows whose query did not select it
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int c = nt * 8 + 2 * t4;
            const uint32_t mA = s.mask[st][c], mB = s.mask[st][c + 1];
            const float2 kc = *reinterpret_cast<const float2*>(&s.ks[st][c]);
            sc[nt][0] = ((mA >> j0) & 1u) ? sc[nt][0] * kc.x : -INFINITY;
            sc[nt][1] = ((mB >> j0) & 1u) ? sc[nt][1] * kc.y : -INFINITY;
            sc[nt][2] = ((mA >> j1) & 1u) ? sc[nt][2] * kc.x : -INFINITY;
            sc[nt][3] = ((mB >> j1) & 1u) ? sc[nt][3] * kc.y : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
        uint32_t pa[8][2];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = fast_exp2(sc[nt][0] - mu0), p1 = fast_exp2(sc[nt][1] - mu0);
            const float p2 = fast_exp2(sc[nt][2] - mu1), p3 = fast_exp2(sc[nt][3] - mu1);
            pa[nt][0] = pack_bf16x2(p0, p1);
            pa[nt][1] = pack_bf16x2(p2, p3);
            // the normaliser sums the same BF16-rounded weights that enter P V
            ps0 += bf16_lo(pa[nt][0]) + bf16_hi(pa[nt][0]);
            ps1 += bf16_lo(pa[nt][1]) + bf16_hi(pa[nt][1]);
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            o[dt][0] *= al0; o[dt][1] *= al0;
            o[dt][2] *= al1; o[dt][3] *= al1;
        }
        // O += P V'
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
            const uint32_t af[4] = {pa[2 * kc][0], pa[2 * kc][1], pa[2 * kc + 1][0], pa[2 * kc + 1][1]};
            const int cell = kc * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
            for (int dn = 0; dn < 16; dn += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vb_base + swz(cell, dn + (lane >> 4)), b0, b1, b2, b3);
                mma_bf16(o[dn], af, b0, b1);
                mma_bf16(o[dn + 1], af, b2, b3);
            }
        }

        // finish chunk i+1's table (its scale loads have landed by now) and rotate
        write_table(e1, st ^ 1, ks1, vs1);
        e1 = e2;
        e2 = e3;
        __syncthreads();
    }

    // ---- epilogue: O / l ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    float* out0 = a.out + ((size_t)(q_begin + j0) * n_heads + h * kHeadsPerKv + r0 % kHeadsPerKv) * kHeadDim;
    float* out1 = a.out + ((size_t)(q_begin + j1) * n_heads + h * kHeadsPerKv + r1 % kHeadsPerKv) * kHeadDim;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
        const int d = dt * 8 + 2 * t4;
        if (v0) *reinterpret_cast<float2*>(out0 + d) = make_float2(o[dt][0] * inv0, o[dt][1] * inv0);
        if (v1) *reinterpret_cast<float2*>(out1 + d) = make_float2(o[dt][2] * inv1, o[dt][3] * inv1);
    }
}

}  // namespace

cudaError_t launch_attn_mma(const AttnArgs& a, cudaStream_t stream) {
    const int smem = (int)sizeof(SmemMma);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((a.n_q + kGroup - 1) / kGroup, a.n_kv);
    attn_mma_kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
