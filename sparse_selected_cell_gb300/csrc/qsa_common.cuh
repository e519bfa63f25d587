// qsa_common.cuh -- constants and small device helpers shared by the sm_103a
// kernels of libqsa.so (union build and union attention).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kHeadDim = 128;     // d
constexpr int kHeadsPerKv = 12;   // grouped query heads per KV head
constexpr int kGroup = 8;         // queries per union group
constexpr int kRows = kGroup * kHeadsPerKv;   // 96 query-head rows per (group, KV head)
constexpr int kPage = 64;         // cells per page
constexpr int kChunk = 64;        // union cells per dequantised chunk
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void report(int32_t* status, int bits) {
    if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------- conversions
// FP32 pairs rounded (to nearest even) into packed 16-bit pairs, low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Exact int8 -> bf16 (|x| <= 128 fits bf16's 8-bit significand).  Each byte b
// sits in the low byte of a 16-bit lane whose high byte is 0x43: keeping b's low
// 7 bits gives the bf16 value 128 + (b & 127); keeping only b's bit 7 gives 128
// or 256 (that bit lands on the exponent's lowest bit).  Their bf16 difference is
// the two's-complement value of b, computed exactly.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void int8x4_to_bf16(uint32_t w, uint32_t& out01, uint32_t& out23) {
    const uint32_t l01 = __byte_perm(w, 0x4343u, 0x5140);   // [b0, 0x43, b1, 0x43]
    const uint32_t l23 = __byte_perm(w, 0x4343u, 0x5342);   // [b2, 0x43, b3, 0x43]
    out01 = bf16x2_sub(l01 & 0xFF7FFF7Fu, l01 & 0xFF80FF80u);
    out23 = bf16x2_sub(l23 & 0xFF7FFF7Fu, l23 & 0xFF80FF80u);
}

// Exact int8 -> fp16 (fp16's 11-bit significand holds any integer below 2048):
// the byte biased by 128 (b ^ 0x80 = x + 128, 0..255) becomes the low mantissa
// byte of fp16 1024 (0x6400), giving 1152 + x; subtracting 1152 (0x6480) leaves x.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void int8x4_to_f16(uint32_t w, uint32_t& out01, uint32_t& out23) {
    const uint32_t u = w ^ 0x80808080u;
    out01 = f16x2_sub(__byte_perm(u, 0x6464u, 0x5140), 0x64806480u);   // [u0, 0x64, u1, 0x64]
    out23 = f16x2_sub(__byte_perm(u, 0x6464u, 0x5342), 0x64806480u);   // [u2, 0x64, u3, 0x64]
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// floor(log2 |x|) of a finite, normal, non-zero float (its unbiased exponent field).
__device__ __forceinline__ int f32_exponent(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }

// 2^e exactly, for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- launchers
// Implemented in union_build.cu / attn_tc.cu / attn_sm.cu; called by capi.cu
// after argument validation.  They return cudaGetLastError() of the launch.
cudaError_t launch_union_build(const int32_t* sel, const int32_t* sel_count, int n_q, int sel_stride,
                               int32_t* union_cells, uint8_t* union_mask, int32_t* union_count,
                               int union_stride, int32_t* dev_status, cudaStream_t stream);

struct AttnArgs {
    const uint16_t* q;
    const int8_t* k_pool;
    const int8_t* v_pool;
    const uint16_t* k_scale;
    const uint16_t* v_scale;
    const int32_t* page_table;
    int n_lpages, n_ppages, n_kv;
    const int32_t* union_cells;
    const uint8_t* union_mask;
    const int32_t* union_count;
    int union_stride, n_q;
    float sm_scale;
    float* out;
    int32_t* dev_status;
    // the per-position lists, read by the fused kernel instead of the union arrays
    const int32_t* sel;
    const int32_t* sel_count;
    int sel_stride;
};

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_sm(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_fused(const AttnArgs& a, cudaStream_t stream);
// Dynamic shared memory of the fused kernel for lists of sel_stride entries.
size_t attn_fused_smem_bytes(int sel_stride);

// Per-position attention (no union): each query over its own selection list,
// with one shared page table (prompt) or one table per query (decode).
struct SelArgs {
    const uint16_t* q;
    const int8_t* k_pool;
    const int8_t* v_pool;
    const uint16_t* k_scale;
    const uint16_t* v_scale;
    const int32_t* page_table;   // query i's table: page_table + i * pt_stride (0: one shared table)
    int n_lpages, n_ppages, n_kv;
    const int32_t* sel;
    const int32_t* sel_count;
    int sel_stride, n_q;
    float sm_scale;
    float* out;
    int32_t* dev_status;
    int pt_stride;
};

cudaError_t launch_select_attn(const SelArgs& a, cudaStream_t stream);

}  // namespace qsa
