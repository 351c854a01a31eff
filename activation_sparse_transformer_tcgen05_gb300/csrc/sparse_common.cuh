// sparse_common.cuh — device helpers shared by the CUDA-core kernels of the
// TwELL library (warp reductions and scans, TwELL row addressing, bf16 dot
// products and FMAs with fp32 accumulation). Each translation unit gets its
// own inlined copy.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace twell {
namespace {

constexpr int kWarps = 8;  // warps per block of the sparse kernels

__device__ __forceinline__ int warp_sum_i(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_max_i(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

__device__ __forceinline__ int nz_bf16(uint32_t half) { return (half & 0x7fffu) != 0u; }

// First slot of row r and its tile width.
__device__ __forceinline__ int64_t row_base(const TwellView& tw, int r, int* Kt)
{
    const int t = r / tw.T;
    *Kt = tw.K[t];
    return tw.off[t] + (int64_t)(r - t * tw.T) * (*Kt);
}

// acc[0..7] += v * (8 bf16 in w)
__device__ __forceinline__ void fma8(float (&acc)[8], float v, const uint4& w)
{
    acc[0] = fmaf(v, bf16_lo(w.x), acc[0]);
    acc[1] = fmaf(v, bf16_hi(w.x), acc[1]);
    acc[2] = fmaf(v, bf16_lo(w.y), acc[2]);
    acc[3] = fmaf(v, bf16_hi(w.y), acc[3]);
    acc[4] = fmaf(v, bf16_lo(w.z), acc[4]);
    acc[5] = fmaf(v, bf16_hi(w.z), acc[5]);
    acc[6] = fmaf(v, bf16_lo(w.w), acc[6]);
    acc[7] = fmaf(v, bf16_hi(w.w), acc[7]);
}

// acc[0..7] += v * (8 bf16 in w) with v a bf16 value (low 16 bits of vbits):
// fma.rn.f32.bf16 multiplies two bf16 factors and accumulates in fp32. Their
// product is exact in fp32, so this rounds exactly like fmaf on the widened
// values, without the widening instructions.
__device__ __forceinline__ void fma2_bf16(float& a0, float& a1, uint32_t w2, uint32_t vbits)
{
    asm("{\n"
        ".reg .b16 lo, hi, vb;\n"
        "mov.b32 {lo, hi}, %2;\n"
        "cvt.u16.u32 vb, %3;\n"
        "fma.rn.f32.bf16 %0, vb, lo, %0;\n"
        "fma.rn.f32.bf16 %1, vb, hi, %1;\n"
        "}\n"
        : "+f"(a0), "+f"(a1)
        : "r"(w2), "r"(vbits));
}

__device__ __forceinline__ void fma8_bf16(float (&acc)[8], uint32_t vbits, const uint4& w)
{
    fma2_bf16(acc[0], acc[1], w.x, vbits);
    fma2_bf16(acc[2], acc[3], w.y, vbits);
    fma2_bf16(acc[4], acc[5], w.z, vbits);
    fma2_bf16(acc[6], acc[7], w.w, vbits);
}

// sum_k a[k] * b[k] over 8 bf16 pairs in two independent fp32 chains.
__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b)
{
    float s0 = 0.f, s1 = 0.f;
    asm("{\n"
        ".reg .b16 a0, a1, b0, b1;\n"
        "mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %6;\n"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n fma.rn.f32.bf16 %1, a1, b1, %1;\n"
        "mov.b32 {a0, a1}, %3;\n mov.b32 {b0, b1}, %7;\n"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n fma.rn.f32.bf16 %1, a1, b1, %1;\n"
        "mov.b32 {a0, a1}, %4;\n mov.b32 {b0, b1}, %8;\n"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n fma.rn.f32.bf16 %1, a1, b1, %1;\n"
        "mov.b32 {a0, a1}, %5;\n mov.b32 {b0, b1}, %9;\n"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n fma.rn.f32.bf16 %1, a1, b1, %1;\n"
        "}\n"
        : "+f"(s0), "+f"(s1)
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
    return s0 + s1;
}

// sum_k a[k] * b[k] over 8 bf16 pairs
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b)
{
    float s = bf16_lo(a.x) * bf16_lo(b.x);
    s = fmaf(bf16_hi(a.x), bf16_hi(b.x), s);
    s = fmaf(bf16_lo(a.y), bf16_lo(b.y), s);
    s = fmaf(bf16_hi(a.y), bf16_hi(b.y), s);
    s = fmaf(bf16_lo(a.z), bf16_lo(b.z), s);
    s = fmaf(bf16_hi(a.z), bf16_hi(b.z), s);
    s = fmaf(bf16_lo(a.w), bf16_lo(b.w), s);
    s = fmaf(bf16_hi(a.w), bf16_hi(b.w), s);
    return s;
}

// 16 bytes from read-only global memory. Written as a plain inline-PTX load
// rather than __ldg: the gathers issue their row loads where they are written,
// ahead of the FMAs that use them, and measured 2-3 % faster this way.
__device__ __forceinline__ uint4 ldg16(const uint16_t* p)
{
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ bool over_capacity(const TwellView& tw)
{
    return tw.off[tw.n_tiles] > tw.cap;
}

inline unsigned grid_for_warps(int64_t warps) { return (unsigned)((warps + kWarps - 1) / kWarps); }

}  // namespace
}  // namespace twell
