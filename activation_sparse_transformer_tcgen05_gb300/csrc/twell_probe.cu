// twell_probe.cu — the gather ceiling the sparse kernels run against.
//
// Every sparse kernel of the library (down-projection, SDDMM, dx, weight
// gradients) is a row gather: a warp reads one 512-byte stretch of a bf16 row
// named by a TwELL index with 128-bit loads, over and over, from rows that
// stay in L2 (W_down and W_up of one layer are tens of MB). Their time is set
// by how fast the GPU delivers such gathers, not by HBM bandwidth or FMA
// issue. This kernel performs exactly that access pattern with no arithmetic
// beyond a checksum, so its rate is the ceiling the sparse kernels are
// measured against.
#include "common.cuh"
#include "launch.h"

namespace twell {
namespace {

constexpr int kProbeWarps = 8;
constexpr int kProbeInFlight = 8;  // 128-bit loads per lane in flight, as in the sparse kernels

// Warp task (row r, 256-column group g): for k < nnz, lane reads the 16 bytes
// at W[idx[r, k], 256 g + 8 lane]. Indices are clamped into [0, F).
__global__ void __launch_bounds__(kProbeWarps * 32) k_gather_probe(const uint16_t* __restrict__ W, int F, int d,
                                                                   const int32_t* __restrict__ idx, int rows,
                                                                   int nnz, float* __restrict__ sink)
{
    const int lane = threadIdx.x & 31;
    const int G = (d + 255) >> 8;
    const long long task = (long long)blockIdx.x * kProbeWarps + (threadIdx.x >> 5);
    if (task >= (long long)rows * G) return;
    const int r = (int)(task / G), g = (int)(task % G);
    const int c0 = g * 256 + lane * 8;
    const bool col_ok = c0 < d;
    const int32_t* ir = idx + (size_t)r * nnz;
    uint32_t acc = 0;
    for (int k0 = 0; k0 < nnz; k0 += 32) {
        const int m = min(32, nnz - k0);
        int jl = 0;
        if (lane < m) jl = min(max(ir[k0 + lane], 0), F - 1);
        int u = 0;
        for (; u + kProbeInFlight <= m; u += kProbeInFlight) {
            uint4 v[kProbeInFlight];
#pragma unroll
            for (int q = 0; q < kProbeInFlight; ++q) {
                const int j = __shfl_sync(0xffffffffu, jl, u + q);
                v[q] = col_ok ? __ldg(reinterpret_cast<const uint4*>(W + (size_t)j * d + c0)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kProbeInFlight; ++q) acc ^= v[q].x ^ v[q].y ^ v[q].z ^ v[q].w;
        }
        for (; u < m; ++u) {
            const int j = __shfl_sync(0xffffffffu, jl, u);
            const uint4 v = col_ok ? __ldg(reinterpret_cast<const uint4*>(W + (size_t)j * d + c0)) : make_uint4(0, 0, 0, 0);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sink[task] = __uint_as_float(acc & 0x007fffffu);  // a finite value, so the loads stay live
}

}  // namespace
}  // namespace twell

extern "C" twell_status twell_gather_probe(const uint16_t* W, int F, int d, const int32_t* idx, int rows, int nnz,
                                           float* sink, void* stream)
{
    if (!W || !idx || !sink || F <= 0 || d <= 0 || (d & 7) != 0 || rows <= 0 || nnz < 0)
        return TWELL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return TWELL_ERR_INVALID_ARG;
    const long long tasks = (long long)rows * ((d + 255) / 256);
    const long long blocks = (tasks + twell::kProbeWarps - 1) / twell::kProbeWarps;
    if (blocks > 0x7fffffffLL) return TWELL_ERR_UNSUPPORTED;
    twell::count_launches(1);
    twell::k_gather_probe<<<(unsigned)blocks, twell::kProbeWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        W, F, d, idx, rows, nnz, sink);
    return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
