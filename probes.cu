// probes.cu — measurement probes of the benchmark (not part of the library).
//
// The TwELL sparse kernels (down-projection, SDDMM, dx, weight gradients) run
// on the CUDA cores: each stored entry pulls one stretch of a bf16 row, named
// by a TwELL index, from L2 into the SM and does fp32 FMAs on it. Their
// ceilings are therefore neither HBM bandwidth nor the tensor-core peak but
//   - the FP32 FMA rate of the SMs (probe_fma), and
//   - how fast row stretches named by random indices reach the SMs
//     (128-bit loads into registers in the kernels' own orders; and, for
//     comparison, asynchronous bulk copies into shared memory, which keep
//     more bytes in flight per SM than registers allow but were measured
//     slower).
// bench.py builds this file into _build/libprobes.so and reports each kernel
// against the measured figures. Every wait is bounded; a probe that gives up
// reports it in its status word.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ unsigned long long now_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ FMA --

// Each thread runs 8 independent fp32 FMA chains for `iters` steps; the FLOP
// count is 2 * 8 * iters per thread. mode 0: fmaf on fp32 operands; mode 1:
// fma.rn.f32.bf16 (two bf16 factors, fp32 accumulator), the sparse kernels'
// product form.
template <int MODE>
__global__ void __launch_bounds__(256) k_fma(int iters, float seed, float* sink)
{
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = seed * (float)(threadIdx.x + i);
    const float a = seed + 1.0f, b = 0.999f;
    uint32_t ab = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xffff0000u);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 16; ++u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (MODE == 0) {
                    acc[i] = fmaf(a, acc[i], b);
                } else {
                    asm volatile("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nfma.rn.f32.bf16 %0, lo, hi, %0;\n}\n"
                                 : "+f"(acc[i])
                                 : "r"(ab));
                }
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += acc[i];
    if (s == 1234.5f) sink[blockIdx.x * blockDim.x + threadIdx.x] = s;  // keeps the chains live
}

// --------------------------------------------------------------- gathers --

constexpr int kWarps = 8;
constexpr int kColsWarps = 2;  // the down-projection's block: 2 warps, 14 blocks per SM

// 16 bytes from read-only global memory, in the same form as the library's
// gathers (a plain inline-PTX load).
__device__ __forceinline__ uint4 ldg16(const uint16_t* p)
{
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// One warp per (row r, 256-column group g): for k < nnz the lane reads the 16
// bytes at W[idx[r, k], 256 g + 8 lane], IN_FLIGHT 128-bit loads at a time.
template <int IN_FLIGHT>
__global__ void __launch_bounds__(kWarps * 32) k_gather_ldg(const uint16_t* __restrict__ W, int F, int d,
                                                            const int32_t* __restrict__ idx, int rows, int nnz,
                                                            float* __restrict__ sink)
{
    const int lane = threadIdx.x & 31;
    const int G = (d + 255) >> 8;
    const long long task = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
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
        for (; u + IN_FLIGHT <= m; u += IN_FLIGHT) {
            uint4 v[IN_FLIGHT];
#pragma unroll
            for (int q = 0; q < IN_FLIGHT; ++q) {
                const int j = __shfl_sync(0xffffffffu, jl, u + q);
                v[q] = col_ok ? __ldg(reinterpret_cast<const uint4*>(W + (size_t)j * d + c0)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < IN_FLIGHT; ++q) acc ^= v[q].x ^ v[q].y ^ v[q].z ^ v[q].w;
        }
        for (; u < m; ++u) {
            const int j = __shfl_sync(0xffffffffu, jl, u);
            const uint4 v =
                col_ok ? __ldg(reinterpret_cast<const uint4*>(W + (size_t)j * d + c0)) : make_uint4(0, 0, 0, 0);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sink[task] = __uint_as_float(acc & 0x007fffffu);
}

// The down-projection's own order and launch shape: warp task (column group g
// of 512 columns, row r), task = g * rows + r, so the grid walks W one
// 512-column slice at a time; the lane reads 16 bytes in each of its two
// 256-column chunks, four entries (eight 128-bit loads) in flight; 2-warp
// blocks, 14 per SM.
__global__ void __launch_bounds__(kColsWarps * 32, 14) k_gather_cols(const uint16_t* __restrict__ W, int F, int d,
                                                                     const int32_t* __restrict__ idx, int rows,
                                                                     int nnz, float* __restrict__ sink)
{
    const int lane = threadIdx.x & 31;
    const int G = (d + 511) >> 9;
    const long long task = (long long)blockIdx.x * kColsWarps + (threadIdx.x >> 5);
    if (task >= (long long)rows * G) return;
    const int g = (int)(task / rows), r = (int)(task % rows);
    const int c0 = g * 512 + lane * 8, c1 = c0 + 256;
    const bool ok0 = c0 < d, ok1 = c1 < d;
    const int32_t* ir = idx + (size_t)r * nnz;
    uint32_t acc = 0;
    for (int k0 = 0; k0 < nnz; k0 += 32) {
        const int m = min(32, nnz - k0);
        int jl = 0;
        if (lane < m) jl = min(max(ir[k0 + lane], 0), F - 1);
        for (int u = 0; u < m; u += 4) {
            uint4 v[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = __shfl_sync(0xffffffffu, jl, u + q < m ? u + q : u);
                const bool live = u + q < m;
                v[q][0] = (live && ok0) ? ldg16(W + (size_t)j * d + c0) : make_uint4(0, 0, 0, 0);
                v[q][1] = (live && ok1) ? ldg16(W + (size_t)j * d + c1) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                acc ^= v[q][0].x ^ v[q][0].y ^ v[q][0].z ^ v[q][0].w ^ v[q][1].x ^ v[q][1].y ^ v[q][1].z ^ v[q][1].w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sink[task] = __uint_as_float(acc & 0x007fffffu);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    const unsigned long long t0 = now_ns();
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 63u) == 63u && now_ns() - t0 > kWaitLimitNs) return false;
    }
}

constexpr int kBulkWarps = 4;   // warps per block
constexpr int kBatch = 8;       // entries per batch (one bulk copy of 512 bytes each)
constexpr int kSlotBytes = 512; // 256 bf16 columns

// Same task and bytes as k_gather_ldg, but each warp's lanes 0..7 copy a
// batch of 8 row stretches (512 bytes each) into a shared-memory ring with
// cp.async.bulk, completion counted on the batch's mbarrier; RING batches are
// in flight per warp. The consumer reads its 16 bytes of every stretch.
// Dynamic shared memory: kBulkWarps * RING * kBatch * kSlotBytes bytes.
template <int RING>
__global__ void __launch_bounds__(kBulkWarps * 32) k_gather_bulk(const uint16_t* __restrict__ W, int F, int d,
                                                                 const int32_t* __restrict__ idx, int rows, int nnz,
                                                                 float* __restrict__ sink, int32_t* status)
{
    extern __shared__ __align__(128) uint8_t dyn[];
    __shared__ __align__(8) uint64_t bars[kBulkWarps][RING];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = dyn + (size_t)warp * RING * kBatch * kSlotBytes;
    const int G = (d + 255) >> 8;
    if (lane < RING) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[warp][lane])) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    const long long task = (long long)blockIdx.x * kBulkWarps + warp;
    if (task >= (long long)rows * G) return;
    const int r = (int)(task / G), g = (int)(task % G);
    const int32_t* ir = idx + (size_t)r * nnz;
    const int nb = (nnz + kBatch - 1) / kBatch;
    auto issue = [&](int b) {
        const int slot = b % RING;
        const int k0 = b * kBatch;
        const int m = min(kBatch, nnz - k0);
        if (lane == 0) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bars[warp][slot])),
                         "r"((uint32_t)(m * kSlotBytes))
                         : "memory");
        }
        __syncwarp();
        if (lane < m) {
            const int j = min(max(ir[k0 + lane], 0), F - 1);
            const uint16_t* src = W + (size_t)j * d + g * 256;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(ring + (size_t)slot * kBatch * kSlotBytes + lane * kSlotBytes)),
                "l"(src), "r"((uint32_t)kSlotBytes), "r"(smem_u32(&bars[warp][slot]))
                : "memory");
        }
    };
    int issued = 0;
    for (; issued < nb && issued < RING; ++issued) issue(issued);
    uint32_t acc = 0;
    int b = 0;
    for (; b < nb; ++b) {
        const int slot = b % RING;
        if (!mbar_wait(&bars[warp][slot], (uint32_t)((b / RING) & 1))) break;
        const int m = min(kBatch, nnz - b * kBatch);
        const uint8_t* sl = ring + (size_t)slot * kBatch * kSlotBytes;
        for (int u = 0; u < m; ++u) {
            const uint4 v = *reinterpret_cast<const uint4*>(sl + u * kSlotBytes + lane * 16);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        __syncwarp();  // every lane has read the slot before it is refilled
        if (issued < nb) issue(issued++);
    }
    if (b < nb) {
        if (lane == 0) atomicExch(status, 1);
        // the copies still in flight land before the block's shared memory goes away
        for (int q = b; q < issued; ++q) (void)mbar_wait(&bars[warp][q % RING], (uint32_t)((q / RING) & 1));
        return;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sink[task] = __uint_as_float(acc & 0x007fffffu);
}

template <int RING>
int launch_bulk(const uint16_t* W, int F, int d, const int32_t* idx, int rows, int nnz, float* sink,
                int32_t* status, cudaStream_t s, long long blocks)
{
    const int smem = kBulkWarps * RING * kBatch * kSlotBytes;
    if (cudaFuncSetAttribute(k_gather_bulk<RING>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 2;
    k_gather_bulk<RING><<<(unsigned)blocks, kBulkWarps * 32, smem, s>>>(W, F, d, idx, rows, nnz, sink, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace

extern "C" {

// FP32 FMA peak probe: 2 * 8 * 16 * iters FLOP per thread over blocks x 256 threads.
int probe_fma(int mode, int blocks, int iters, float* sink, void* stream)
{
    if (blocks <= 0 || iters <= 0 || !sink || (mode != 0 && mode != 1)) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == 0)
        k_fma<0><<<blocks, 256, 0, s>>>(iters, 0.5f, sink);
    else
        k_fma<1><<<blocks, 256, 0, s>>>(iters, 0.5f, sink);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// Gather probe: W [F, d] bf16 (16-byte aligned, d % 8 == 0), idx [rows, nnz]
// int32 (clamped into [0, F)), sink [rows * ceil(d/256)] float.
// mode 0: 128-bit loads, 4 in flight per lane; mode 1: 8 in flight; modes 2
// and 3: bulk copies into shared memory, 3 or 6 batches of 8 rows in flight
// per warp (d % 256 == 0); mode 4: 128-bit loads in the down-projection's
// column-group-major order, 512 columns per task (sink then holds
// rows * ceil(d/512) floats, task g * rows + r). status: int32 device word,
// set to 1 if a bounded wait gave up.
int probe_gather(int mode, const uint16_t* W, int F, int d, const int32_t* idx, int rows, int nnz, float* sink,
                 int32_t* status, void* stream)
{
    if (!W || !idx || !sink || !status || F <= 0 || d <= 0 || (d & 7) != 0 || rows <= 0 || nnz < 0) return 1;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) != 0) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long tasks = (long long)rows * ((d + 255) / 256);
    if (mode == 0 || mode == 1) {
        const long long blocks = (tasks + kWarps - 1) / kWarps;
        if (blocks > 0x7fffffffLL) return 1;
        if (mode == 0)
            k_gather_ldg<4><<<(unsigned)blocks, kWarps * 32, 0, s>>>(W, F, d, idx, rows, nnz, sink);
        else
            k_gather_ldg<8><<<(unsigned)blocks, kWarps * 32, 0, s>>>(W, F, d, idx, rows, nnz, sink);
    } else if (mode == 4) {
        const long long t4 = (long long)rows * ((d + 511) / 512);
        const long long blocks = (t4 + kColsWarps - 1) / kColsWarps;
        if (blocks > 0x7fffffffLL) return 1;
        k_gather_cols<<<(unsigned)blocks, kColsWarps * 32, 0, s>>>(W, F, d, idx, rows, nnz, sink);
    } else if (mode == 2 || mode == 3) {
        if (d % 256 != 0) return 1;
        const long long blocks = (tasks + kBulkWarps - 1) / kBulkWarps;
        if (blocks > 0x7fffffffLL) return 1;
        return mode == 2 ? launch_bulk<3>(W, F, d, idx, rows, nnz, sink, status, s, blocks)
                         : launch_bulk<6>(W, F, d, idx, rows, nnz, sink, status, s, blocks);
    } else {
        return 1;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
