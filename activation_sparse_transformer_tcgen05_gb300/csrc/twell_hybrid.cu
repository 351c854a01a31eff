// twell_hybrid.cu — backward of the layer on the hybrid format.
//
// "Sparser, Faster, Lighter Transformer Language Models", Resumo Técnico §2,
// "Formato Híbrido para Treinamento": rows with more nonzeros than the compact
// format holds are kept as a dense backup matrix. In the backward the TwELL
// rows go through the sparse kernels (twell_ffn_bwd) and the n dense overflow
// rows R through tcgen05 GEMMs:
//   dpre_R  = (dy[R] W_down^T + l1) masked by h_R != 0       [n, F] fp32
//   db     += column sums of dpre_R (rows in order)
//   dx[R]   = dpre_R W_up                                      (bf16 rows of dx)
//   dW_up  += dpre_R^T x[R],   dW_down += h_R^T dy[R]          (fp32)
// The tensor cores take bf16 operands; dpre_R enters as the sum of two bf16
// parts (hi = RNE(dpre), lo = RNE(dpre - hi), ~2^-17 relative), so each GEMM
// on it runs twice and accumulates in fp32. The GEMMs whose inner dimension is
// the token axis take transposed copies ([F or d, rows], zero past n).
// The host never reads n: every kernel takes it from the device count.
#include "common.cuh"
#include "launch.h"

namespace twell {
namespace {

// Overflow rows in use: the device count, never more than the block holds.
__device__ __forceinline__ int live_rows(const int32_t* n_rows, int cap_rows)
{
    const int n = *n_rows;
    return n < 0 ? 0 : (n < cap_rows ? n : cap_rows);
}

// Rows of the token axis the GEMMs read: the live rows rounded up to the GEMM's
// 64-deep k-block (the rows between are zeros). Kernels skip every row past it.
__device__ __forceinline__ int used_rows(int n) { return (n + 63) / 64 * 64; }

// dst[i, :] = src[rows[i], :] for i < n, zeros for n <= i < cap (bf16 rows of d).
__global__ void k_gather_rows(const uint16_t* __restrict__ src, int d, const int32_t* __restrict__ rows,
                              const int32_t* __restrict__ n_rows, int cap_rows, int cap,
                              uint16_t* __restrict__ dst)
{
    const int i = blockIdx.x;
    if (i >= cap) return;
    const int n = live_rows(n_rows, cap_rows);
    if (i >= used_rows(n)) return;
    uint4* out = reinterpret_cast<uint4*>(dst + (size_t)i * d);
    if (i < n) {
        const uint4* in = reinterpret_cast<const uint4*>(src + (size_t)rows[i] * d);
        for (int c = threadIdx.x; c < d / 8; c += blockDim.x) out[c] = in[c];
    } else {
        for (int c = threadIdx.x; c < d / 8; c += blockDim.x) out[c] = make_uint4(0, 0, 0, 0);
    }
}

// hi/lo bf16 parts of the fp32 rows of dpre (zeros past n).
__global__ void k_split_rows(const float* __restrict__ src, int cols, const int32_t* __restrict__ n_rows,
                             int cap_rows, int cap, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo)
{
    const int i = blockIdx.x;
    if (i >= cap) return;
    const int n = live_rows(n_rows, cap_rows);
    if (i >= used_rows(n)) return;
    const bool live = i < n;
    for (int c = threadIdx.x; c < cols; c += blockDim.x) {
        const size_t k = (size_t)i * cols + c;
        const float v = live ? src[k] : 0.f;
        const uint16_t h = f32_to_bf16_bits(v);
        hi[k] = h;
        lo[k] = f32_to_bf16_bits(v - bf16_to_f32(h));
    }
}

// out[j] += sum over i < n of src[i, j], i ascending (one thread per column).
__global__ void k_colsum_add(const float* __restrict__ src, int cols, const int32_t* __restrict__ n_rows,
                             int cap_rows, float* __restrict__ out)
{
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= cols) return;
    const int n = live_rows(n_rows, cap_rows);
    float s = 0.f;
    for (int i = 0; i < n; ++i) s += src[(size_t)i * cols + j];
    out[j] += s;
}

// dst [cols, stride] = src [rows, cols]^T for the first n rows of src (n
// clamped to cap_rows, the rows src holds); columns n .. stride-1 of dst are
// zero. 32 x 32 tiles through shared memory (padded against bank conflicts);
// grid.y * 32 == stride.
__global__ void k_transpose(const uint16_t* __restrict__ src, int cols, const int32_t* __restrict__ n_rows,
                            int cap_rows, int stride, uint16_t* __restrict__ dst)
{
    __shared__ uint16_t t[32][33];
    const int n = live_rows(n_rows, cap_rows);
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    if (r0 >= used_rows(n)) return;  // uniform over the block
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    for (int k = ty; k < 32; k += 8) {
        const int r = r0 + k, c = c0 + tx;
        t[k][tx] = (r < n && c < cols) ? src[(size_t)r * cols + c] : (uint16_t)0;
    }
    __syncthreads();
    for (int k = ty; k < 32; k += 8) {
        const int c = c0 + k, r = r0 + tx;
        if (c < cols && r < stride) dst[(size_t)c * stride + r] = t[tx][k];
    }
}

// dx[rows[i], :] = bf16(src[i, :]) for i < n.
__global__ void k_scatter_rows_bf16(const float* __restrict__ src, int d, const int32_t* __restrict__ rows,
                                    const int32_t* __restrict__ n_rows, int cap_rows, uint16_t* __restrict__ dst)
{
    const int i = blockIdx.x;
    if (i >= live_rows(n_rows, cap_rows)) return;
    uint16_t* out = dst + (size_t)rows[i] * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) out[c] = f32_to_bf16_bits(src[(size_t)i * d + c]);
}

struct Carver {
    char* p;
    size_t used = 0;
    template <typename T>
    T* take(size_t n)
    {
        const size_t off = (used + 255) & ~size_t(255);
        used = off + n * sizeof(T);
        return p ? reinterpret_cast<T*>(p + off) : nullptr;
    }
};

struct HybridBwdWs {
    uint16_t *dyR, *xR, *hi, *lo, *hiT, *loT, *hT, *xRT, *dyRT;
    float *dpre, *dxR;
    char* sparse;  // twell_ffn_bwd's own workspace
    size_t sparse_bytes;
};

constexpr int kRowPad = 64;  // token axis of the overflow block, padded to the GEMM's k-block

size_t carve_hybrid_bwd(void* ws, int M, int d, int F, int T, int64_t cap_slots, int cap_rows, HybridBwdWs* out)
{
    const size_t cap = (size_t)((cap_rows + kRowPad - 1) / kRowPad) * kRowPad;
    Carver c{static_cast<char*>(ws)};
    HybridBwdWs w{};
    w.dyR = c.take<uint16_t>(cap * d);
    w.xR = c.take<uint16_t>(cap * d);
    w.dpre = c.take<float>(cap * F);
    w.hi = c.take<uint16_t>(cap * F);
    w.lo = c.take<uint16_t>(cap * F);
    w.hiT = c.take<uint16_t>(cap * F);
    w.loT = c.take<uint16_t>(cap * F);
    w.hT = c.take<uint16_t>(cap * F);
    w.xRT = c.take<uint16_t>(cap * d);
    w.dyRT = c.take<uint16_t>(cap * d);
    w.dxR = c.take<float>(cap * d);
    w.sparse_bytes = twell_workspace_bytes(TWELL_OP_FFN_BWD, M, d, F, T, cap_slots);
    w.sparse = c.take<char>(w.sparse_bytes);
    if (out) *out = w;
    return c.used;
}

cudaError_t dense_gemm_f32(const uint16_t* A, const uint16_t* B, int rowsA, const int32_t* rowsA_dev, int rowsB,
                           int K, float* out, int ldo, int accumulate, const uint16_t* mask, int ldm, float add,
                           int32_t* status, int sms, cudaStream_t s, const int32_t* K_dev = nullptr)
{
    GemmArgs g{};
    g.rowsA = rowsA;
    g.rowsA_dev = rowsA_dev;
    g.K_dev = K_dev;
    g.rowsB = rowsB;
    g.K = K;
    g.out_f32 = out;
    g.ldo = ldo;
    g.accumulate = accumulate;
    g.mask = mask;
    g.ldm = ldm;
    g.add_scalar = add;
    g.status = status;
    return launch_gemm(GEMM_DENSE, A, B, g, sms, s);
}

int sms_now()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return 0;
    return n;
}

}  // namespace
}  // namespace twell

using namespace twell;

extern "C" size_t twell_hybrid_bwd_workspace_bytes(int M, int d, int F, int T, int64_t cap_slots, int cap_rows)
{
    if (M <= 0 || d <= 0 || F <= 0 || T <= 0 || cap_rows < 0) return 0;
    return carve_hybrid_bwd(nullptr, M, d, F, T, cap_slots, cap_rows, nullptr);
}

extern "C" twell_status twell_hybrid_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down,
                                             const uint16_t* W_upT, const twell_buf* h, const twell_overflow* ov,
                                             const uint16_t* dy, int d, float l1_coef, uint16_t* dx, float* dW_up,
                                             float* dW_down, float* db, void* ws, size_t ws_bytes,
                                             int32_t* status, void* stream)
{
    if (!h || !ov || !W_upT || !ov->n_rows || ov->cap_rows < 0 || ov->C < 0) return TWELL_ERR_INVALID_ARG;
    if (ov->cap_rows > 0 && (!ov->rows || !ov->dense)) return TWELL_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W_upT) & 15u) != 0 ||
        (ov->dense && (reinterpret_cast<uintptr_t>(ov->dense) & 15u) != 0))
        return TWELL_ERR_INVALID_ARG;
    const int M = h->M, F = h->F, T = h->T;
    const size_t need = twell_hybrid_bwd_workspace_bytes(M, d, F, T, h->cap_slots, ov->cap_rows);
    if (need == 0) return TWELL_ERR_INVALID_ARG;
    if (!ws || ws_bytes < need) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;
    HybridBwdWs w;
    carve_hybrid_bwd(ws, M, d, F, T, h->cap_slots, ov->cap_rows, &w);

    // the TwELL rows (overflow rows are empty there): dx, dW_up, dW_down, db
    twell_status st = twell_ffn_bwd(x, W_up, W_down, h, dy, d, l1_coef, dx, dW_up, dW_down, db, w.sparse,
                                    w.sparse_bytes, status, stream);
    if (st != TWELL_OK || ov->cap_rows == 0) return st;
    const int sms = sms_now();
    if (sms <= 0) return TWELL_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int cap = ((ov->cap_rows + kRowPad - 1) / kRowPad) * kRowPad;
    const int32_t* n = ov->n_rows;

    count_launches(2);
    k_gather_rows<<<cap, 256, 0, s>>>(dy, d, ov->rows, n, ov->cap_rows, cap, w.dyR);
    k_gather_rows<<<cap, 256, 0, s>>>(x, d, ov->rows, n, ov->cap_rows, cap, w.xR);
    cudaError_t e = cudaGetLastError();
    // dpre_R = (dy_R W_down^T + l1) where h_R != 0
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.dyR, W_down, ov->cap_rows, n, F, d, w.dpre, F, 0, ov->dense, F, l1_coef, status, sms, s);
    if (e == cudaSuccess) {
        count_launches(2);
        k_split_rows<<<cap, 256, 0, s>>>(w.dpre, F, n, ov->cap_rows, cap, w.hi, w.lo);
        k_colsum_add<<<(F + 255) / 256, 256, 0, s>>>(w.dpre, F, n, ov->cap_rows, db);
        e = cudaGetLastError();
    }
    // dx[R] = (hi + lo) W_up, fp32, then bf16 rows into dx
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.hi, W_upT, ov->cap_rows, n, d, F, w.dxR, d, 0, nullptr, 0, 0.f, status, sms, s);
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.lo, W_upT, ov->cap_rows, n, d, F, w.dxR, d, 1, nullptr, 0, 0.f, status, sms, s);
    if (e == cudaSuccess) {
        count_launches(1);
        k_scatter_rows_bf16<<<ov->cap_rows, 256, 0, s>>>(w.dxR, d, ov->rows, n, ov->cap_rows, dx);
        e = cudaGetLastError();
    }
    // transposed operands for the weight gradients (token axis innermost)
    if (e == cudaSuccess) {
        const dim3 blk(32, 8);
        const dim3 gF((F + 31) / 32, cap / 32), gd((d + 31) / 32, cap / 32);
        count_launches(5);
        k_transpose<<<gF, blk, 0, s>>>(w.hi, F, n, ov->cap_rows, cap, w.hiT);
        k_transpose<<<gF, blk, 0, s>>>(w.lo, F, n, ov->cap_rows, cap, w.loT);
        k_transpose<<<gF, blk, 0, s>>>(ov->dense, F, n, ov->cap_rows, cap, w.hT);
        k_transpose<<<gd, blk, 0, s>>>(w.xR, d, n, ov->cap_rows, cap, w.xRT);
        k_transpose<<<gd, blk, 0, s>>>(w.dyR, d, n, ov->cap_rows, cap, w.dyRT);
        e = cudaGetLastError();
    }
    // dW_up += (hi + lo)^T x_R, dW_down += h_R^T dy_R
    // (the token axis is their depth: only the live rows, read from the device count)
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.hiT, w.xRT, F, nullptr, d, cap, dW_up, d, 1, nullptr, 0, 0.f, status, sms, s, n);
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.loT, w.xRT, F, nullptr, d, cap, dW_up, d, 1, nullptr, 0, 0.f, status, sms, s, n);
    if (e == cudaSuccess)
        e = dense_gemm_f32(w.hT, w.dyRT, F, nullptr, d, cap, dW_down, d, 1, nullptr, 0, 0.f, status, sms, s, n);
    return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
