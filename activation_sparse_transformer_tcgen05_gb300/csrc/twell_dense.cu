// twell_dense.cu — the dense baseline layer, forward and backward.
//
// The same ReLU feed-forward layer and L1 loss as the TwELL path, computed
// with dense tcgen05 GEMMs on CTA pairs: the comparison the sparse path is
// measured against ("Sparser, Faster, Lighter Transformer Language Models",
// Resumo Técnico §4 Resultados compares against the dense model). Nothing here
// is part of the method.
//
// Backward of L = <dy, y> + l1 sum|h| with h = relu(x W_up^T + b), y = h W_down:
//   G1  dpre    = (dy W_down^T + l1) * 1[h != 0]   A = dy (K-major), B = W_down (K-major);
//               bf16 output, per-128-row column sums of the fp32 values for db
//   G2  dx      = dpre W_up                        A = dpre (K-major), B = W_up (MN-major)
//   G3  dW_up   = dpre^T x                         A = dpre (MN-major), B = x (MN-major)
//   G4  dW_down = h^T dy                           A = h (MN-major), B = dy (MN-major)
//   db  = the column sums of G1 added over the row blocks in order
// MN-major operands are read through their own TMA layout (two 64-wide boxes
// per CTA half), so no operand is transposed in memory.
#include "common.cuh"
#include "launch.h"

namespace twell {
namespace {

// db[j] = sum over row blocks b (ascending) of part[b * F + j].
__global__ void k_rowblock_sum(const float* __restrict__ part, int nblocks, int F, float* __restrict__ db)
{
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= F) return;
    float s = 0.f;
    for (int b = 0; b < nblocks; ++b) s += part[(size_t)b * F + j];
    db[j] = s;
}

int sms_current()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return 0;
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dims_ok(int M, int d, int F) { return M > 0 && d > 0 && F > 0 && d % 8 == 0 && F % 8 == 0; }

constexpr int kRowBlock = 128;  // rows per column-sum block of G1's epilogue

size_t carve(void* ws, int M, int F, uint16_t** dpre, float** part)
{
    const size_t dpre_bytes = ((size_t)M * F * 2 + 255) & ~size_t(255);
    const size_t nb = (size_t)((M + kRowBlock - 1) / kRowBlock);
    if (ws) {
        *dpre = static_cast<uint16_t*>(ws);
        *part = reinterpret_cast<float*>(static_cast<char*>(ws) + dpre_bytes);
    }
    return dpre_bytes + nb * F * 4;
}

}  // namespace
}  // namespace twell

using namespace twell;

extern "C" twell_status twell_dense_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const float* b,
                                            const uint16_t* W_down, int M, int d, int F, uint16_t* h_dense,
                                            uint16_t* y, int32_t* status, void* stream)
{
    if (!x || !W_up || !W_down || !h_dense || !y || !status || !dims_ok(M, d, F)) return TWELL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(h_dense) || !aligned16(y))
        return TWELL_ERR_INVALID_ARG;
    const int sms = sms_current();
    if (sms <= 0) return TWELL_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmArgs g1{};
    g1.rowsA = M;
    g1.rowsB = F;
    g1.K = d;
    g1.bias = b;
    g1.relu = 1;
    g1.out = h_dense;
    g1.ldo = F;
    g1.status = status;
    cudaError_t e = launch_gemm(GEMM_DENSE, x, W_up, g1, sms, s);
    GemmArgs g2{};
    g2.rowsA = M;
    g2.rowsB = d;
    g2.K = F;
    g2.b_mn = 1;  // W_down [F, d]: K = F rows, N = d contiguous
    g2.out = y;
    g2.ldo = d;
    g2.status = status;
    if (e == cudaSuccess) e = launch_gemm(GEMM_DENSE, h_dense, W_down, g2, sms, s);
    return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

extern "C" size_t twell_dense_bwd_workspace_bytes(int M, int d, int F)
{
    if (!dims_ok(M, d, F)) return 0;
    return carve(nullptr, M, F, nullptr, nullptr);
}

extern "C" twell_status twell_dense_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down,
                                            const uint16_t* h_dense, const uint16_t* dy, int M, int d, int F,
                                            float l1_coef, uint16_t* dx, float* dW_up, float* dW_down, float* db,
                                            void* ws, size_t ws_bytes, int32_t* status, void* stream)
{
    if (!x || !W_up || !W_down || !h_dense || !dy || !dx || !dW_up || !dW_down || !db || !status ||
        !dims_ok(M, d, F))
        return TWELL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(h_dense) || !aligned16(dy) ||
        !aligned16(dx) || !aligned16(dW_up) || !aligned16(dW_down))
        return TWELL_ERR_INVALID_ARG;
    const size_t need = carve(nullptr, M, F, nullptr, nullptr);
    if (!ws || ws_bytes < need) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;
    const int sms = sms_current();
    if (sms <= 0) return TWELL_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* dpre = nullptr;
    float* part = nullptr;
    carve(ws, M, F, &dpre, &part);

    // G1: dpre = (dy W_down^T + l1) where h != 0; column sums per 128 rows
    GemmArgs g1{};
    g1.rowsA = M;
    g1.rowsB = F;
    g1.K = d;
    g1.out = dpre;
    g1.ldo = F;
    g1.mask = h_dense;
    g1.ldm = F;
    g1.add_scalar = l1_coef;
    g1.colsum = part;
    g1.ldc = F;
    g1.status = status;
    cudaError_t e = launch_gemm(GEMM_DENSE, dy, W_down, g1, sms, s);
    if (e == cudaSuccess) {
        count_launches(1);
        k_rowblock_sum<<<(F + 255) / 256, 256, 0, s>>>(part, (M + kRowBlock - 1) / kRowBlock, F, db);
        e = cudaGetLastError();
    }
    // G2: dx = dpre W_up
    GemmArgs g2{};
    g2.rowsA = M;
    g2.rowsB = d;
    g2.K = F;
    g2.b_mn = 1;
    g2.out = dx;
    g2.ldo = d;
    g2.status = status;
    if (e == cudaSuccess) e = launch_gemm(GEMM_DENSE, dpre, W_up, g2, sms, s);
    // G3: dW_up = dpre^T x ; G4: dW_down = h^T dy (fp32)
    GemmArgs g3{};
    g3.rowsA = F;
    g3.rowsB = d;
    g3.K = M;
    g3.a_mn = 1;
    g3.b_mn = 1;
    g3.out_f32 = dW_up;
    g3.ldo = d;
    g3.status = status;
    if (e == cudaSuccess) e = launch_gemm(GEMM_DENSE, dpre, x, g3, sms, s);
    GemmArgs g4 = g3;
    g4.out_f32 = dW_down;
    if (e == cudaSuccess) e = launch_gemm(GEMM_DENSE, h_dense, dy, g4, sms, s);
    return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
