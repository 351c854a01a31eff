// launch.h — host-side launchers of the TwELL kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace twell {

// Kernels launched by this library in this process (read by twell_kernel_launches).
extern std::atomic<long long> g_kernel_launches;
inline void count_launches(int n) { g_kernel_launches.fetch_add(n, std::memory_order_relaxed); }

// Measurement hook (twell_set_kernel_timer): events recorded around one call site.
struct KernelTimer {
    int site;
    cudaEvent_t begin, end;
};
extern KernelTimer g_timer;
inline void timer_begin(int site, cudaStream_t s)
{
    if (g_timer.site == site && g_timer.begin) cudaEventRecord(g_timer.begin, s);
}
inline void timer_end(int site, cudaStream_t s)
{
    if (g_timer.site == site && g_timer.end) cudaEventRecord(g_timer.end, s);
}

// Device view of a TwELL (same fields as the public twell_buf).
struct TwellView {
    int M, F, T, n_tiles;
    int64_t cap;
    int32_t* nnz;
    int32_t* K;
    int64_t* off;
    int32_t* idx;
    uint16_t* val;
};

// ---- TwELL construction (twell_sparse.cu)
// nnz[r] of a dense bf16 matrix.
cudaError_t launch_count_dense(const uint16_t* h, int ldh, const TwellView& tw, int32_t* status, cudaStream_t s);
// K[t] = max nnz over tile t, off[] = compact prefix; capacity check.
cudaError_t launch_tile_layout(const TwellView& tw, int32_t* status, cudaStream_t s);
// Slots from a dense bf16 matrix.
cudaError_t launch_fill_dense(const uint16_t* h, int ldh, const TwellView& tw, int32_t* status, cudaStream_t s);
// Slots from GEMM-epilogue staging. ReLU staging: uint32 (bf16 << 16 | local col);
// gate staging: uint2 (global col, fp32 gate bits) and gate values go to gval[slot].
// ov_pos (hybrid format, else null): rows with ov_pos[r] >= 0 are left empty.
cudaError_t launch_fill_staged_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int stride,
                                    const TwellView& tw, const int32_t* ov_pos, int32_t* status, cudaStream_t s);
// Layout and fill of a ReLU TwELL in one launch (tile widths and offsets
// recomputed by every block), for n_tiles <= the fused kernel's limit.
bool fused_fill_ok(int n_tiles);
cudaError_t launch_layout_fill_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int stride,
                                    const TwellView& tw, int sm_count, int32_t* status, cudaStream_t s);
// Hybrid format: overflow rows (nnz > C) in ascending order, nnz of those rows
// set to 0 (run before launch_tile_layout), then their dense hidden rows.
cudaError_t launch_overflow_rows(const TwellView& tw, int C, int cap_rows, int32_t* ov_pos, int32_t* ov_rows,
                                 int32_t* n_rows, int32_t* status, cudaStream_t s);
cudaError_t launch_overflow_dense(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int F,
                                  const int32_t* ov_rows, const int32_t* n_rows, int cap_rows, uint16_t* dense,
                                  const int32_t* status, cudaStream_t s);
cudaError_t launch_fill_staged_gate(const uint2* stage, const int32_t* stage_cnt, int NB, int BM,
                                    const TwellView& tw, float* gval, int32_t* status, cudaStream_t s);

// One-block layout + fill for small problems (M <= 1024, M * NB <= 8192).
bool small_fill_ok(int M, int NB);
cudaError_t launch_layout_fill_small_gate(const uint2* stage, const int32_t* stage_cnt, int NB, int BM,
                                          const TwellView& tw, float* gval, int32_t* status, cudaStream_t s);
cudaError_t launch_layout_fill_small_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN,
                                          int stride, const TwellView& tw, int32_t* status, cudaStream_t s);

// ---- Sparse products (twell_sparse.cu)
// y[r,:] = sum_k v[r,k] * W[idx[r,k], :]; v is the TwELL's bf16 val (vals_f32 == nullptr)
// or an fp32 array indexed by slot.
cudaError_t launch_spmm_rows(const TwellView& tw, const float* vals_f32, const uint16_t* W, int d,
                             uint16_t* y, int32_t* status, cudaStream_t s);
// The SDDMM's dot products dy[r] . W[idx] on the stored slots, over column
// slices of up to 1024 columns: part holds sddmm_slices(d) * tw.cap floats of
// per-slice sums (workspace). launch_sddmm_combine_scatter (after the column
// lists' index kernels) then adds them into dpre[slot] (+ l1 on stored slots,
// 0 on padding) and scatters every entry's row, h and dpre into the lists.
int sddmm_slices(int d);
cudaError_t launch_sddmm_slices(const TwellView& tw, const uint16_t* dy, const uint16_t* W, int d, float* part,
                                int32_t* status, cudaStream_t s);
// Gated: val[slot] = bf16(relu(g) * (x[r] . W_up[idx])) on stored slots.
cudaError_t launch_gated_up(const TwellView& tw, const uint16_t* x, const uint16_t* W_up, int d,
                            const float* gval, int32_t* status, cudaStream_t s);

// ---- Column lists (CSC) of a TwELL, rows ascending inside a column
struct CscWork {
    int row_blocks, rows_per_block;
    unsigned long long* masks;  // [row_blocks, F]
    int32_t* start;             // [row_blocks, F]
    int32_t* colcnt;            // [F]
    int32_t* colptr;            // [F + 1]
    int32_t* crow;              // [cap] row of each column-list entry
    uint16_t* cval;             // [cap] its h (bf16)
    float* cdpre;               // [cap] its dpre
};
void csc_plan(int M, int F, int* row_blocks, int* rows_per_block);
// Column lists of the stored entries: masks, per-(block, column) starts and
// column pointers (the TwELL indices only) ...
cudaError_t launch_csc_lists(const TwellView& tw, const CscWork& w, int32_t* status, cudaStream_t s);
// ... then dpre from the SDDMM's slice sums, and every entry's row, h and dpre
// at its place in the lists.
cudaError_t launch_sddmm_combine_scatter(const TwellView& tw, int d, const float* part, float l1, float* dpre,
                                         const CscWork& w, int32_t* status, cudaStream_t s);
// dW_down[j] = sum h dy[r], dW_up[j] = sum dpre x[r], db[j] = sum dpre over column j.
cudaError_t launch_wgrad(const TwellView& tw, const CscWork& w, const float* dpre, const uint16_t* x,
                         const uint16_t* dy, int d, float* dW_up, float* dW_down, float* db, int32_t* status,
                         cudaStream_t s);

// ---- tcgen05 GEMM (twell_gemm.cu)
enum GemmMode { GEMM_TWELL_RELU = 0, GEMM_GATE_SWAP = 1, GEMM_DENSE = 2 };
// ---- gated decode tail (twell_sparse.cu): layout, fill, gated up and
// down-projection in one cooperative launch; y == nullptr skips the
// down-projection. `counter` must be 0 when it starts (grid barrier).
bool decode_tail_ok(int M, int NB, int n_tiles);
// Bounded-wait self-test: which 0 = mbarrier, 1 = grid barrier (*counter must be 0).
cudaError_t launch_wait_selftest(int which, int32_t* counter, int32_t* status, cudaStream_t s);
cudaError_t launch_decode_tail(const uint2* gstage, const int32_t* stage_cnt, int NB, int BM, const uint16_t* x,
                               const uint16_t* W_up, const uint16_t* W_down, int d, const TwellView& tw,
                               uint16_t* y, int32_t* counter, int32_t* status, cudaStream_t s);

struct GemmArgs {
    int rowsA, rowsB, K;   // A [rowsA, K], B [rowsB, K] bf16, K-major unless a_mn / b_mn
    int a_mn, b_mn;        // DENSE only: the operand is stored MN-major, i.e. as [K, rowsA] ([K, rowsB])
                           //   row-major (its transpose); the GEMM then runs on CTA pairs only
    const float* bias;     // TWELL_RELU: per B row; GATE_SWAP: per A row; DENSE: per B row or null
    int relu;              // DENSE only
    uint32_t* stage;       // TWELL_RELU staging [rowsA, NB, stage_cap]
    int stage_cap;         // TWELL_RELU: entries a (row, BN-column block) segment holds (<= BN)
    uint2* gstage;         // GATE_SWAP staging [rowsB, NB, 128]
    int32_t* stage_cnt;    // [rows, NB]
    int32_t* nnz;          // [rows], zeroed by the caller before the launch; null: not counted
    int32_t* zero_word;    // if set, written 0 by the kernel (a counter the next kernel starts from)
    const int32_t* rowsA_dev;  // if set, rows of A actually used: min(*rowsA_dev, rowsA), read on the device
    const int32_t* K_dev;      // if set, depth actually used: *K_dev rounded up to 64, at most K, read on the
                               //   device (both operands must be zero between *K_dev and that rounding)
    const int32_t* row_map;    // DENSE only: if set, output row of A's row i is row_map[i]
    const void* pf0;           // GATE_SWAP: rows of pf0 and pf1 (pf_row_bytes each) of the
    const void* pf1;           //   active units are prefetched into L2 (pf_row_bytes 0: off)
    int pf_row_bytes;
    int NB;                // column blocks of the staging
    uint16_t* out;         // DENSE output [rowsA, ldo] bf16
    int ldo;
    float* out_f32;        // DENSE: if set, fp32 output [rowsA, ldo] instead of out
    int accumulate;        //   out_f32 += result (else =)
    const uint16_t* mask;  //   if set, [rowsA, ldm] bf16: result kept only where mask is nonzero
    int ldm;
    float add_scalar;      //   added to every result before the mask (fp32 and bf16 outputs)
    float* colsum;         // DENSE, bf16 output only: if set, column sums of the (masked) fp32 results per
                           //   128-row block: colsum[(row / 128) * ldc + col]
    int ldc;
    int32_t* status;
};
// ---- Down-projection on the tensor cores over token-group unions (twell_union.cu)
struct UnionWork {
    int32_t* ucnt;     // [groups] |U| of each 128-token group
    int32_t* ulist;    // [groups * F + 64] ascending active units of each group
    int32_t* kbptr;    // [groups, kb_stride] bucket starts per 64-deep k-block of U
    int kb_stride;     // union_kb_stride(F)
    int64_t* gbase;    // [groups] first TwELL slot of the group
    uint32_t* ent;     // [cap + 4] bucketed entries (bf16 | pos % 64 << 16 | row << 22)
};
int union_kb_stride(int F);
size_t union_smem_bytes(int F);  // shared memory of the GEMM kernel
cudaError_t launch_union_build(const TwellView& tw, const UnionWork& w, int32_t* status, cudaStream_t s);
cudaError_t launch_spmm_union(const TwellView& tw, const uint16_t* W, int d, const UnionWork& w, uint16_t* y,
                              int32_t* status, cudaStream_t s);

// Returns the column-block width BN the GEMM uses for this mode/shape.
int gemm_block_n(int mode, int rowsB);
cudaError_t launch_gemm(int mode, const uint16_t* A, const uint16_t* B, const GemmArgs& a, int sm_count,
                        cudaStream_t s);

}  // namespace twell
