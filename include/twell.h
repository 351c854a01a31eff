/*
 * twell.h — C ABI of the TwELL activation-sparse feed-forward layer (sm_103a).
 *
 * The layer is the ReLU (or ReLU-gated) transformer feed-forward block of
 * "Sparser, Faster, Lighter Transformer Language Models" (Cetin, Peluchetti,
 * Castillo, Naruse, Murakami, Jones, 2026; gist.science summary, Resumo Técnico
 * §2 Metodologia). L1-regularised training leaves more than 99 % of the hidden
 * activations at zero; the post-ReLU hidden matrix h is packed into TwELL
 * (Tile-wise ELLPACK) straight from the up-projection's epilogue, and the
 * down-projection and the backward run only over the stored entries.
 *
 * TwELL layout (one tile = T consecutive token rows spanning all F hidden units):
 *   nnz_row[r]   number of active entries of row r
 *   K_tile[t]    max nnz_row over the rows of tile t (the tile's width)
 *   tile_off[t]  first slot of tile t; tile_off[0] = 0,
 *                tile_off[t+1] = tile_off[t] + rows(t) * K_tile[t],
 *                rows(t) = min(T, M - t*T)
 *   slot off[t] + i*K[t] + k of row i of tile t holds, for k < nnz, the k-th
 *   active column in ascending order (idx, int32) and h there (val, bf16 bits);
 *   for k >= nnz it holds idx = -1, val = +0.
 * Active set: h != 0 for the ReLU layer and for twell_pack (-0 counts as zero,
 * NaN as nonzero); pre_gate > 0 for the gated layer.
 *
 * Conventions for every entry point:
 *   - Pointers named in the argument list are DEVICE pointers unless marked
 *     "host". bf16 tensors are passed as uint16_t bit arrays; all matrices are
 *     row-major and densely packed (row stride = column count) unless a leading
 *     dimension is given. Weights are [F, d]: one row per hidden unit.
 *   - The caller owns and allocates every buffer. The library never allocates
 *     memory, frees or synchronises (twell_check is the one call that
 *     synchronises); each call only enqueues work on `stream` (a cudaStream_t
 *     passed as void*, NULL = the legacy default stream) and returns. Buffers
 *     must stay alive until that work has finished. twell_ffn_bwd forks part
 *     of its work onto a library stream and joins it back through events: one
 *     stream and two events per host thread and device, created by the first
 *     call that is not being stream-captured and kept until the process ends
 *     (cudaDeviceReset invalidates them; later backward calls on that thread
 *     and device then return TWELL_ERR_CUDA).
 *   - Host-side argument errors are returned at once and nothing is enqueued.
 *     Errors found on the device (capacity, bounded-wait timeout) are written
 *     to `*status`, a caller-owned device int32 that the caller sets to 0
 *     before the first call; the first nonzero code sticks and later kernels of
 *     the same call skip their work. Read it after synchronising the stream, or
 *     with twell_check().
 *   - Alignment: every device pointer of a bf16 matrix must be 16-byte aligned
 *     and d, F must be multiples of 8 (128-bit loads, TMA strides).
 *   - All calls are deterministic: the same inputs give the same bits.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum twell_status {
    TWELL_OK = 0,
    TWELL_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, misaligned pointer, bad d/F */
    TWELL_ERR_UNSUPPORTED = 2, /* shape or mode this build does not implement */
    TWELL_ERR_WORKSPACE = 3,   /* ws_bytes smaller than twell_workspace_bytes() */
    TWELL_ERR_CAPACITY = 4,    /* device: TwELL needs more slots than cap_slots */
    TWELL_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel expired */
    TWELL_ERR_CUDA = 6         /* a CUDA runtime call or launch failed */
} twell_status;

/* Host struct describing one TwELL held in device memory (layout above).
 * M, F, T, n_tiles = ceil(M/T) and cap_slots are set by the caller; the five
 * device arrays are caller-allocated: nnz_row[M], K_tile[n_tiles],
 * tile_off[n_tiles+1], idx[cap_slots], val[cap_slots]. */
typedef struct twell_buf {
    int32_t M, F, T, n_tiles;
    int64_t cap_slots;
    int32_t* nnz_row;
    int32_t* K_tile;
    int64_t* tile_off;
    int32_t* idx;
    uint16_t* val;
} twell_buf;

/* Operation codes for twell_workspace_bytes. */
enum { TWELL_OP_PACK = 0, TWELL_OP_SPMM_DOWN = 1, TWELL_OP_FFN_FWD = 2,
       TWELL_OP_FFN_BWD = 3, TWELL_OP_GATED_FWD = 4, TWELL_OP_HYBRID_FWD = 5 };

/* Human-readable name of a status code (static string, never NULL). */
const char* twell_status_string(int status);

/* Worst-case slot count of a TwELL of an M x F matrix with tile height T:
 * M*F (every entry active). Returns -1 for non-positive sizes. */
int64_t twell_buf_slots_bound(int M, int F, int T);

/* Device workspace, in bytes, that `op` needs for these sizes. cap_slots is the
 * TwELL capacity (used by TWELL_OP_FFN_BWD and TWELL_OP_GATED_FWD). 0 means
 * none is needed. */
size_t twell_workspace_bytes(int op, int M, int d, int F, int T, int64_t cap_slots);

/*
 * twell_fwd_workspace_bytes — workspace of the ReLU forward (twell_up_pack /
 * twell_ffn_fwd without a gate) whose up-projection epilogue stages at most
 * stage_cap nonzeros per (row, 256-column block): the capacity the method
 * predicts for N_nz (Resumo Técnico §2, "Formato Híbrido para Treinamento").
 * stage_cap is 256, 64 or 32 (the capacities the epilogue is compiled for);
 * 256 never overflows and equals twell_workspace_bytes(TWELL_OP_FFN_FWD, ...).
 * The forward uses the largest of them its ws_bytes allows; a block with more
 * nonzeros than that makes the call report TWELL_ERR_CAPACITY. Returns 0 for
 * invalid arguments.
 */
size_t twell_fwd_workspace_bytes(int M, int d, int F, int T, int64_t cap_slots, int stage_cap);

/* Number of streaming multiprocessors the library sizes its grids for. */
int twell_device_sm_count(void);

/*
 * twell_pack — TwELL of a dense hidden matrix (the "Formato de Dados TwELL"
 * paragraph of Resumo Técnico §2).
 *   h      [M, ldh] bf16, entries (r, j < F) are read; ldh >= F, ldh % 8 == 0
 *   out    host struct with out->M == M, out->F == F, out->T == T
 * Writes nnz_row, K_tile, tile_off always; writes the slots only if
 * tile_off[n_tiles] <= cap_slots, else sets *status = TWELL_ERR_CAPACITY.
 */
twell_status twell_pack(const uint16_t* h, int M, int F, int ldh, int T,
                        const twell_buf* out, int32_t* status, void* stream);

/*
 * twell_up_pack — rows a1-a3 of the forward alone: the tcgen05 up (or gate)
 * projection whose epilogue packs h into h_out, without the down-projection.
 * Same arguments, workspace and error behaviour as twell_ffn_fwd minus W_down
 * and y; in gated mode h_out's val holds h = bf16(relu(g) * u) on return.
 * twell_ffn_fwd is exactly twell_up_pack followed by twell_spmm_down.
 */
twell_status twell_up_pack(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate,
                           const float* b, int M, int d, int F, int T, const twell_buf* h_out,
                           void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * twell_spmm_down — y = h W_down over the stored entries of a TwELL (Resumo
 * Técnico §2, "Kernels de Inferência": iterate only over the active neurons).
 *   h       host struct of a valid TwELL (F rows of W_down are indexed)
 *   W_down  [F, d] bf16
 *   y       [M, d] bf16 output; fp32 accumulation, one rounding to bf16
 */
twell_status twell_spmm_down(const twell_buf* h, const uint16_t* W_down, int d,
                             uint16_t* y, int32_t* status, void* stream);

/*
 * twell_spmm_down_tc — the same product y = h W_down on the tensor cores
 * (Resumo Técnico §2, "Kernels de Inferência": only the active neurons are
 * visited and the tensor cores do the multiplication). For each group of 128
 * consecutive tokens, U is the ascending union of their active units; then
 * y[group] = h[group, U] W_down[U, :] runs as one tcgen05 GEMM with K = |U|
 * (A built in shared memory from the TwELL, B the gathered rows of W_down).
 * Same arguments, result and error behaviour as twell_spmm_down, plus:
 *   ws        device workspace of at least
 *             twell_spmm_down_tc_workspace_bytes(h->M, h->F, h->cap_slots)
 *             bytes, 256-byte aligned; contents are scratch
 * h->F must be a multiple of 8 and at most 65536, and the device must offer
 * the kernel's shared memory (about 227 KB per block; else
 * TWELL_ERR_UNSUPPORTED). y equals twell_spmm_down's up to fp32 summation
 * order. Launches two kernels: the groups' unions and entry buckets, then the
 * GEMM.
 */
size_t twell_spmm_down_tc_workspace_bytes(int M, int F, int64_t cap_slots);
twell_status twell_spmm_down_tc(const twell_buf* h, const uint16_t* W_down, int d, uint16_t* y,
                                void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * twell_ffn_fwd — the layer's forward pass.
 *   ReLU  (W_gate == NULL): h = relu(x W_up^T + b), packed into TwELL inside the
 *          tcgen05 up-projection's epilogue (Resumo Técnico §2: TwELL materialised
 *          in the epilogue of the dense matmul), then y = h W_down.
 *   Gated (W_gate != NULL): the gate GEMM x W_gate^T + b gives the active set and
 *          is packed the same way; then for each active (r, j):
 *          u = x[r] . W_up[j], h = bf16(relu(g) * u), y[r] += h W_down[j] (the
 *          sparse up+down inference kernels of the same section).
 *   x [M, d] bf16; W_up, W_gate, W_down [F, d] bf16; b [F] fp32 (added to the
 *   ReLU pre-activation, or to the gate); y [M, d] bf16.
 *   h_out: TwELL of h (M, F, T as given), its val holding h.
 *   ws: device workspace of at least twell_workspace_bytes(TWELL_OP_FFN_FWD or
 *   TWELL_OP_GATED_FWD, M, d, F, T, h_out->cap_slots) bytes, 256-byte aligned;
 *   contents need no init.
 * Capacity overflow of h_out: nnz/K/off are written, slots and y are not, and
 * *status = TWELL_ERR_CAPACITY.
 */
twell_status twell_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate,
                           const float* b, const uint16_t* W_down, int M, int d, int F, int T,
                           const twell_buf* h_out, uint16_t* y, void* ws, size_t ws_bytes,
                           int32_t* status, void* stream);

/*
 * Hybrid format (Resumo Técnico §2, "Formato Híbrido para Treinamento"): rows
 * are partitioned dynamically; a row with more than C nonzeros is an overflow
 * row and goes to a dense backup matrix, every other row stays in the TwELL.
 * Overflow rows are empty rows of the TwELL (nnz 0), so every TwELL entry point
 * applies to the TwELL part unchanged.
 *   C         ELL capacity per row, >= 0
 *   cap_rows  rows the dense block can hold, >= 0
 *   n_rows    [1] int32 device, written: number of overflow rows
 *   rows      [cap_rows] int32 device, written: overflow row ids, ascending
 *   dense     [cap_rows, F] bf16 device, written: row i is the hidden row of
 *             rows[i] (all F columns, zeros included)
 * More than cap_rows overflow rows: *status = TWELL_ERR_CAPACITY and the first
 * cap_rows are kept. All arrays are caller-owned.
 */
typedef struct {
    int32_t C;
    int32_t cap_rows;
    int32_t* n_rows;
    int32_t* rows;
    uint16_t* dense;
} twell_overflow;

/*
 * twell_hybrid_up_pack — ReLU up-projection (as twell_up_pack) packed into the
 * hybrid format: h_out holds the rows with nnz <= ov->C, ov the others.
 *   x [M, d] bf16; W_up [F, d] bf16; b [F] fp32; ws: at least
 *   twell_workspace_bytes(TWELL_OP_HYBRID_FWD, M, d, F, T, 0) bytes,
 *   256-byte aligned.
 */
twell_status twell_hybrid_up_pack(const uint16_t* x, const uint16_t* W_up, const float* b, int M, int d, int F,
                                  int T, const twell_buf* h_out, const twell_overflow* ov, void* ws,
                                  size_t ws_bytes, int32_t* status, void* stream);

/*
 * twell_hybrid_spmm_down — y = h W_down on the hybrid format: the TwELL rows by
 * the sparse down-projection (twell_spmm_down), the overflow rows by the
 * tcgen05 dense GEMM on ov->dense, its output rows placed by ov->rows.
 *   W_down [F, d] bf16 (rows gathered by the TwELL part); W_downT [d, F] bf16,
 *   the same matrix transposed (the dense GEMM's K-major operand); y [M, d]
 *   bf16, every row written.
 */
twell_status twell_hybrid_spmm_down(const twell_buf* h, const twell_overflow* ov, const uint16_t* W_down,
                                    const uint16_t* W_downT, int d, uint16_t* y, int32_t* status, void* stream);

/* twell_hybrid_ffn_fwd — twell_hybrid_up_pack followed by twell_hybrid_spmm_down. */
twell_status twell_hybrid_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const float* b, const uint16_t* W_down,
                                  const uint16_t* W_downT, int M, int d, int F, int T, const twell_buf* h_out,
                                  const twell_overflow* ov, uint16_t* y, void* ws, size_t ws_bytes,
                                  int32_t* status, void* stream);

/*
 * twell_hybrid_ffn_bwd — the backward of twell_ffn_bwd (same loss, outputs,
 * layouts and determinism) for a layer whose forward ran on the hybrid format
 * (Resumo Técnico §2, "Formato Híbrido para Treinamento"): the TwELL rows of h
 * through the sparse kernels, the dense overflow rows of ov through tcgen05
 * GEMMs (dpre of those rows masked by their h, dx rows, and their shares of
 * dW_up, dW_down and db added to the sparse part's).
 *   W_upT [d, F] bf16: W_up transposed (K-major operand of the dense dx).
 *   ws: at least twell_hybrid_bwd_workspace_bytes(M, d, F, T, h->cap_slots,
 *   ov->cap_rows) bytes, 256-byte aligned. Limits as twell_ffn_bwd.
 * The overflow rows' dpre enters the GEMMs as the sum of two bf16 parts
 * (~2^-17 relative), accumulated in fp32.
 */
size_t twell_hybrid_bwd_workspace_bytes(int M, int d, int F, int T, int64_t cap_slots, int cap_rows);
twell_status twell_hybrid_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down,
                                  const uint16_t* W_upT, const twell_buf* h, const twell_overflow* ov,
                                  const uint16_t* dy, int d, float l1_coef, uint16_t* dx, float* dW_up,
                                  float* dW_down, float* db, void* ws, size_t ws_bytes, int32_t* status,
                                  void* stream);

/*
 * twell_ffn_bwd — backward of L = <dy, y> + l1_coef * sum |h| for the ReLU
 * layer (Resumo Técnico §2, "Técnicas de Treinamento": L1 on the ReLU
 * activations), restricted to the stored entries of h:
 *   dpre[r,j] = (dy[r] . W_down[j] + l1_coef) on active (r, j), 0 elsewhere
 *   dx        = dpre W_up                       [M, d] bf16
 *   dW_up     = dpre^T x                        [F, d] fp32 (every row written)
 *   dW_down   = h^T dy                          [F, d] fp32 (every row written)
 *   db        = column sums of dpre             [F]    fp32
 *   x, dy [M, d] bf16; W_up, W_down [F, d] bf16; M and F are h->M and h->F.
 *   h: the forward's TwELL; ws: at least twell_workspace_bytes(TWELL_OP_FFN_BWD,
 *   M, d, F, T, h->cap_slots) bytes, 256-byte aligned (it grows with d: the
 *   dot products of dpre are summed over column slices of 1024, one fp32 per
 *   stored slot and slice). Limit of this build: h->cap_slots < 2^31 (else
 *   TWELL_ERR_UNSUPPORTED).
 * The reduction order of every sum is fixed (no floating-point atomics).
 * The column lists' index-only kernels run on the library's side stream while
 * the SDDMM runs on `stream`; the call's work is complete when `stream`'s is.
 */
twell_status twell_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down,
                           const twell_buf* h, const uint16_t* dy, int d, float l1_coef,
                           uint16_t* dx, float* dW_up, float* dW_down, float* db,
                           void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * twell_dense_ffn_fwd — the same ReLU layer computed densely with the same
 * tcgen05 GEMM (a baseline for the sparse path, not part of the method):
 *   h_dense = bf16(relu(x W_up^T + b))   [M, F] bf16 (written; the dense
 *                                        backward's mask)
 *   y       = h_dense W_down             [M, d] bf16
 * Every argument has the layout of twell_ffn_fwd's; W_down [F, d] is read as
 * the MN-major operand of the second GEMM (no transposed copy). All pointers
 * 16-byte aligned; d % 8 == 0, F % 8 == 0. Runs on CTA pairs (TWELL_ERR_CUDA
 * if a cluster of two cannot be launched).
 */
twell_status twell_dense_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const float* b,
                                 const uint16_t* W_down, int M, int d, int F,
                                 uint16_t* h_dense, uint16_t* y, int32_t* status, void* stream);

/*
 * twell_dense_ffn_bwd — backward of the dense baseline layer, the loss and
 * gradients of twell_ffn_bwd (L = <dy, y> + l1_coef * sum |h|) computed with
 * dense tcgen05 GEMMs (a baseline, not part of the method):
 *   dpre    = bf16((dy W_down^T + l1_coef) * 1[h_dense != 0])  [M, F] (workspace)
 *   db      = sum over rows of the fp32 values before that rounding
 *   dx      = dpre W_up          [M, d] bf16
 *   dW_up   = dpre^T x           [F, d] fp32
 *   dW_down = h_dense^T dy       [F, d] fp32
 * dpre is a bf16 GEMM operand, as in a bf16 training step. The token axis is
 * the inner dimension of the two weight-gradient GEMMs: x, dy, dpre and
 * h_dense are read as MN-major operands, so nothing is transposed.
 *   h_dense: the forward's [M, F] bf16 hidden matrix (twell_dense_ffn_fwd).
 *   ws: at least twell_dense_bwd_workspace_bytes(M, d, F) bytes, 256-byte
 *   aligned (dpre and per-128-row column sums of it).
 * All pointers 16-byte aligned; d % 8 == 0, F % 8 == 0. Fixed summation order
 * (no atomics). Runs on CTA pairs (TWELL_ERR_CUDA if a cluster of two cannot
 * be launched).
 */
size_t twell_dense_bwd_workspace_bytes(int M, int d, int F);
twell_status twell_dense_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down,
                                 const uint16_t* h_dense, const uint16_t* dy, int M, int d, int F,
                                 float l1_coef, uint16_t* dx, float* dW_up, float* dW_down, float* db,
                                 void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * twell_ffn_fwd_static_ws — twell_ffn_fwd for callers that cannot allocate
 * device memory. The paper has no counterpart; this is a convenience of this
 * library. It is meant for code that has no allocator to call (a plugin inside
 * a host framework that owns all device memory) or must not call one (a
 * latency-critical decode loop, where cudaMalloc/cudaFree synchronise the
 * device). Same arguments and results as twell_ffn_fwd, without ws/ws_bytes:
 * the workspace is a library-owned device array of TWELL_STATIC_WS_BYTES that
 * every GPU which loads the library keeps until the process exits.
 *   - Returns TWELL_ERR_WORKSPACE, with nothing enqueued, when the problem
 *     needs more workspace than the array holds: gated, when
 *     twell_workspace_bytes(TWELL_OP_GATED_FWD, M, d, F, T, h_out->cap_slots)
 *     > TWELL_STATIC_WS_BYTES; ReLU, when even the smallest epilogue staging
 *     (twell_fwd_workspace_bytes(M, d, F, T, h_out->cap_slots, 32)) does not
 *     fit. A ReLU call that fits runs with the largest staging capacity (256,
 *     64 or 32 entries per row and 256-column block) the array holds, and a
 *     block with more active units than that reports TWELL_ERR_CAPACITY in
 *     *status. Decode shapes such as M <= 64, d_model = 4096, d_ff = 14336
 *     fit in both modes, and so does the ReLU layer at M = 4096, d_model =
 *     2048, d_ff = 8192 (32-entry staging).
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress) and keeps it for the life of the process;
 *     make that first call before any stream capture. The kept address is
 *     that of the device's current context: after cudaDeviceReset on a device,
 *     do not call this entry point on it again.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents: calls whose work overlaps on the GPU (different streams, or
 *     different host threads, without ordering between them) race on it and
 *     corrupt each other's results. Serialise them, e.g. on one stream.
 *   - The allocation-free guarantee covers this call only; the caller still
 *     owns x, the weights, b, y, h_out's arrays and status.
 */
#define TWELL_STATIC_WS_BYTES (32u * 1024u * 1024u)
twell_status twell_ffn_fwd_static_ws(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate,
                                     const float* b, const uint16_t* W_down, int M, int d, int F, int T,
                                     const twell_buf* h_out, uint16_t* y, int32_t* status, void* stream);

/*
 * twell_set_kernel_timer — measurement hook. While set, every launch of the
 * kernel at call site `site` is bracketed by cudaEventRecord(ev_begin) and
 * cudaEventRecord(ev_end) on the launch's stream; ev_begin/ev_end are
 * caller-created cudaEvent_t handles passed as void*. site = 0 (or NULL
 * events) turns the hook off. Process-wide setting, not thread-safe: set it
 * from the thread that launches. Sites:
 *   1 up-projection GEMM (twell_up_pack / twell_ffn_fwd)
 *   2 sparse down-projection (twell_spmm_down / twell_ffn_fwd)
 *   3 backward SDDMM            4 backward dx
 *   5 backward column lists: the kernels that read only the TwELL indices
 *     (on the library's side stream, concurrently with the SDDMM)
 *   6 backward weight gradients
 *   7 gated decode tail (M <= 64: layout, gated up products and, in
 *     twell_ffn_fwd, the down-projection, in one launch)
 *   8 dense GEMM of the hybrid format's overflow rows (twell_hybrid_spmm_down)
 *   9 union down-projection on the tensor cores (twell_spmm_down_tc, both kernels)
 *  10 its first kernel alone (the groups' unions and entry buckets)
 */
enum { TWELL_SITE_NONE = 0, TWELL_SITE_UP_GEMM = 1, TWELL_SITE_SPMM_DOWN = 2, TWELL_SITE_SDDMM = 3,
       TWELL_SITE_DX = 4, TWELL_SITE_CSC = 5, TWELL_SITE_WGRAD = 6, TWELL_SITE_DECODE_TAIL = 7,
       TWELL_SITE_OVERFLOW_GEMM = 8, TWELL_SITE_SPMM_UNION = 9, TWELL_SITE_UNION_BUILD = 10 };
twell_status twell_set_kernel_timer(int site, void* ev_begin, void* ev_end);

/*
 * twell_wait_selftest — diagnostic of the library's bounded waits: runs a
 * wait that nothing will complete, with the same helpers the kernels use
 * (which = 0: an mbarrier no thread arrives on; which = 1: the decode tail's
 * grid barrier with a target the grid cannot reach). After its limit (about
 * one second) the wait gives up and writes TWELL_ERR_TIMEOUT to *status
 * (first error sticks); the CUDA context stays usable.
 *   scratch: one int32 of device memory (zeroed by the call).
 * Asynchronous on `stream`; TWELL_ERR_INVALID_ARG for another `which` or null
 * pointers.
 */
twell_status twell_wait_selftest(int which, int32_t* scratch, int32_t* status, void* stream);

/* Number of kernels this library has launched in this process (host-side
 * counter, all devices). Lets a caller count the library's launches in a
 * timed region. */
int64_t twell_kernel_launches(void);

/*
 * twell_check — synchronises `stream`, copies *status (device) to
 * *host_status (host) and returns TWELL_OK, or TWELL_ERR_CUDA if the stream
 * reported an error. This is the one entry point that synchronises.
 */
twell_status twell_check(const int32_t* status, void* stream, int32_t* host_status);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */
