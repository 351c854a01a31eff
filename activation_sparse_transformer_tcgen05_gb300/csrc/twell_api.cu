// twell_api.cu — the C ABI declared in include/twell.h: argument checks,
// workspace carving and the kernel sequence of each entry point. No entry
// point allocates, frees or synchronises (except twell_check).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/twell.h"
#include "launch.h"

using namespace twell;

namespace {

constexpr int kMaxDevices = 64;

int sm_count_current()
{
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A second stream and two events per (host thread, device), created on first
// use and kept until the process ends: the backward forks independent kernels
// onto it. Null if they cannot be created (the kernels then run in order).
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    int state = 0;  // 0 not tried, 1 ready, -1 unavailable
};

SideStream* side_stream(cudaStream_t caller)
{
    thread_local SideStream per_device[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream& ss = per_device[dev];
    if (ss.state == 0) {
        // never create resources while the caller's stream is being captured
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
            (void)cudaGetLastError();
            return nullptr;
        }
        const bool ok = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) == cudaSuccess &&
                        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) == cudaSuccess &&
                        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) (void)cudaGetLastError();
        ss.state = ok ? 1 : -1;
    }
    return ss.state == 1 ? &ss : nullptr;
}
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace carving: consecutive 256-byte-aligned regions.
struct Carver {
    char* base;
    size_t used = 0;
    template <typename T>
    T* take(size_t count)
    {
        T* p = reinterpret_cast<T*>(base ? base + used : nullptr);
        used = round_up(used + count * sizeof(T), 256);
        return p;
    }
};

constexpr int kReluBN = 256;  // column block of the ReLU GEMM epilogue
constexpr int kGateBM = 128;  // hidden-unit block of the gate GEMM epilogue

struct FwdWs {
    int32_t* stage_cnt;
    uint32_t* stage;
    uint2* gstage;
    float* gval;
    int32_t* counter;  // grid-barrier counter of the gated decode tail
    int32_t* ov_pos;   // hybrid: position of row r in the overflow block, or -1
};

size_t carve_fwd(void* ws, bool gated, int M, int F, int64_t cap, FwdWs* out, bool hybrid = false,
                 int stage_cap = kReluBN)
{
    Carver c{static_cast<char*>(ws)};
    FwdWs w{};
    if (!gated) {
        const size_t NB = (F + kReluBN - 1) / kReluBN;
        w.stage_cnt = c.take<int32_t>((size_t)M * NB);
        // + slack: a segment that overflows writes up to BN - cap words past its end
        w.stage = c.take<uint32_t>((size_t)M * NB * (size_t)stage_cap + (size_t)(kReluBN - stage_cap));
        if (hybrid) w.ov_pos = c.take<int32_t>((size_t)M);
    } else {
        const size_t NB = (F + kGateBM - 1) / kGateBM;
        w.stage_cnt = c.take<int32_t>((size_t)M * NB);
        w.gstage = c.take<uint2>((size_t)M * NB * kGateBM);
        w.gval = c.take<float>((size_t)(cap > 0 ? cap : 1));
        w.counter = c.take<int32_t>(1);
    }
    if (out) *out = w;
    return c.used;
}

struct BwdWs {
    float* dpre;
    float* part;  // per-column-slice SDDMM sums
    CscWork csc;
};

size_t carve_bwd(void* ws, int M, int d, int F, int64_t cap, BwdWs* out)
{
    Carver c{static_cast<char*>(ws)};
    BwdWs w{};
    csc_plan(M, F, &w.csc.row_blocks, &w.csc.rows_per_block);
    const size_t capn = (size_t)(cap > 0 ? cap : 1);
    w.dpre = c.take<float>(capn);
    w.part = c.take<float>(capn * (size_t)sddmm_slices(d > 0 ? d : 1));
    w.csc.masks = c.take<unsigned long long>((size_t)w.csc.row_blocks * F);
    w.csc.start = c.take<int32_t>((size_t)w.csc.row_blocks * F);
    w.csc.colcnt = c.take<int32_t>((size_t)F);
    w.csc.colptr = c.take<int32_t>((size_t)F + 1);
    w.csc.crow = c.take<int32_t>(capn);
    w.csc.cval = c.take<uint16_t>(capn);
    w.csc.cdpre = c.take<float>(capn);
    if (out) *out = w;
    return c.used;
}

// Workspace of the union down-projection; 16-byte aligned pieces.
size_t carve_union(void* ws, int M, int F, int64_t cap, UnionWork* out)
{
    Carver c{static_cast<char*>(ws)};
    UnionWork w{};
    const size_t ng = (size_t)((M + 127) / 128);
    w.kb_stride = union_kb_stride(F);
    w.ucnt = c.take<int32_t>(ng);
    w.gbase = c.take<int64_t>(ng);
    w.kbptr = c.take<int32_t>(ng * (size_t)w.kb_stride);
    w.ulist = c.take<int32_t>(ng * (size_t)F + 64);
    w.ent = c.take<uint32_t>((size_t)(cap > 0 ? cap : 0) + 4);
    if (out) *out = w;
    return c.used;
}

twell_status check_buf(const twell_buf* b, int M, int F, int T)
{
    if (!b) return TWELL_ERR_INVALID_ARG;
    if (b->M != M || b->F != F || b->T != T || T <= 0) return TWELL_ERR_INVALID_ARG;
    if (b->n_tiles != (M + T - 1) / T || b->cap_slots < 0) return TWELL_ERR_INVALID_ARG;
    if (!b->nnz_row || !b->K_tile || !b->tile_off) return TWELL_ERR_INVALID_ARG;
    if (b->cap_slots > 0 && (!b->idx || !b->val)) return TWELL_ERR_INVALID_ARG;
    return TWELL_OK;
}

TwellView view_of(const twell_buf* b)
{
    TwellView v;
    v.M = b->M;
    v.F = b->F;
    v.T = b->T;
    v.n_tiles = b->n_tiles;
    v.cap = b->cap_slots;
    v.nnz = b->nnz_row;
    v.K = b->K_tile;
    v.off = b->tile_off;
    v.idx = b->idx;
    v.val = b->val;
    return v;
}

twell_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA; }

bool dims_ok(int M, int d, int F) { return M > 0 && d > 0 && F > 0 && d % 8 == 0 && F % 8 == 0; }

// Limits of this build's kernels.
constexpr int kUnionMaxF = 65536;  // the union kernel keeps a group's bucket starts in shared memory

}  // namespace

extern "C" {

const char* twell_status_string(int status)
{
    switch (status) {
        case TWELL_OK: return "ok";
        case TWELL_ERR_INVALID_ARG: return "invalid argument";
        case TWELL_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case TWELL_ERR_WORKSPACE: return "workspace too small";
        case TWELL_ERR_CAPACITY: return "TwELL capacity exceeded";
        case TWELL_ERR_TIMEOUT: return "bounded device wait expired";
        case TWELL_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int64_t twell_buf_slots_bound(int M, int F, int T)
{
    if (M <= 0 || F <= 0 || T <= 0) return -1;
    return (int64_t)M * (int64_t)F;
}

size_t twell_workspace_bytes(int op, int M, int d, int F, int T, int64_t cap_slots)
{
    (void)T;
    if (M <= 0 || F <= 0) return 0;
    if (op == TWELL_OP_FFN_BWD && d <= 0) return 0;
    switch (op) {
        case TWELL_OP_FFN_FWD: return carve_fwd(nullptr, false, M, F, cap_slots, nullptr);
        case TWELL_OP_GATED_FWD: return carve_fwd(nullptr, true, M, F, cap_slots, nullptr);
        case TWELL_OP_FFN_BWD: return carve_bwd(nullptr, M, d, F, cap_slots, nullptr);
        case TWELL_OP_HYBRID_FWD: return carve_fwd(nullptr, false, M, F, cap_slots, nullptr, true);
        default: return 0;
    }
}

// Staging capacities per (row, 256-column block) the ReLU epilogue is built
// for, largest first.
constexpr int kStageCaps[] = {256, 64, 32};

// The largest staging capacity a ReLU-forward workspace of ws_bytes allows, or 0.
static int relu_stage_cap(int M, int F, int64_t cap, size_t ws_bytes)
{
    for (int S : kStageCaps)
        if (carve_fwd(nullptr, false, M, F, cap, nullptr, false, S) <= ws_bytes) return S;
    return 0;
}

size_t twell_fwd_workspace_bytes(int M, int d, int F, int T, int64_t cap_slots, int stage_cap)
{
    (void)d;
    (void)T;
    bool ok = false;
    for (int S : kStageCaps) ok = ok || S == stage_cap;
    if (M <= 0 || F <= 0 || !ok) return 0;
    return carve_fwd(nullptr, false, M, F, cap_slots, nullptr, false, stage_cap);
}

int twell_device_sm_count(void) { return sm_count_current(); }

twell_status twell_pack(const uint16_t* h, int M, int F, int ldh, int T, const twell_buf* out, int32_t* status,
                        void* stream)
{
    if (!h || !status || M <= 0 || F <= 0 || F % 8 != 0 || ldh < F || ldh % 8 != 0 || !aligned16(h))
        return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(out, M, F, T);
    if (st != TWELL_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const TwellView tw = view_of(out);
    cudaError_t e = launch_count_dense(h, ldh, tw, status, s);
    if (e == cudaSuccess) e = launch_tile_layout(tw, status, s);
    if (e == cudaSuccess) e = launch_fill_dense(h, ldh, tw, status, s);
    return cuda_status(e);
}

twell_status twell_spmm_down(const twell_buf* h, const uint16_t* W_down, int d, uint16_t* y, int32_t* status,
                             void* stream)
{
    if (!h || !W_down || !y || !status || d <= 0 || d % 8 != 0 || !aligned16(W_down) || !aligned16(y))
        return TWELL_ERR_INVALID_ARG;
    if (h->M <= 0 || h->F <= 0) return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(h, h->M, h->F, h->T);
    if (st != TWELL_OK) return st;
    const TwellView tw = view_of(h);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    timer_begin(TWELL_SITE_SPMM_DOWN, s);
    const cudaError_t e = launch_spmm_rows(tw, nullptr, W_down, d, y, status, s);
    timer_end(TWELL_SITE_SPMM_DOWN, s);
    return cuda_status(e);
}

size_t twell_spmm_down_tc_workspace_bytes(int M, int F, int64_t cap_slots)
{
    if (M <= 0 || F <= 0 || F % 8 != 0 || F > kUnionMaxF || cap_slots < 0) return 0;
    return carve_union(nullptr, M, F, cap_slots, nullptr);
}

twell_status twell_spmm_down_tc(const twell_buf* h, const uint16_t* W_down, int d, uint16_t* y, void* ws,
                                size_t ws_bytes, int32_t* status, void* stream)
{
    if (!h || !W_down || !y || !status || d <= 0 || d % 8 != 0 || !aligned16(W_down) || !aligned16(y))
        return TWELL_ERR_INVALID_ARG;
    if (h->M <= 0 || h->F <= 0 || h->F % 8 != 0) return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(h, h->M, h->F, h->T);
    if (st != TWELL_OK) return st;
    if (h->F > kUnionMaxF) return TWELL_ERR_UNSUPPORTED;
    {
        int dev = 0, optin = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return TWELL_ERR_CUDA;
        if (union_smem_bytes(h->F) > (size_t)optin) return TWELL_ERR_UNSUPPORTED;
    }
    if (!ws) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;
    if (ws_bytes < carve_union(nullptr, h->M, h->F, h->cap_slots, nullptr)) return TWELL_ERR_WORKSPACE;
    UnionWork w;
    carve_union(ws, h->M, h->F, h->cap_slots, &w);
    const TwellView tw = view_of(h);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    timer_begin(TWELL_SITE_SPMM_UNION, s);
    timer_begin(TWELL_SITE_UNION_BUILD, s);
    cudaError_t e = launch_union_build(tw, w, status, s);
    timer_end(TWELL_SITE_UNION_BUILD, s);
    if (e == cudaSuccess) e = launch_spmm_union(tw, W_down, d, w, y, status, s);
    timer_end(TWELL_SITE_SPMM_UNION, s);
    return cuda_status(e);
}

namespace {

// The up-projection and TwELL packing. For gated decode batches the whole tail
// after the gate GEMM runs as one launch, which then also computes
// y = h W_down when W_down and y are given (*fused_down = true).
twell_status up_pack_impl(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate, const float* b, int M,
                          int d, int F, int T, const twell_buf* h_out, void* ws, size_t ws_bytes, int32_t* status,
                          void* stream, const uint16_t* W_down, uint16_t* y, bool* fused_down)
{
    *fused_down = false;
    if (!x || !W_up || !b || !status || !dims_ok(M, d, F)) return TWELL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_up) || (W_gate && !aligned16(W_gate))) return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(h_out, M, F, T);
    if (st != TWELL_OK) return st;
    const bool gated = W_gate != nullptr;
    // ReLU: the epilogue staging holds as many entries per (row, 256-column
    // block) as the workspace allows (the "predicted N_nz" capacity); gated:
    // full blocks
    const int stage_cap = gated ? kReluBN : relu_stage_cap(M, F, h_out->cap_slots, ws_bytes);
    if (!ws || stage_cap == 0) return TWELL_ERR_WORKSPACE;
    const size_t need = carve_fwd(nullptr, gated, M, F, h_out->cap_slots, nullptr, false, stage_cap);
    if (ws_bytes < need) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;
    const int sms = sm_count_current();
    if (sms <= 0) return TWELL_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const TwellView tw = view_of(h_out);
    FwdWs w;
    carve_fwd(ws, gated, M, F, h_out->cap_slots, &w, false, stage_cap);
    const bool tail = gated && decode_tail_ok(M, (F + kGateBM - 1) / kGateBM, tw.n_tiles);
    // the decode tail derives nnz from the staged counts; the other paths count into it
    cudaError_t e = tail ? cudaSuccess : cudaMemsetAsync(tw.nnz, 0, sizeof(int32_t) * (size_t)M, s);
    GemmArgs ga{};
    ga.K = d;
    ga.bias = b;
    ga.stage_cnt = w.stage_cnt;
    ga.nnz = tw.nnz;
    ga.status = status;
    if (!gated) {
        ga.rowsA = M;
        ga.rowsB = F;
        ga.stage = w.stage;
        ga.stage_cap = stage_cap;
        ga.NB = (F + kReluBN - 1) / kReluBN;
        timer_begin(TWELL_SITE_UP_GEMM, s);
        if (e == cudaSuccess) e = launch_gemm(GEMM_TWELL_RELU, x, W_up, ga, sms, s);
        timer_end(TWELL_SITE_UP_GEMM, s);
        if (small_fill_ok(M, ga.NB)) {
            if (e == cudaSuccess)
                e = launch_layout_fill_small_relu(w.stage, w.stage_cnt, ga.NB, kReluBN, stage_cap, tw, status, s);
        } else if (fused_fill_ok(tw.n_tiles)) {
            if (e == cudaSuccess)
                e = launch_layout_fill_relu(w.stage, w.stage_cnt, ga.NB, kReluBN, stage_cap, tw, sms, status, s);
        } else {
            if (e == cudaSuccess) e = launch_tile_layout(tw, status, s);
            if (e == cudaSuccess)
                e = launch_fill_staged_relu(w.stage, w.stage_cnt, ga.NB, kReluBN, stage_cap, tw, nullptr, status, s);
        }
    } else {
        ga.rowsA = F;
        ga.rowsB = M;
        ga.gstage = w.gstage;
        ga.NB = (F + kGateBM - 1) / kGateBM;
        if (tail) {
            ga.nnz = nullptr;
            ga.zero_word = w.counter;
            // the tail gathers the active units' W_up (and W_down) rows next
            ga.pf0 = W_up;
            ga.pf1 = W_down ? W_down : W_up;
            ga.pf_row_bytes = 2 * d;
        }
        timer_begin(TWELL_SITE_UP_GEMM, s);
        if (e == cudaSuccess) e = launch_gemm(GEMM_GATE_SWAP, W_gate, x, ga, sms, s);
        timer_end(TWELL_SITE_UP_GEMM, s);
        if (tail) {
            const bool down = W_down && y;
            timer_begin(TWELL_SITE_DECODE_TAIL, s);
            if (e == cudaSuccess)
                e = launch_decode_tail(w.gstage, w.stage_cnt, ga.NB, kGateBM, x, W_up, W_down, d, tw,
                                       down ? y : nullptr, w.counter, status, s);
            timer_end(TWELL_SITE_DECODE_TAIL, s);
            *fused_down = down;
            return cuda_status(e);
        }
        if (small_fill_ok(M, ga.NB)) {
            if (e == cudaSuccess)
                e = launch_layout_fill_small_gate(w.gstage, w.stage_cnt, ga.NB, kGateBM, tw, w.gval, status, s);
        } else {
            if (e == cudaSuccess) e = launch_tile_layout(tw, status, s);
            if (e == cudaSuccess)
                e = launch_fill_staged_gate(w.gstage, w.stage_cnt, ga.NB, kGateBM, tw, w.gval, status, s);
        }
        if (e == cudaSuccess) e = launch_gated_up(tw, x, W_up, d, w.gval, status, s);
    }
    return cuda_status(e);
}

}  // namespace

twell_status twell_up_pack(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate, const float* b, int M,
                           int d, int F, int T, const twell_buf* h_out, void* ws, size_t ws_bytes, int32_t* status,
                           void* stream)
{
    bool fused = false;
    return up_pack_impl(x, W_up, W_gate, b, M, d, F, T, h_out, ws, ws_bytes, status, stream, nullptr, nullptr,
                        &fused);
}

twell_status twell_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate, const float* b,
                           const uint16_t* W_down, int M, int d, int F, int T, const twell_buf* h_out, uint16_t* y,
                           void* ws, size_t ws_bytes, int32_t* status, void* stream)
{
    if (!W_down || !y || !aligned16(W_down) || !aligned16(y)) return TWELL_ERR_INVALID_ARG;
    bool fused = false;
    twell_status st =
        up_pack_impl(x, W_up, W_gate, b, M, d, F, T, h_out, ws, ws_bytes, status, stream, W_down, y, &fused);
    if (st != TWELL_OK || fused) return st;
    const TwellView tw = view_of(h_out);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    timer_begin(TWELL_SITE_SPMM_DOWN, s);
    const cudaError_t e = launch_spmm_rows(tw, nullptr, W_down, d, y, status, s);
    timer_end(TWELL_SITE_SPMM_DOWN, s);
    return cuda_status(e);
}

// ----------------------------------------------------------------- hybrid --

namespace {

bool overflow_ok(const twell_overflow* ov, int F)
{
    if (!ov || ov->C < 0 || ov->cap_rows < 0 || !ov->n_rows) return false;
    if (ov->cap_rows > 0 && (!ov->rows || !ov->dense || !aligned16(ov->dense))) return false;
    (void)F;
    return true;
}

}  // namespace

twell_status twell_hybrid_up_pack(const uint16_t* x, const uint16_t* W_up, const float* b, int M, int d, int F,
                                  int T, const twell_buf* h_out, const twell_overflow* ov, void* ws,
                                  size_t ws_bytes, int32_t* status, void* stream)
{
    if (!x || !W_up || !b || !status || !dims_ok(M, d, F) || !overflow_ok(ov, F)) return TWELL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_up)) return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(h_out, M, F, T);
    if (st != TWELL_OK) return st;
    const size_t need = carve_fwd(nullptr, false, M, F, h_out->cap_slots, nullptr, true);
    if (!ws || ws_bytes < need) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;
    const int sms = sm_count_current();
    if (sms <= 0) return TWELL_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const TwellView tw = view_of(h_out);
    FwdWs w;
    carve_fwd(ws, false, M, F, h_out->cap_slots, &w, true);
    cudaError_t e = cudaMemsetAsync(tw.nnz, 0, sizeof(int32_t) * (size_t)M, s);
    GemmArgs ga{};
    ga.K = d;
    ga.bias = b;
    ga.stage_cnt = w.stage_cnt;
    ga.nnz = tw.nnz;
    ga.status = status;
    ga.rowsA = M;
    ga.rowsB = F;
    ga.stage = w.stage;
    ga.stage_cap = kReluBN;  // overflow rows can be dense: full blocks
    ga.NB = (F + kReluBN - 1) / kReluBN;
    timer_begin(TWELL_SITE_UP_GEMM, s);
    if (e == cudaSuccess) e = launch_gemm(GEMM_TWELL_RELU, x, W_up, ga, sms, s);
    timer_end(TWELL_SITE_UP_GEMM, s);
    if (e == cudaSuccess)
        e = launch_overflow_rows(tw, ov->C, ov->cap_rows, w.ov_pos, ov->rows, ov->n_rows, status, s);
    if (e == cudaSuccess) e = launch_tile_layout(tw, status, s);
    if (e == cudaSuccess)
        e = launch_fill_staged_relu(w.stage, w.stage_cnt, ga.NB, kReluBN, kReluBN, tw, w.ov_pos, status, s);
    if (e == cudaSuccess)
        e = launch_overflow_dense(w.stage, w.stage_cnt, ga.NB, kReluBN, F, ov->rows, ov->n_rows, ov->cap_rows,
                                  ov->dense, status, s);
    return cuda_status(e);
}

twell_status twell_hybrid_spmm_down(const twell_buf* h, const twell_overflow* ov, const uint16_t* W_down,
                                    const uint16_t* W_downT, int d, uint16_t* y, int32_t* status, void* stream)
{
    if (!h || !W_downT || !aligned16(W_downT) || !overflow_ok(ov, h->F)) return TWELL_ERR_INVALID_ARG;
    twell_status st = twell_spmm_down(h, W_down, d, y, status, stream);
    if (st != TWELL_OK || ov->cap_rows == 0) return st;
    const int sms = sm_count_current();
    if (sms <= 0) return TWELL_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmArgs g{};
    g.rowsA = ov->cap_rows;  // upper bound; the kernel reads the actual count
    g.rowsA_dev = ov->n_rows;
    g.row_map = ov->rows;
    g.rowsB = d;
    g.K = h->F;
    g.bias = nullptr;
    g.relu = 0;
    g.out = y;
    g.ldo = d;
    g.status = status;
    timer_begin(TWELL_SITE_OVERFLOW_GEMM, s);
    const cudaError_t e = launch_gemm(GEMM_DENSE, ov->dense, W_downT, g, sms, s);
    timer_end(TWELL_SITE_OVERFLOW_GEMM, s);
    return cuda_status(e);
}

twell_status twell_hybrid_ffn_fwd(const uint16_t* x, const uint16_t* W_up, const float* b, const uint16_t* W_down,
                                  const uint16_t* W_downT, int M, int d, int F, int T, const twell_buf* h_out,
                                  const twell_overflow* ov, uint16_t* y, void* ws, size_t ws_bytes,
                                  int32_t* status, void* stream)
{
    if (!W_down || !W_downT || !y) return TWELL_ERR_INVALID_ARG;
    twell_status st = twell_hybrid_up_pack(x, W_up, b, M, d, F, T, h_out, ov, ws, ws_bytes, status, stream);
    if (st != TWELL_OK) return st;
    return twell_hybrid_spmm_down(h_out, ov, W_down, W_downT, d, y, status, stream);
}

twell_status twell_ffn_bwd(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_down, const twell_buf* h,
                           const uint16_t* dy, int d, float l1_coef, uint16_t* dx, float* dW_up, float* dW_down,
                           float* db, void* ws, size_t ws_bytes, int32_t* status, void* stream)
{
    if (!x || !W_up || !W_down || !h || !dy || !dx || !dW_up || !dW_down || !db || !status)
        return TWELL_ERR_INVALID_ARG;
    const int M = h->M, F = h->F;
    if (!dims_ok(M, d, F)) return TWELL_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(dy) || !aligned16(dx) ||
        !aligned16(dW_up) || !aligned16(dW_down))
        return TWELL_ERR_INVALID_ARG;
    twell_status st = check_buf(h, M, F, h->T);
    if (st != TWELL_OK) return st;
    if (h->cap_slots >= (int64_t)INT32_MAX) return TWELL_ERR_UNSUPPORTED;
    const size_t need = carve_bwd(nullptr, M, d, F, h->cap_slots, nullptr);
    if (!ws || ws_bytes < need) return TWELL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return TWELL_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const TwellView tw = view_of(h);
    BwdWs w;
    carve_bwd(ws, M, d, F, h->cap_slots, &w);
    // The column lists' first kernels read only the TwELL indices: they run on
    // a side stream under the SDDMM (fork and join by events, which stream
    // capture also records); without a side stream they run first on s.
    SideStream* side = side_stream(s);
    cudaError_t e = cudaSuccess;
    if (side) {
        e = cudaEventRecord(side->fork, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
        timer_begin(TWELL_SITE_CSC, side->s);
        if (e == cudaSuccess) e = launch_csc_lists(tw, w.csc, status, side->s);
        timer_end(TWELL_SITE_CSC, side->s);
        if (e == cudaSuccess) e = cudaEventRecord(side->join, side->s);
    } else {
        timer_begin(TWELL_SITE_CSC, s);
        e = launch_csc_lists(tw, w.csc, status, s);
        timer_end(TWELL_SITE_CSC, s);
    }
    timer_begin(TWELL_SITE_SDDMM, s);
    if (e == cudaSuccess) e = launch_sddmm_slices(tw, dy, W_down, d, w.part, status, s);
    // the column lists' positions are needed from here on
    if (e == cudaSuccess && side) e = cudaStreamWaitEvent(s, side->join, 0);
    if (e == cudaSuccess) e = launch_sddmm_combine_scatter(tw, d, w.part, l1_coef, w.dpre, w.csc, status, s);
    timer_end(TWELL_SITE_SDDMM, s);
    timer_begin(TWELL_SITE_DX, s);
    if (e == cudaSuccess) e = launch_spmm_rows(tw, w.dpre, W_up, d, dx, status, s);
    timer_end(TWELL_SITE_DX, s);
    timer_begin(TWELL_SITE_WGRAD, s);
    if (e == cudaSuccess) e = launch_wgrad(tw, w.csc, w.dpre, x, dy, d, dW_up, dW_down, db, status, s);
    timer_end(TWELL_SITE_WGRAD, s);
    return cuda_status(e);
}

twell_status twell_set_kernel_timer(int site, void* ev_begin, void* ev_end)
{
    if (site < TWELL_SITE_NONE || site > TWELL_SITE_UNION_BUILD) return TWELL_ERR_INVALID_ARG;
    g_timer.site = (ev_begin && ev_end) ? site : TWELL_SITE_NONE;
    g_timer.begin = static_cast<cudaEvent_t>(ev_begin);
    g_timer.end = static_cast<cudaEvent_t>(ev_end);
    return TWELL_OK;
}

int64_t twell_kernel_launches(void) { return (int64_t)g_kernel_launches.load(std::memory_order_relaxed); }

twell_status twell_wait_selftest(int which, int32_t* scratch, int32_t* status, void* stream)
{
    if ((which != 0 && which != 1) || !scratch || !status) return TWELL_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = launch_wait_selftest(which, scratch, status, s);
    return cuda_status(e);
}

twell_status twell_check(const int32_t* status, void* stream, int32_t* host_status)
{
    if (!status || !host_status) return TWELL_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return TWELL_ERR_CUDA;
    if (cudaMemcpy(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TWELL_ERR_CUDA;
    return TWELL_OK;
}

}  // extern "C"
