// twell_decode.cu — the gated forward's tail for decode batches.
//
// For decode batches (the method's gated inference, "Sparser, Faster, Lighter
// Transformer Language Models", Resumo Técnico §2 Metodologia: fused gated up
// and down products over the gate's active units) everything after the gate
// GEMM runs as one cooperative launch; its grid-wide barrier and the bounded
// waits' self-test live here too.
#include "sparse_common.cuh"

namespace twell {

namespace {

// ---------------------------------------------------------- decode tail --
//
// Everything of the gated forward after the gate GEMM, for decode batches
// (M <= 64), in one cooperative launch of one 512-thread block per SM. At
// these sizes each separate kernel costs a launch, a drain and a chain of
// dependent global round trips while moving well under a megabyte, so:
//   A. every block reads the staged per-(token, 128-unit block) counts and
//      computes the TwELL layout (token prefixes, nnz, tile widths, offsets)
//      in shared memory; block 0 writes nnz / K / off, and each block writes
//      the padding of its share of the tokens;
//   B. one warp per active (token, unit) entry, over all warps of the GPU:
//      u = x[t] . W_up[j], h = bf16(relu(g) * u), written to its slot;
//   C. after a grid barrier (bounded wait; on expiry the block reports
//      TWELL_ERR_TIMEOUT and leaves), y[t, 256-column group] = sum over the
//      token's entries of h * W_down[j, group], split over `split` warps whose
//      partial sums are added in warp order (deterministic), as in k_spmm_rows.
// With y == nullptr only A and B run (the TwELL without the down-projection).
constexpr int kTailWarps = 16;
constexpr int kTailMaxM = 64;
constexpr int kTailMaxSeg = 8192;  // M * NB staged segments held in shared memory

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of a cooperative launch: every block adds one to *counter
// and waits until it reaches `target`. Bounded: after kWaitLimitNs without
// getting there it returns false (in every thread of the block) instead of
// waiting on. `flag` is a shared int of the block.
__device__ __forceinline__ bool grid_barrier(int32_t* counter, int target, int* flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1);
        const uint64_t t0 = globaltimer_ns();
        int go = 1;
        while (ld_acquire_gpu(counter) < target) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                go = 0;
                break;
            }
        }
        *flag = go;
    }
    __syncthreads();
    return *flag != 0;
}

// Self-test of the bounded waits (twell_wait_selftest): a wait that nothing
// will complete runs out and reports TWELL_ERR_TIMEOUT. which = 0: an
// mbarrier nobody arrives on; which = 1: the grid barrier with a target the
// grid cannot reach.
__global__ void k_wait_selftest(int which, int32_t* counter, int32_t* status)
{
    __shared__ uint64_t bar;
    __shared__ int flag;
    if (which == 0) {
        if (threadIdx.x == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0 && !mbar_wait(&bar, 0, nullptr)) set_error(status, TWELL_ERR_TIMEOUT);
    } else {
        if (!grid_barrier(counter, (int)gridDim.x + 1, &flag) && threadIdx.x == 0)
            set_error(status, TWELL_ERR_TIMEOUT);
    }
}

__global__ void __launch_bounds__(kTailWarps * 32, 1)
    k_decode_tail(const uint2* __restrict__ gstage, const int32_t* __restrict__ stage_cnt, int NB, int BM,
                  const uint16_t* __restrict__ x, const uint16_t* __restrict__ W_up,
                  const uint16_t* __restrict__ W_down, int d, TwellView tw, uint16_t* __restrict__ y, int split,
                  int32_t* counter, int32_t* status)
{
    __shared__ union {
        int pre[kTailMaxSeg];                 // A, B: exclusive prefix of a token's staged counts
        float red[kTailWarps][256];           // C: partial sums of split tasks
    } sm;
    __shared__ int s_nnz[kTailMaxM], s_tok[kTailMaxM + 1], s_K[kTailMaxM];
    __shared__ long long s_off[kTailMaxM + 1];
    __shared__ int s_go;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int M = tw.M, nseg = M * NB;
    if (has_error(status)) return;

    // ---------------------------------------------------------------- A --
    // eight independent loads in flight per thread: at 64 tokens the staged
    // counts are 14 per thread, and one at a time they cost a round trip each
    for (int i0 = tid; i0 < nseg; i0 += 8 * kTailWarps * 32) {
        int c[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kTailWarps * 32;
            c[q] = i < nseg ? __ldcg(stage_cnt + i) : 0;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + q * kTailWarps * 32;
            if (i < nseg) sm.pre[i] = c[q];
        }
    }
    __syncthreads();
    // one warp per token, four consecutive counts per lane and round
    for (int t = warp; t < M; t += kTailWarps) {
        int* pt = sm.pre + t * NB;
        int carry = 0;
        for (int nb0 = 0; nb0 < NB; nb0 += 128) {
            const int b0 = nb0 + lane * 4;
            int c[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) c[u] = b0 + u < NB ? pt[b0 + u] : 0;
            const int sum = c[0] + c[1] + c[2] + c[3];
            const int incl = warp_incl_scan(sum, lane);
            int run = carry + incl - sum;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (b0 + u < NB) pt[b0 + u] = run;
                run += c[u];
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_nnz[t] = carry;
    }
    __syncthreads();
    // tile widths (one warp per tile), the tokens' entry prefix (warp 0 over
    // M <= 64 tokens, two per lane), then the tile offsets in order
    for (int tt = warp; tt < tw.n_tiles; tt += kTailWarps) {
        const int r0 = tt * tw.T, rows = min(tw.T, M - r0);
        int mx = 0;
        for (int i = lane; i < rows; i += 32) mx = max(mx, s_nnz[r0 + i]);
        mx = warp_max_i(mx);
        if (lane == 0) s_K[tt] = mx;
    }
    if (warp == 0) {
        const int a0 = lane < M ? s_nnz[lane] : 0;
        const int a1 = lane + 32 < M ? s_nnz[lane + 32] : 0;
        const int i0 = warp_incl_scan(a0, lane);
        const int tot0 = __shfl_sync(0xffffffffu, i0, 31);
        const int i1 = warp_incl_scan(a1, lane) + tot0;
        if (lane < M) s_tok[lane] = i0 - a0;
        if (lane + 32 < M) s_tok[lane + 32] = i1 - a1;
        if (lane == 31) s_tok[M] = i1;
    }
    __syncthreads();
    if (tid == 0) {
        long long off = 0;
        for (int tt = 0; tt < tw.n_tiles; ++tt) {
            s_off[tt] = off;
            off += (long long)min(tw.T, M - tt * tw.T) * s_K[tt];
        }
        s_off[tw.n_tiles] = off;
    }
    __syncthreads();
    const bool over = s_off[tw.n_tiles] > tw.cap;
    if (blockIdx.x == 0) {
        for (int t = tid; t < M; t += blockDim.x) tw.nnz[t] = s_nnz[t];
        for (int tt = tid; tt <= tw.n_tiles; tt += blockDim.x) {
            if (tt < tw.n_tiles) tw.K[tt] = s_K[tt];
            tw.off[tt] = s_off[tt];
        }
        if (tid == 0 && over) set_error(status, TWELL_ERR_CAPACITY);
    }
    if (over) return;  // uniform: every block computed the same layout
    for (int t = blockIdx.x + warp * gridDim.x; t < M; t += gridDim.x * kTailWarps) {
        const int tt = t / tw.T;
        const long long base = s_off[tt] + (long long)(t - tt * tw.T) * s_K[tt];
        for (int k = s_nnz[t] + lane; k < s_K[tt]; k += 32) {
            tw.idx[base + k] = -1;
            tw.val[base + k] = 0;
        }
    }

    // ---------------------------------------------------------------- B --
    const int E = s_tok[M];
    const int nwarps = gridDim.x * kTailWarps;
    for (int e = blockIdx.x * kTailWarps + warp; e < E; e += nwarps) {
        int lo = 0, hi = M;  // token: last t with s_tok[t] <= e
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tok[mid] <= e) lo = mid; else hi = mid;
        }
        const int t = lo, k = e - s_tok[t];
        const int* pre = sm.pre + t * NB;
        int a = 0, b = NB;  // staged segment: last nb with pre[nb] <= k
        while (b - a > 1) {
            const int mid = (a + b) >> 1;
            if (pre[mid] <= k) a = mid; else b = mid;
        }
        const uint2 ent = gstage[((size_t)t * NB + a) * BM + (k - pre[a])];
        const int j = (int)ent.x;
        const uint16_t* xr = x + (size_t)t * d + lane * 8;
        const uint16_t* wr = W_up + (size_t)j * d + lane * 8;
        float acc = 0.f;
        for (int c0 = 0; c0 < d; c0 += 8 * 256) {
            uint4 av[8], wv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + q * 256;
                const bool ok = c + lane * 8 < d;
                av[q] = ok ? ldg16(xr + c) : make_uint4(0, 0, 0, 0);
                wv[q] = ok ? ldg16(wr + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) acc += dot8_bf16(av[q], wv[q]);
        }
        acc = warp_sum_f(acc);
        if (lane == 0) {
            const int tt = t / tw.T;
            const long long slot = s_off[tt] + (long long)(t - tt * tw.T) * s_K[tt] + k;
            tw.idx[slot] = j;
            tw.val[slot] = f32_to_bf16_bits(fmaxf(__uint_as_float(ent.y), 0.f) * acc);
        }
    }
    if (!y) return;

    // ------------------------------------------------------ grid barrier --
    if (!grid_barrier(counter, (int)gridDim.x, &s_go)) {
        if (tid == 0) set_error(status, TWELL_ERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------------- C --
    const int G = (d + 255) >> 8;
    const long long tasks = (long long)M * G;
    const int tpb = kTailWarps / split;  // tasks per block and round
    const int sub = warp % split;
    for (long long t0 = (long long)blockIdx.x * tpb; t0 < tasks; t0 += (long long)gridDim.x * tpb) {
        const long long task = t0 + warp / split;
        const bool task_ok = task < tasks;
        const int t = task_ok ? (int)(task / G) : 0, g = task_ok ? (int)(task % G) : 0;
        const int c0 = g * 256 + lane * 8;
        const bool col_ok = task_ok && c0 < d;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        if (task_ok) {
            const int tt = t / tw.T;
            const long long base = s_off[tt] + (long long)(t - tt * tw.T) * s_K[tt];
            const int n = s_nnz[t];
            const int per = (n + split - 1) / split;
            const int kb = min(n, sub * per), ke = min(n, kb + per);
            const uint16_t* Wc = W_down + c0;
            for (int k0 = kb; k0 < ke; k0 += 32) {
                const int m = min(32, ke - k0);
                int jl = 0;
                uint32_t vb = 0;
                if (lane < m) {
                    jl = __ldcg(tw.idx + base + k0 + lane);
                    vb = __ldcg(tw.val + base + k0 + lane);
                }
                // 8 W_down rows in flight: a decode task walks its entries
                // alone, so its time is the number of dependent round trips
                int u = 0;
                for (; u + 8 <= m; u += 8) {
                    uint4 w[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int jj = __shfl_sync(0xffffffffu, jl, u + q);
                        w[q] = col_ok ? ldg16(Wc + (size_t)jj * d) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) fma8_bf16(acc, __shfl_sync(0xffffffffu, vb, u + q), w[q]);
                }
                for (; u < m; ++u) {
                    const int jj = __shfl_sync(0xffffffffu, jl, u);
                    const uint4 w = col_ok ? ldg16(Wc + (size_t)jj * d) : make_uint4(0, 0, 0, 0);
                    fma8_bf16(acc, __shfl_sync(0xffffffffu, vb, u), w);
                }
            }
        }
        if (split > 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) sm.red[warp][lane * 8 + e] = acc[e];
            __syncthreads();
            if (sub == 0) {
                for (int s2 = 1; s2 < split; ++s2) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] += sm.red[warp + s2][lane * 8 + e];
                }
            }
        }
        if (sub == 0 && col_ok) {
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(y + (size_t)t * d + c0) = o;
        }
        if (split > 1) __syncthreads();  // red is rewritten in the next round
    }
}

}  // namespace

cudaError_t launch_wait_selftest(int which, int32_t* counter, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    // one block for the mbarrier case; a small grid for the barrier (all blocks
    // resident at once, as the cooperative launch of the decode tail guarantees)
    k_wait_selftest<<<which == 0 ? 1 : 4, 64, 0, s>>>(which, counter, status);
    return cudaGetLastError();
}

int decode_tail_grid()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_tail, kTailWarps * 32, 0) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            cached[dev] = -1;
        } else {
            cached[dev] = per_sm >= 1 ? sms : -1;
        }
    }
    return cached[dev];
}

bool decode_tail_ok(int M, int NB, int n_tiles)
{
    return M <= kTailMaxM && (long long)M * NB <= kTailMaxSeg && n_tiles <= kTailMaxM && decode_tail_grid() > 0;
}

cudaError_t launch_decode_tail(const uint2* gstage, const int32_t* stage_cnt, int NB, int BM, const uint16_t* x,
                               const uint16_t* W_up, const uint16_t* W_down, int d, const TwellView& tw,
                               uint16_t* y, int32_t* counter, int32_t* status, cudaStream_t s)
{
    const int grid = decode_tail_grid();
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    // warps per down-projection task: as many as keep every warp of the grid busy
    const long long tasks = (long long)tw.M * ((d + 255) / 256);
    int split = kTailWarps;
    while (split > 1 && tasks * split > (long long)grid * kTailWarps) split >>= 1;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all blocks resident: the grid barrier can complete
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kTailWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, k_decode_tail, gstage, stage_cnt, NB, BM, x, W_up, W_down, d, tw, y, split,
                              counter, status);
}

}  // namespace twell
