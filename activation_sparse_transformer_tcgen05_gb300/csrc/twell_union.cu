// twell_union.cu — the down-projection y = h W_down on the tensor cores, over
// the union of a token group's active units.
//
// The inference kernel of "Sparser, Faster, Lighter Transformer Language
// Models" (Resumo Técnico §2, "Kernels de Inferência") visits only the active
// hidden units of each token and keeps the tensor cores busy. On this GPU the
// row-by-row gather of k_spmm_rows runs on the CUDA cores; this variant feeds
// tcgen05 instead. For a group of G = 128 consecutive tokens let U be the
// ascending union of their active units. Then
//     y[group, :] = h[group, U] · W_down[U, :],
// a GEMM with K = |U| whose A operand (128 x |U|, mostly zeros) is built in
// shared memory from the TwELL and whose B operand is the |U| gathered rows of
// W_down. It does |U| / F of the dense layer's MMA work and moves |U| rows of
// W_down per group, so it pays where the union is well below F (high sparsity
// with a small group) and where rows are too dense for the row gather
// (low sparsity, where U is all of F and this is a dense GEMM).
//
//   k_union_build   one block of 1024 threads per group: the union bitmap, its
//                   ascending list ulist[g][0, |U|), and the group's entries
//                   bucketed by 64-deep k-block of U: ent = bf16 | (pos & 63)
//                   << 16 | row-in-group << 22, with kbptr[g][kb] the start of
//                   bucket kb (relative to the group's first TwELL slot,
//                   gbase[g]). A warp walks one row, four 32-entry chunks per
//                   batch of loads.
//   k_spmm_union    one CTA per (BN-column block of d, group), 416 threads:
//     warps 4-11    loaders: per k-block, cp.async of the 64 gathered W_down
//                   row pieces (B ring, MN-major: d is the contiguous axis,
//                   128-byte swizzle) and, EA k-blocks ahead, of a bucket;
//                   completion is signalled on the slot barriers by the
//                   copies themselves (cp.async.mbarrier.arrive.noinc). Waiting
//                   for copy groups instead and arriving plainly was slower:
//                   it ties the loader to copies issued a few k-blocks back.
//     warps 0-3     builders, then epilogue: per k-block, once its bucket has
//                   landed (its W rows may still be in flight), zero the A
//                   slot (token row per thread, K-major, 128-byte swizzle),
//                   scatter the bucket into it, fence the generic-proxy writes
//                   for the tensor cores and arrive on the slot's full
//                   barrier. After the loop each thread reads its accumulator
//                   row from TMEM and writes bf16 y.
//     warp 12       TMEM owner and MMA issuer (M = 128 tokens, N = BN, K = 16):
//                   per k-block it waits for the A tile and for the landed W
//                   rows, and fences the latter for the tensor cores.
// Measured limit: the loaders' cp.async gathers. Issuing a k-block's 32 KB
// takes ~0.6 us per SM whatever the ring depths (about 53 GB/s per SM), where
// the row gather of k_spmm_rows, with plain loads from many warps, reaches
// ~90 GB/s per SM; eight loader warps instead of four gave 18 % at 99 %
// sparsity.
// Every wait is bounded (1 s); on expiry the kernel records TWELL_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "launch.h"

namespace twell {
namespace {

constexpr int UG = 128;        // tokens per group (MMA M)
constexpr int UBK = 64;        // units per k-block (one 128-byte swizzle row of bf16)
constexpr int kUnionThreads = 1024;
constexpr int kLoaders = 256;                // loader threads (warps 4 .. 4 + kLoaders / 32 - 1)
constexpr int kMmaWarp = 4 + kLoaders / 32;  // TMEM owner and MMA issuer
constexpr int kUnionGemmThreads = 32 * (kMmaWarp + 1);
constexpr int ENT_WORDS = 1024;  // entry words staged per k-block; the rest is read from global

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Orders the generic-proxy shared-memory writes this thread made, or has seen
// complete through a barrier, before its later async-proxy (tensor core) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// First TwELL slot of row r.
__device__ __forceinline__ int64_t row_base(const TwellView& tw, int r)
{
    const int t = r / tw.T;
    return tw.off[t] + (int64_t)(r - t * tw.T) * tw.K[t];
}

// Block-wide exclusive scan of one int per thread (kUnionThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kUnionThreads / 32; ++w) {
        const int s = warp_sums[w];
        before += w < warp ? s : 0;
        all += s;
    }
    __syncthreads();  // warp_sums may be reused by the caller
    *total = all;
    return before + incl - v;
}

// Calls fn(k, j, valid) for every entry k of row r, 32 at a time with the whole
// warp (lanes past the row's end get valid = false), after loading four such
// chunks at once so that their latencies overlap.
template <typename Fn>
__device__ __forceinline__ void for_row_entries(const TwellView& tw, int r, int64_t base, int lane, Fn fn)
{
    const int n = min(tw.nnz[r], tw.K[r / tw.T]);  // a row never holds more than its tile's width
    for (int k0 = 0; k0 < n; k0 += 128) {
        int jq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = k0 + 32 * q + lane;
            jq[q] = k < n ? tw.idx[base + k] : -1;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (k0 + 32 * q >= n) break;  // uniform over the warp
            fn(k0 + 32 * q + lane, jq[q], (unsigned)jq[q] < (unsigned)tw.F);
        }
    }
}

__global__ void __launch_bounds__(kUnionThreads) k_union_build(TwellView tw, int32_t* __restrict__ ucnt,
                                                                int32_t* __restrict__ ulist,
                                                                int32_t* __restrict__ kbptr, int kb_stride,
                                                                int64_t* __restrict__ gbase,
                                                                uint32_t* __restrict__ ent, const int32_t* status)
{
    extern __shared__ uint32_t us[];
    const int nw = (tw.F + 31) >> 5;
    uint32_t* bits = us;                                          // [nw]
    int* pre = reinterpret_cast<int*>(us + nw);                   // [nw]
    int* kbc = pre + nw;                                          // [kb_stride]
    __shared__ int warp_sums[kUnionThreads / 32];
    if (has_error(status)) return;  // uniform over the block

    const int g = blockIdx.x;
    const int r0 = g * UG, r1 = min(tw.M, r0 + UG);
    const int64_t gb = row_base(tw, r0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int w = threadIdx.x; w < nw; w += kUnionThreads) bits[w] = 0u;
    for (int k = threadIdx.x; k < kb_stride; k += kUnionThreads) kbc[k] = 0;
    __syncthreads();

    // the group's active units (lanes that hit the same word OR together first)
    for (int r = r0 + warp; r < r1; r += kUnionThreads / 32) {
        for_row_entries(tw, r, row_base(tw, r), lane, [&](int, int j, bool ok) {
            const int key = ok ? j >> 5 : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, key);
            const uint32_t m = __reduce_or_sync(peers, ok ? 1u << (j & 31) : 0u);
            if (ok && (peers & lanemask_lt()) == 0u) atomicOr(&bits[key], m);
        });
    }
    __syncthreads();

    // prefix of the bitmap: pre[w] = set bits in words before w
    const int per = (nw + kUnionThreads - 1) / kUnionThreads;
    const int w0 = min(nw, threadIdx.x * per), w1 = min(nw, w0 + per);
    int mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(bits[w]);
    int U = 0;
    int run = block_exclusive_scan(mine, warp_sums, &U);
    for (int w = w0; w < w1; ++w) {
        pre[w] = run;
        run += __popc(bits[w]);
    }
    __syncthreads();

    // ascending list of U
    int32_t* ul = ulist + (size_t)g * tw.F;
    for (int w = threadIdx.x; w < nw; w += kUnionThreads) {
        uint32_t b = bits[w];
        int p = pre[w];
        while (b) {
            ul[p++] = (w << 5) + __ffs(b) - 1;
            b &= b - 1;
        }
    }
    if (threadIdx.x == 0) {
        ucnt[g] = U;
        gbase[g] = gb;
    }

    // bucket sizes per k-block of U (a row's entries are ascending, so the
    // lanes of a warp mostly share a bucket: one atomic per bucket and warp)
    for (int r = r0 + warp; r < r1; r += kUnionThreads / 32) {
        for_row_entries(tw, r, row_base(tw, r), lane, [&](int, int j, bool ok) {
            const int key = ok ? (pre[j >> 5] + __popc(bits[j >> 5] & ((1u << (j & 31)) - 1u))) >> 6 : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, key);
            if (ok && (peers & lanemask_lt()) == 0u) atomicAdd(&kbc[key], __popc(peers));
        });
    }
    __syncthreads();
    const int nkb = (U + UBK - 1) / UBK;
    const int kper = (nkb + 1 + kUnionThreads - 1) / kUnionThreads;
    const int k0 = min(nkb + 1, threadIdx.x * kper), k1 = min(nkb + 1, k0 + kper);
    int kmine = 0;
    for (int k = k0; k < k1; ++k) kmine += k < nkb ? kbc[k] : 0;
    int tot = 0;
    int krun = block_exclusive_scan(kmine, warp_sums, &tot);
    for (int k = k0; k < k1; ++k) {
        const int c = k < nkb ? kbc[k] : 0;
        kbptr[(size_t)g * kb_stride + k] = krun;
        kbc[k] = krun;  // becomes the bucket's fill cursor
        krun += c;
    }
    __syncthreads();

    // entries into their buckets (order inside a bucket is free: the A tile
    // built from it is the same)
    for (int r = r0 + warp; r < r1; r += kUnionThreads / 32) {
        const int64_t base = row_base(tw, r);
        for_row_entries(tw, r, base, lane, [&](int k, int j, bool ok) {
            const int pos = ok ? pre[j >> 5] + __popc(bits[j >> 5] & ((1u << (j & 31)) - 1u)) : 0;
            const int key = ok ? pos >> 6 : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, key);
            const int leader = __ffs(peers) - 1;
            int at = 0;
            if (ok && lane == leader) at = atomicAdd(&kbc[key], __popc(peers));
            at = __shfl_sync(0xffffffffu, at, leader) + __popc(peers & lanemask_lt());
            if (ok)
                ent[gb + at] = (uint32_t)tw.val[base + k] | ((uint32_t)(pos & 63) << 16) |
                               ((uint32_t)(r - r0) << 22);
        });
    }
}

// B ring: NBS slots of gathered W rows; E ring: NE slots of entry buckets,
// fetched EA k-blocks ahead of B; A ring: NA slots of the densified h tile;
// per loader warp a ring of unit ids.
template <int BN, int NBS, int NE, int EA, int NA>
struct ULayout {
    static constexpr int A_BYTES = UG * UBK * 2;          // 16 KB
    static constexpr int B_BYTES = BN * UBK * 2;          // 64 rows x BN columns
    static constexpr int E_BYTES = ENT_WORDS * 4;
    static constexpr int E_OFF = NBS * B_BYTES;
    static constexpr int A_OFF = E_OFF + NE * E_BYTES;
    static constexpr int BAR_OFF = A_OFF + NA * A_BYTES;
    static constexpr int NBARS = 2 * NBS + 2 * NE + 2 * NA + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int UL_AHEAD = NBS;                   // k-blocks of unit ids fetched ahead
    static constexpr int UL_RING = UL_AHEAD + 1;
    static constexpr int UL_OFF = (MISC_OFF + 32 + 15) & ~15;
    static constexpr int KB_OFF = UL_OFF + (kLoaders / 32) * UL_RING * UBK * 4;
    static_assert(B_BYTES % 1024 == 0 && A_OFF % 1024 == 0 && A_BYTES % 1024 == 0,
                  "operand tiles must stay 1024-byte aligned");
    static_assert(EA >= 1 && EA < NE, "a bucket slot is refilled only after its A tile was built");
};

// Arrive once on `bar` when every cp.async this thread issued so far has
// completed; the arrival counts toward the barrier's expected count.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int BN, int NBS, int NE, int EA, int NA>
__global__ void __launch_bounds__(kUnionGemmThreads, 1)
    k_spmm_union(TwellView tw, const uint16_t* __restrict__ W, int d, const int32_t* __restrict__ ucnt,
                 const int32_t* __restrict__ ulist, const int32_t* __restrict__ kbptr, int kb_stride,
                 const int64_t* __restrict__ gbase, const uint32_t* __restrict__ ent, uint16_t* __restrict__ y,
                 int32_t* status)
{
    using L = ULayout<BN, NBS, NE, EA, NA>;
    // bf16 A (K-major) and B (MN-major: bit 16), fp32 D, M = 128, N = BN
    constexpr uint32_t IDESC = idesc_bf16_f32(UG, BN) | kIdescBMn;
    constexpr int CPU = BN / 8;           // 16-byte pieces per gathered row
    constexpr int UPW = 32 / CPU;         // rows per warp instruction
    constexpr int NCP = UBK * CPU / kLoaders;  // pieces per loader thread per k-block
    constexpr int NLW = kLoaders / 32;         // loader warps
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* landed = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);  // B slot copies done
    uint64_t* emptyB = landed + NBS;                                     // B slot read by the MMAs
    uint64_t* elanded = emptyB + NBS;                                    // bucket copies done
    uint64_t* eempty = elanded + NE;                                     // bucket scattered into A
    uint64_t* fullA = eempty + NE;                                       // A tile built
    uint64_t* emptyA = fullA + NA;                                       // A tile read by the MMAs
    uint64_t* tfull = emptyA + NA;
    uint64_t* mma_done = tfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* skip = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* pstop = reinterpret_cast<volatile int*>(tmem_slot + 3);
    volatile int* epi_fail = reinterpret_cast<volatile int*>(tmem_slot + 4);
    int* s_kb = reinterpret_cast<int*>(smem + L::KB_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;
    const int n0 = blockIdx.x * BN;
    if (threadIdx.x == 0) {
        *skip = has_error(status) ? 1 : 0;
        *abort_flag = 0;
        *pstop = 0;
        *epi_fail = 0;
        for (int s = 0; s < NBS; ++s) {
            mbar_init(&landed[s], kLoaders);
            mbar_init(&emptyB[s], 1);
        }
        for (int s = 0; s < NE; ++s) {
            mbar_init(&elanded[s], kLoaders);
            mbar_init(&eempty[s], 128);
        }
        for (int s = 0; s < NA; ++s) {
            mbar_init(&fullA[s], 128);
            mbar_init(&emptyA[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (*skip) return;  // an earlier kernel of this call failed; uniform over the block
    // (the union lists below exist only if it did not)
    const int U = min(max(ucnt[g], 0), tw.F);
    const int nkb = (U + UBK - 1) / UBK;
    for (int k = threadIdx.x; k <= nkb; k += blockDim.x) s_kb[k] = kbptr[(size_t)g * kb_stride + k];
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t gb = gbase[g];

    if (warp >= 4 && warp < kMmaWarp) {
        // -------------------------------------------------------- loaders --
        // B piece p of this thread in a k-block: row u = (p * NLW + lw) * UPW + lane / CPU,
        // column piece lane % CPU (one warp instruction reads UPW whole row pieces).
        const int lt = threadIdx.x - 128, lw = lt >> 5;
        const int cc = lane % CPU;
        const int col = n0 + cc * 8;
        const bool col_ok = col < d;
        const int32_t* ul = ulist + (size_t)g * tw.F;
        int* ring = reinterpret_cast<int*>(smem + L::UL_OFF) + lw * L::UL_RING * UBK;  // this warp's unit ids
        for (int q = lane; q < L::UL_AHEAD * UBK; q += 32) ring[q] = q < U ? ul[q] : 0;
        __syncwarp();
        // bucket of k-block k into E slot k % NE, 16-byte pieces from the aligned start
        auto issue_bucket = [&](int k) {
            const int64_t e0 = gb + s_kb[k], e1 = gb + s_kb[k + 1];
            const int64_t a0 = e0 & ~int64_t(3);
            const int64_t npc64 = (e1 - a0 + 3) >> 2;
            const int npc = npc64 < ENT_WORDS / 4 ? (int)npc64 : ENT_WORDS / 4;
            const uint32_t se = smem_u32(smem + L::E_OFF + (k % NE) * L::E_BYTES);
            for (int p = lt; p < npc; p += kLoaders) cp_async16(se + p * 16, ent + a0 + 4 * p, 16u);
            cp_async_arrive_noinc(&elanded[k % NE]);
        };
        for (int k = 0; k < EA && k < nkb; ++k) issue_bucket(k);
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            __syncwarp();  // every lane is done with the ring slot refilled below
            // unit ids of k-block i + UL_AHEAD (ulist rows are padded by UBK ids)
            const int kn = i + L::UL_AHEAD;
            if (lane < UBK / 4 && kn < nkb)
                cp_async16(smem_u32(ring + (kn % L::UL_RING) * UBK + 4 * lane), ul + (size_t)kn * UBK + 4 * lane, 16u);
            // the bucket of k-block i + EA, once the bucket NE k-blocks before it has been used
            const int ke = i + EA;
            int stop = 0;
            if (ke < nkb) {
                if (lane == 0 && ke >= NE &&
                    !mbar_wait(&eempty[ke % NE], ((uint32_t)(ke / NE) & 1u) ^ 1u, abort_flag))
                    stop = 1;
                if (__shfl_sync(0xffffffffu, stop, 0)) {
                    ok = false;
                    break;
                }
                issue_bucket(ke);
            }
            const int bs = i % NBS;
            if (lane == 0 && !mbar_wait(&emptyB[bs], ((uint32_t)(i / NBS) & 1u) ^ 1u, abort_flag)) stop = 1;
            if (__shfl_sync(0xffffffffu, stop, 0)) {
                ok = false;
                break;
            }
            // the unit ids of k-block i (committed UL_AHEAD groups ago) have landed:
            // at most UL_AHEAD - 1 of the committed groups still pending
            cp_async_wait<L::UL_AHEAD - 1>();
            __syncwarp();
            const int* uk = ring + (i % L::UL_RING) * UBK;
            // gathered W rows, MN-major 128-byte-swizzled: row u at atom (u / 8) of its
            // 64-column block, 16-byte piece c at c ^ (u % 8)
            const uint32_t sb = smem_u32(smem + bs * L::B_BYTES);
#pragma unroll
            for (int p = 0; p < NCP; ++p) {
                const int u = (p * NLW + lw) * UPW + lane / CPU;
                const bool ok_u = i * UBK + u < U;
                const int j = ok_u ? uk[u] : 0;
                const uint32_t dst = sb + (cc >> 3) * (UBK * 128) + (u >> 3) * 1024 + (u & 7) * 128 +
                                     ((((cc & 7) ^ (u & 7))) << 4);
                const uint16_t* src = W + (size_t)j * d + (col_ok ? col : 0);
                cp_async16(dst, src, (ok_u && col_ok) ? 16u : 0u);
            }
            cp_async_commit();
            cp_async_arrive_noinc(&landed[bs]);
        }
        cp_async_wait_all();
        if (!ok) {
            set_error(status, TWELL_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp < 4) {
        // ------------------------------------------------------- builders --
        const int t = threadIdx.x;  // token row of the group
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            const int as = j % NA, es = j % NE;
            if (t == 0 && (!mbar_wait(&elanded[es], (uint32_t)(j / NE) & 1u, abort_flag) ||
                           !mbar_wait(&emptyA[as], ((uint32_t)(j / NA) & 1u) ^ 1u, abort_flag)))
                *pstop = 1;
            __syncwarp();
            named_bar_sync(1, 128);
            if (*pstop) {
                ok = false;
                break;
            }
            uint8_t* sa = smem + L::A_OFF + as * L::A_BYTES;
            // zero this token row (pieces in a rotated order: no bank conflicts)
            uint8_t* arow = sa + t * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(arow + (((c + t) & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            named_bar_sync(1, 128);
            const uint32_t* se = reinterpret_cast<const uint32_t*>(smem + L::E_OFF + es * L::E_BYTES);
            const int64_t e0 = gb + s_kb[j], e1 = gb + s_kb[j + 1];
            const int64_t a0 = e0 & ~int64_t(3);
            for (int64_t e = e0 + t; e < e1; e += 128) {
                const int64_t off = e - a0;
                const uint32_t w = off < ENT_WORDS ? se[off] : ent[e];
                const int er = (int)(w >> 22), ek = (int)((w >> 16) & 63u);
                *reinterpret_cast<uint16_t*>(sa + er * 128 + ((((ek >> 3) ^ (er & 7))) << 4) + (ek & 7) * 2) =
                    (uint16_t)(w & 0xffffu);
            }
            fence_proxy_async_smem();  // this thread's A writes, before the MMAs read them
            mbar_arrive(&fullA[as]);
            mbar_arrive(&eempty[es]);
        }
        if (!ok) {
            set_error(status, TWELL_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        // --------------------------------------------------------- epilogue --
        const int row = g * UG + t;
        const bool have = nkb > 0;
        if (ok) {
            // one decision for all builder threads: the TMEM loads below are warp-collective
            if (have && !mbar_wait(tfull, 0, abort_flag)) *epi_fail = 1;
            named_bar_sync(1, 128);
            if (*epi_fail) {
                set_error(status, TWELL_ERR_TIMEOUT);
                *abort_flag = 1;
                ok = false;
            }
        }
        if (ok) {
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t v[32];
                if (have) {
                    tmem_ld32_wait(tb + ch * 32, v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                if (row < tw.M) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        const int c = n0 + ch * 32 + g8 * 8;
                        if (c < d) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[g8 * 8 + 0]), __uint_as_float(v[g8 * 8 + 1]));
                            o.y = pack_bf16x2(__uint_as_float(v[g8 * 8 + 2]), __uint_as_float(v[g8 * 8 + 3]));
                            o.z = pack_bf16x2(__uint_as_float(v[g8 * 8 + 4]), __uint_as_float(v[g8 * 8 + 5]));
                            o.w = pack_bf16x2(__uint_as_float(v[g8 * 8 + 6]), __uint_as_float(v[g8 * 8 + 7]));
                            *reinterpret_cast<uint4*>(y + (size_t)row * d + c) = o;
                        }
                    }
                }
            }
        }
    } else if (lane == 0) {
        // ------------------------------------------------------ MMA issuer --
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            const int as = j % NA, bs = j % NBS;
            if (!mbar_wait(&fullA[as], (uint32_t)(j / NA) & 1u, abort_flag) ||
                !mbar_wait(&landed[bs], (uint32_t)(j / NBS) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();  // the landed copies, before the tensor cores read them
            tc_fence_after();
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(smem + L::A_OFF + as * L::A_BYTES));
            const uint64_t bdesc = sw128_mnmajor_desc(smem_u32(smem + bs * L::B_BYTES), UBK * 128);
#pragma unroll
            for (int k = 0; k < UBK / 16; ++k)  // K = 16: 32 bytes along A's rows, two 8-row atoms of B
                umma_bf16(tmem_base, adesc + 2u * k, bdesc + (uint64_t)(128u * k), IDESC, (j | k) != 0);
            umma_commit(&emptyA[as]);
            umma_commit(&emptyB[bs]);
        }
        if (ok && nkb > 0) umma_commit(tfull);
        if (!ok) {
            set_error(status, TWELL_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        umma_commit(mma_done);  // every MMA issued above has finished once this arrives
        mbar_wait(mma_done, 0, nullptr);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, BN);
    }
}

template <int BN, int NBS, int NE, int EA, int NA>
cudaError_t run_union(const TwellView& tw, const uint16_t* W, int d, const UnionWork& w, uint16_t* y,
                      int32_t* status, cudaStream_t s)
{
    using L = ULayout<BN, NBS, NE, EA, NA>;
    const int ng = (tw.M + UG - 1) / UG;
    const size_t smem = 1024 + L::KB_OFF + (size_t)w.kb_stride * 4;
    auto kern = k_spmm_union<BN, NBS, NE, EA, NA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    count_launches(1);
    kern<<<dim3((unsigned)((d + BN - 1) / BN), (unsigned)ng), kUnionGemmThreads, smem, s>>>(
        tw, W, d, w.ucnt, w.ulist, w.kbptr, w.kb_stride, w.gbase, w.ent, y, status);
    return cudaGetLastError();
}

// Tile shapes: 128 x 256 (B ring 5 x 32 KB, bucket ring 4 x 4 KB, A ring 2 x 16 KB)
// and, for d <= 128, 128 x 128 (B ring 8 x 16 KB, bucket ring 4 x 4 KB, A ring 3 x 16 KB).
#define TWELL_UNION_WIDE 256, 5, 4, 2, 2
#define TWELL_UNION_NARROW 128, 8, 4, 2, 3
using Wide = ULayout<TWELL_UNION_WIDE>;
using Narrow = ULayout<TWELL_UNION_NARROW>;

}  // namespace

int union_kb_stride(int F) { return (F + UBK - 1) / UBK + 1; }

size_t union_smem_bytes(int F)
{
    const size_t kb = 1024 + (size_t)union_kb_stride(F) * 4;
    return (Wide::KB_OFF > Narrow::KB_OFF ? Wide::KB_OFF : Narrow::KB_OFF) + kb;
}

cudaError_t launch_union_build(const TwellView& tw, const UnionWork& w, int32_t* status, cudaStream_t s)
{
    const int ng = (tw.M + UG - 1) / UG;
    const int nw = (tw.F + 31) >> 5;
    const size_t smem = (size_t)(2 * nw + w.kb_stride) * 4;
    cudaError_t e = cudaFuncSetAttribute(k_union_build, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    count_launches(1);
    k_union_build<<<ng, kUnionThreads, smem, s>>>(tw, w.ucnt, w.ulist, w.kbptr, w.kb_stride, w.gbase, w.ent,
                                                  status);
    return cudaGetLastError();
}

cudaError_t launch_spmm_union(const TwellView& tw, const uint16_t* W, int d, const UnionWork& w, uint16_t* y,
                              int32_t* status, cudaStream_t s)
{
    if (d <= 128) return run_union<TWELL_UNION_NARROW>(tw, W, d, w, y, status, s);
    return run_union<TWELL_UNION_WIDE>(tw, W, d, w, y, status, s);
}

}  // namespace twell
