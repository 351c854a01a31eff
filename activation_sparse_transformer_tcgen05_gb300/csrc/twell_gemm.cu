// twell_gemm.cu — persistent tcgen05 GEMM with a TwELL-emitting epilogue.
//
// D = A B^T with A [rowsA, K] and B [rowsB, K] bf16, both K-major, fp32
// accumulation in tensor memory. The method writes TwELL from the epilogue of
// the dense matmul that computes the activations, so that neither a separate
// conversion kernel nor synchronisation between CTAs is needed ("Sparser,
// Faster, Lighter Transformer Language Models", Resumo Técnico §2, "Formato de
// Dados TwELL"). Here each CTA compacts its own output tile independently:
//
//   GEMM_TWELL_RELU  A = x (tokens), B = W_up (hidden units). One epilogue
//                    thread owns one token row of the tile; it adds the bias,
//                    applies ReLU, rounds to bf16 and appends every nonzero as
//                    (bf16 << 16 | column within the tile) to the row's
//                    staging segment for this column block, in ascending
//                    column order. The dense hidden matrix is never written.
//   GEMM_GATE_SWAP   A = W_gate (hidden units), B = x (<= 64 tokens, the
//                    decode shapes). One thread owns one hidden unit; per token
//                    a warp ballot and popcount prefix place the active units
//                    (gate > 0) of the tile in ascending order.
//   GEMM_DENSE       plain bf16 output (optional bias and ReLU): the dense
//                    baseline layer.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0     TMA producer: 128-byte-swizzled A/B tiles into a STAGES-deep ring
//   warp 1     TMEM owner and MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31), double-buffered so the next tile's MMAs overlap
// Every wait is bounded (1 s); on expiry the kernel records TWELL_ERR_TIMEOUT,
// lets the other roles stop, drains its TMA loads and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "launch.h"

namespace twell {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kEpiThreads = 128;

// A stage holds KSUB consecutive 64-deep k-blocks (A then B for each).
template <int BN, int STAGES, int KSUB = 1>
struct Layout {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int SUB_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGE_BYTES = KSUB * SUB_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BIAS_OFF = (MISC_OFF + 16 + 15) & ~15;
    static constexpr int BIAS_BYTES = 4 * (BN > BM ? BN : BM);
    static constexpr int MASK_OFF = BIAS_OFF + BIAS_BYTES;
    static constexpr int MASK_BYTES = 64 * 4 * 4;
    static constexpr int COL_OFF = MASK_OFF + MASK_BYTES;
    static constexpr int COL_BYTES = 4 * BN * 4;  // dense epilogue: per-warp column sums
    static constexpr int TOTAL = COL_OFF + COL_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                        : (2 * BN <= 256) ? 256 : 512;
    static_assert(SUB_BYTES % 1024 == 0, "stages must stay 1024-byte aligned");
};

// Depth of the contraction: a.K, or with a.K_dev the count an earlier kernel
// wrote there, rounded up to the 64-deep k-block (the operands are zero past
// it) and at most a.K.
__device__ __forceinline__ int gemm_k(const GemmArgs& a)
{
    if (!a.K_dev) return a.K;
    const int k = *a.K_dev;
    const int kr = k <= 0 ? 0 : ((k + BK - 1) / BK) * BK;
    return kr < a.K ? kr : a.K;
}

__device__ __forceinline__ void fail(int32_t* status, volatile int* abort_flag)
{
    set_error(status, TWELL_ERR_TIMEOUT);
    *abort_flag = 1;
}

// TwELL epilogue of one accumulator row (one thread): bias, ReLU, bf16
// rounding, and the row's nonzeros of this BN-column block appended to its
// staging segment of CAP words as (bf16 << 16 | column within the block),
// ascending. CAP is a compile-time constant: a run-time segment stride made
// this epilogue slow enough to hold back the MMAs.
template <int BN, int CAP>
__device__ __forceinline__ void epi_twell_row(uint32_t tbase, int row, int rowsA, int nb, const GemmArgs& a,
                                              const float* bias_sm)
{
    const bool row_ok = row < rowsA;
    uint32_t* st = a.stage + ((size_t)(row_ok ? row : 0) * a.NB + nb) * CAP;
    int cnt = 0;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32_wait(tbase + ch * 32, v);
        // Straight-line per column (no branch): bias from 128-bit shared
        // loads, the test, the rounding, and a predicated store, so that the
        // 32 columns of a chunk overlap instead of each waiting on the last.
        const float4* b4 = reinterpret_cast<const float4*>(bias_sm + ch * 32);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const float4 bb = b4[g];
            const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = g * 4 + e;
                const float p = __uint_as_float(v[c]) + bv[e];
                const uint32_t hb = f32_to_bf16_bits(p);
                const bool act = row_ok && p > 0.f && hb != 0u;
                // no capacity test per column: a segment that overflows spills
                // into the next one (the workspace has BN - cap words of slack
                // after the last), and the call then fails with a capacity error
                if (act) st[cnt] = (hb << 16) | (uint32_t)(ch * 32 + c);
                cnt += act ? 1 : 0;
            }
        }
    }
    if (row_ok) {
        // a segment with more nonzeros than the staging holds: the call fails
        // with a capacity error; counts stay within what was staged
        if (cnt > CAP) {
            set_error(a.status, TWELL_ERR_CAPACITY);
            cnt = CAP;
        }
        a.stage_cnt[(size_t)row * a.NB + nb] = cnt;
        if (cnt) atomicAdd(&a.nnz[row], cnt);
    }
}

// Dense epilogue of one accumulator row (one thread; the 128 epilogue threads
// hold the 128 rows of the CTA's tile): bias, optional ReLU, + add_scalar,
// the mask, then bf16 or fp32 stores. With a.colsum (bf16 output) the warp's
// 32 rows are summed per column by a butterfly, the four warps' sums are
// added in warp order through s_col, and row block rt's column sums are
// written for the tile's columns.
template <int BN>
__device__ __forceinline__ void epi_dense_row(uint32_t tbase, int row, int rowsA, int nb, const GemmArgs& a,
                                              const float* bias_sm, float* s_col, int rt, int q, int et)
{
    const int lane = et & 31;
    const bool row_ok = row < rowsA;
    const int orow = (row_ok && a.row_map) ? a.row_map[row] : row;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32_wait(tbase + ch * 32, v);
        if (a.out_f32) {
            if (!row_ok) continue;
            // fp32 output: + add_scalar, kept where mask is nonzero (if given),
            // added to what out_f32 holds (if accumulate)
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int col = nb * BN + ch * 32 + g8 * 8;
                if (col < a.rowsB) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        f[e] = __uint_as_float(v[g8 * 8 + e]) + bias_sm[ch * 32 + g8 * 8 + e] + a.add_scalar;
                    if (a.mask) {
                        const uint4 m = *reinterpret_cast<const uint4*>(a.mask + (size_t)row * a.ldm + col);
                        const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (((mw[e >> 1] >> ((e & 1) * 16)) & 0x7fffu) == 0u) f[e] = 0.f;
                    }
                    float4* o = reinterpret_cast<float4*>(a.out_f32 + (size_t)orow * a.ldo + col);
                    if (a.accumulate) {
                        const float4 p0 = o[0], p1 = o[1];
                        f[0] += p0.x; f[1] += p0.y; f[2] += p0.z; f[3] += p0.w;
                        f[4] += p1.x; f[5] += p1.y; f[6] += p1.z; f[7] += p1.w;
                    }
                    o[0] = make_float4(f[0], f[1], f[2], f[3]);
                    o[1] = make_float4(f[4], f[5], f[6], f[7]);
                }
            }
        } else {
            float cs[32];
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int col = nb * BN + ch * 32 + g8 * 8;
                const bool ok = row_ok && col < a.rowsB;
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    f[e] = __uint_as_float(v[g8 * 8 + e]) + bias_sm[ch * 32 + g8 * 8 + e];
                    if (a.relu) f[e] = fmaxf(f[e], 0.f);
                    f[e] += a.add_scalar;
                }
                if (a.mask && ok) {
                    const uint4 m = *reinterpret_cast<const uint4*>(a.mask + (size_t)row * a.ldm + col);
                    const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (((mw[e >> 1] >> ((e & 1) * 16)) & 0x7fffu) == 0u) f[e] = 0.f;
                }
                if (ok) {
                    uint4 o;
                    o.x = pack_bf16x2(f[0], f[1]);
                    o.y = pack_bf16x2(f[2], f[3]);
                    o.z = pack_bf16x2(f[4], f[5]);
                    o.w = pack_bf16x2(f[6], f[7]);
                    *reinterpret_cast<uint4*>(a.out + (size_t)orow * a.ldo + col) = o;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) cs[g8 * 8 + e] = ok ? f[e] : 0.f;
            }
            if (a.colsum) {
                transpose_reduce32(cs, lane);  // lane u: column ch * 32 + u over the warp's 32 rows
                s_col[q * BN + ch * 32 + lane] = cs[0];
            }
        }
    }
    if (a.colsum && !a.out_f32) {
        named_bar_sync(2, kEpiThreads);
        // a CTA-pair tile's second half can lie wholly past the last row:
        // row block rt exists only if it holds a row
        const bool block_ok = rt * 128 < rowsA;
        for (int c = et; c < BN; c += kEpiThreads) {
            const int col = nb * BN + c;
            if (block_ok && col < a.rowsB)
                a.colsum[(size_t)rt * a.ldc + col] = ((s_col[c] + s_col[BN + c]) + s_col[2 * BN + c]) + s_col[3 * BN + c];
        }
    }
}

template <int BN, int MODE, int STAGES, int CAP = BN, int KSUB = 1>
__global__ void __launch_bounds__(192, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs a, int tok0)
{
    using L = Layout<BN, STAGES, KSUB>;
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* skip = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* epi_fail = reinterpret_cast<volatile int*>(tmem_slot + 3);
    float* bias_sm = reinterpret_cast<float*>(smem + L::BIAS_OFF);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + L::MASK_OFF);
    float* s_col = reinterpret_cast<float*>(smem + L::COL_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        *skip = has_error(a.status) ? 1 : 0;
        *abort_flag = 0;
        *epi_fail = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kEpiThreads);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (*skip) return;  // an earlier kernel of this call failed; uniform over the block
    if (a.zero_word && blockIdx.x == 0 && threadIdx.x == 0) *a.zero_word = 0;
    const int rowsA = a.rowsA_dev ? min(*a.rowsA_dev, a.rowsA) : a.rowsA;  // written by an earlier kernel
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_m = (rowsA + BM - 1) / BM;
    const int num_n = (a.rowsB + BN - 1) / BN;
    const int num_kb = (gemm_k(a) + BK - 1) / BK;
    const int num_tiles = num_kb > 0 ? num_m * num_n : 0;  // no k-block: nothing to add or store

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // the gate GEMM streams W_gate once: its lines go first, so that the
            // W_up / W_down rows the epilogue prefetches for the next kernel stay
            const uint64_t pol_a = l2_policy_evict_first();
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int mb = tile % num_m, nb = tile / num_m;
                // gate GEMM: each tile starts at its own k so that the CTAs do not
                // all ask for the same few lines of x at once (sum order: per tile)
                const int rot = MODE == GEMM_GATE_SWAP ? (int)((unsigned)(tile * 5 * KSUB) % (unsigned)num_kb) : 0;
                for (int kb0 = 0; kb0 < num_kb; kb0 += KSUB) {
                    const int kb = kb0 + rot < num_kb ? kb0 + rot : kb0 + rot - num_kb;
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
#pragma unroll
                    for (int sub = 0; sub < KSUB; ++sub) {
                        uint8_t* ss = sa + sub * L::SUB_BYTES;
                        if constexpr (MODE == GEMM_GATE_SWAP)
                            tma_load_2d_hint(ss, &tmA, (kb + sub) * BK, mb * BM, &full[stage], pol_a);
                        else
                            tma_load_2d(ss, &tmA, (kb + sub) * BK, mb * BM, &full[stage]);
                        tma_load_2d(ss + L::A_BYTES, &tmB, (kb + sub) * BK, nb * BN, &full[stage]);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) fail(a.status, abort_flag);
            // The last load issued into each stage must land before the CTA exits.
            for (int s = 0; s < STAGES; ++s) {
                const long long n_s = issued / STAGES + (s < issued % STAGES ? 1 : 0);
                if (n_s > 0) mbar_wait(&full[s], (uint32_t)((n_s - 1) & 1), nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < num_kb; kb += KSUB) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int sub = 0; sub < KSUB; ++sub) {
                        const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES + sub * L::SUB_BYTES);
                        const uint64_t adesc = sw128_kmajor_desc(sa);
                        const uint64_t bdesc = sw128_kmajor_desc(sa + L::A_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            umma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC, (kb | sub | k) != 0);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) fail(a.status, abort_flag);
            umma_commit(mma_done);  // every MMA issued above has finished once this arrives
            mbar_wait(mma_done, 0, nullptr);
        }
    } else {
        // --------------------------------------------------- epilogue -----
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int et = threadIdx.x - 64;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int mb = tile % num_m, nb = tile / num_m;
            named_bar_sync(1, kEpiThreads);  // previous tile's shared-memory reads are done
            if (MODE == GEMM_TWELL_RELU || MODE == GEMM_DENSE) {
                for (int c = et; c < BN; c += kEpiThreads) {
                    const int col = nb * BN + c;
                    float bv;
                    if (MODE == GEMM_TWELL_RELU)
                        bv = col < a.rowsB ? a.bias[col] : -INFINITY;
                    else
                        bv = (a.bias && col < a.rowsB) ? a.bias[col] : 0.f;
                    bias_sm[c] = bv;
                }
            }
            if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) *epi_fail = 1;
            named_bar_sync(1, kEpiThreads);
            if (*epi_fail) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);

            if constexpr (MODE == GEMM_TWELL_RELU) {
                epi_twell_row<BN, CAP>(tbase, mb * BM + 32 * q + lane, rowsA, nb, a, bias_sm);
            } else if constexpr (MODE == GEMM_GATE_SWAP) {
                // Tokens in chunks of 16 accumulator columns under a loop that
                // is not unrolled: fully unrolled over 64 tokens this code no
                // longer fit the instruction cache and starved the producer
                // and MMA threads. TMEM is read twice (masks, then values).
                const int j = mb * BM + 32 * q + lane;  // hidden unit
                const bool j_ok = j < a.rowsA;
                const float bj = j_ok ? a.bias[j] : 0.f;
                const int ntok = min(BN, a.rowsB);
                bool any = false;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16_wait(tbase + c0, v);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int t = c0 + u;
                        if (t < ntok) {
                            const bool act = j_ok && (__uint_as_float(v[u]) + bj > 0.f);
                            any |= act;
                            const uint32_t m = __ballot_sync(0xffffffffu, act);
                            if (lane == 0) s_mask[t * 4 + q] = m;
                        }
                    }
                }
                if (a.pf_row_bytes > 0) {
                    // the next kernel reads the W_up and W_down rows of every
                    // active unit: start pulling them into L2 now, one warp per row
                    uint32_t units = __ballot_sync(0xffffffffu, any);
                    while (units) {
                        const int jj = mb * BM + 32 * q + __ffs(units) - 1;
                        units &= units - 1;
                        for (int off = lane * 128; off < a.pf_row_bytes; off += 32 * 128) {
                            prefetch_l2_keep(reinterpret_cast<const char*>(a.pf0) + (size_t)jj * a.pf_row_bytes + off);
                            prefetch_l2_keep(reinterpret_cast<const char*>(a.pf1) + (size_t)jj * a.pf_row_bytes + off);
                        }
                    }
                }
                named_bar_sync(1, kEpiThreads);
                const uint32_t lt = lanemask_lt();
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16_wait(tbase + c0, v);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int t = c0 + u;
                        if (t < ntok) {
                            const uint32_t mq = s_mask[t * 4 + q];
                            if ((mq >> lane) & 1u) {
                                int before = __popc(mq & lt);
                                for (int qq = 0; qq < q; ++qq) before += __popc(s_mask[t * 4 + qq]);
                                const float g = __uint_as_float(v[u]) + bj;
                                a.gstage[((size_t)(tok0 + t) * a.NB + mb) * BM + before] =
                                    make_uint2((uint32_t)j, __float_as_uint(g));
                            }
                        }
                    }
                }
                // per-token counts of this tile, one epilogue thread per token
                for (int t = et; t < ntok; t += kEpiThreads) {
                    const int total = __popc(s_mask[t * 4 + 0]) + __popc(s_mask[t * 4 + 1]) +
                                      __popc(s_mask[t * 4 + 2]) + __popc(s_mask[t * 4 + 3]);
                    a.stage_cnt[(size_t)(tok0 + t) * a.NB + mb] = total;
                    if (total && a.nnz) atomicAdd(&a.nnz[tok0 + t], total);
                }
            } else {  // GEMM_DENSE
                epi_dense_row<BN>(tbase, mb * BM + 32 * q + lane, rowsA, nb, a, bias_sm, s_col, mb, q, et);
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (*epi_fail) fail(a.status, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------- CTA pairs --
//
// The same GEMM on 256 x 256 tiles computed by a cluster of two CTAs with
// tcgen05.mma.cta_group::2. Each CTA loads 128 rows of A and 128 of the
// tile's 256 rows of B per k-block (32 KB instead of the 48 KB that a
// 128 x 256 tile per CTA needs): the SM's share of operand traffic falls by a
// third at the same MMA work per SM, which matters because the single-CTA
// kernel is limited by how fast operands reach the SM.
//
//   warp 0 (both CTAs)   TMA producer of its own halves; completions are
//                        counted on the even CTA's full barrier.
//   warp 1 (both CTAs)   pair-collective TMEM allocation (all 512 columns:
//                        two 256-column accumulators); in the even CTA lane 0
//                        also issues the MMAs and commits to the barriers of
//                        both CTAs (multicast).
//   warps 2-5            epilogue of the CTA's own 128 rows x 256 columns;
//                        each warp then arrives on the even CTA's tmem-empty
//                        barrier (8 arrivals per accumulator).
// Both CTAs always reach the pair-collective allocation, the deallocation and
// the cluster barriers: the only early exit is taken by both, on a decision
// read from the even CTA.

constexpr int PAIR_M = 256;   // tile rows over the pair
constexpr int PAIR_N = 256;   // tile columns (B rows over the pair)
constexpr int HALF = 128;     // rows of A and of B held by one CTA

// Tile order of the CTA-pair kernel: groups of kRasterN consecutive column
// tiles; inside a group the column tile varies fastest. The ~76 pairs at work
// at any time then cover about 5 row tiles x 16 column tiles, whose A rows and
// B rows (~42 MB at K = 4096) stay in L2, so A is read from DRAM once per
// group instead of once per column tile. At 16384 x 16384 x 4096: 16 column
// tiles per group 1.6-2 % faster than 8, 32 slower (its group's rows no
// longer stay in L2), 4 slower still.
constexpr int kRasterN = 16;

__device__ __forceinline__ void pair_tile_coords(int tile, int num_m, int num_n, int* mb, int* nb)
{
    const int group = tile / (kRasterN * num_m);
    const int first_n = group * kRasterN;
    const int gn = min(kRasterN, num_n - first_n);
    const int local = tile - group * kRasterN * num_m;
    *mb = local / gn;
    *nb = first_n + local % gn;
}

template <int STAGES>
struct PairLayout {
    static constexpr int A_BYTES = HALF * BK * 2;
    static constexpr int B_BYTES = HALF * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BIAS_OFF = (MISC_OFF + 16 + 15) & ~15;
    static constexpr int COL_OFF = BIAS_OFF + PAIR_N * 4;
    static constexpr int TOTAL = COL_OFF + 4 * PAIR_N * 4 + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 2 * PAIR_N;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned");
};

// Operands stored MN-major (A_MN, B_MN: the matrix is given as its transpose,
// [K, rows] row-major) arrive as two 64-row x 64-element TMA boxes per CTA
// half and k-block, 8 KB apart: the 128-byte-swizzled MN-major layout whose
// 64-element blocks along MN are 8 KB apart and whose 8-row groups along K
// are 1024 bytes apart. A 16-deep K step then advances 2048 bytes instead of
// the K-major operand's 32.
constexpr int kMnBox = 64;

__device__ __forceinline__ uint64_t operand_desc(bool mn, uint32_t addr)
{
    return mn ? sw128_mnmajor_desc(addr, kMnBox * BK * 2) : sw128_kmajor_desc(addr);
}

template <int MODE, int STAGES, int CAP = PAIR_N, bool A_MN = false, bool B_MN = false>
__global__ void __launch_bounds__(192, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs a)
{
    static_assert(MODE == GEMM_TWELL_RELU || MODE == GEMM_DENSE, "row-wise epilogues only");
    static_assert(MODE == GEMM_DENSE || (!A_MN && !B_MN), "MN-major operands: dense epilogue only");
    using L = PairLayout<STAGES>;
    constexpr uint32_t IDESC =
        idesc_bf16_f32(PAIR_M, PAIR_N) | (A_MN ? kIdescAMn : 0u) | (B_MN ? kIdescBMn : 0u);
    constexpr uint64_t A_KSTEP = A_MN ? (16u * 128u) >> 4 : 2u;  // descriptor units (16 B) per 16-deep K step
    constexpr uint64_t B_KSTEP = B_MN ? (16u * 128u) >> 4 : 2u;
    constexpr int kEpiWarps = 2 * (kEpiThreads / 32);  // tmem-empty arrivals: both CTAs
    extern __shared__ uint8_t smem_raw[];
    // Same offset in both CTAs (same kernel, same static shared memory), as the
    // pair MMA addresses the peer's operands with the leader's descriptors.
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* skip = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* epi_fail = reinterpret_cast<volatile int*>(tmem_slot + 3);
    float* bias_sm = reinterpret_cast<float*>(smem + L::BIAS_OFF);
    float* s_col = reinterpret_cast<float*>(smem + L::COL_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        *skip = (leader && has_error(a.status)) ? 1 : 0;
        *abort_flag = 0;
        *epi_fail = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    cluster_sync();  // barriers of both CTAs initialised before either uses the other's
    const int sk = ld_cluster_s32(cluster_addr(const_cast<int*>(skip), 0));
    cluster_sync();  // the leader's flag has been read before anyone may leave
    if (sk) return;  // an earlier kernel of this call failed; uniform over the pair
    const int rowsA = a.rowsA_dev ? min(*a.rowsA_dev, a.rowsA) : a.rowsA;  // same in both CTAs
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_m = (rowsA + PAIR_M - 1) / PAIR_M;
    const int num_n = (a.rowsB + PAIR_N - 1) / PAIR_N;
    const int num_kb = (gemm_k(a) + BK - 1) / BK;  // same in both CTAs
    const int num_tiles = num_kb > 0 ? num_m * num_n : 0;  // no k-block: nothing to add or store
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            const uint32_t full_leader = cluster_addr(full, 0);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                int mb, nb;
                pair_tile_coords(tile, num_m, num_n, &mb, &nb);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * L::STAGE_BYTES);
                    const uint32_t fb = full_leader + 8u * (uint32_t)stage;
                    const int ma = mb * PAIR_M + (int)rank * HALF, nbr = nb * PAIR_N + (int)rank * HALF;
                    if (A_MN) {
                        tma_load_2d_pair(sa, &tmA, ma, kb * BK, fb);
                        tma_load_2d_pair(sa + kMnBox * BK * 2, &tmA, ma + kMnBox, kb * BK, fb);
                    } else {
                        tma_load_2d_pair(sa, &tmA, kb * BK, ma, fb);
                    }
                    if (B_MN) {
                        tma_load_2d_pair(sa + L::A_BYTES, &tmB, nbr, kb * BK, fb);
                        tma_load_2d_pair(sa + L::A_BYTES + kMnBox * BK * 2, &tmB, nbr + kMnBox, kb * BK, fb);
                    } else {
                        tma_load_2d_pair(sa + L::A_BYTES, &tmB, kb * BK, nbr, fb);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) fail(a.status, abort_flag);
            // The last load issued into each stage must land before the CTA
            // exits: the leader sees it on its full barrier, the peer on its
            // empty barrier (the leader's MMAs consumed it).
            for (int s = 0; s < STAGES; ++s) {
                const long long n_s = issued / STAGES + (s < issued % STAGES ? 1 : 0);
                if (n_s > 0) mbar_wait(leader ? &full[s] : &empty[s], (uint32_t)((n_s - 1) & 1), nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------- MMA issuer (even CTA) -----
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PAIR_N);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
                    const uint64_t adesc = operand_desc(A_MN, sa);
                    const uint64_t bdesc = operand_desc(B_MN, sa + L::A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_pair(d_tmem, adesc + A_KSTEP * k, bdesc + B_KSTEP * k, IDESC, (kb | k) != 0);
                    umma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) fail(a.status, abort_flag);
            umma_commit_pair(mma_done, 0x1);  // every MMA issued above has finished once this arrives
            mbar_wait(mma_done, 0, nullptr);
        }
    } else {
        // --------------------------------------------------- epilogue -----
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int et = threadIdx.x - 64;
        const uint32_t tempty_leader = cluster_addr(tempty, 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = pair; tile < num_tiles; tile += num_pairs) {
            int mb, nb;
            pair_tile_coords(tile, num_m, num_n, &mb, &nb);
            named_bar_sync(1, kEpiThreads);  // previous tile's shared-memory reads are done
            for (int c = et; c < PAIR_N; c += kEpiThreads) {
                const int col = nb * PAIR_N + c;
                float bv;
                if (MODE == GEMM_TWELL_RELU)
                    bv = col < a.rowsB ? a.bias[col] : -INFINITY;
                else
                    bv = (a.bias && col < a.rowsB) ? a.bias[col] : 0.f;
                bias_sm[c] = bv;
            }
            if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) *epi_fail = 1;
            named_bar_sync(1, kEpiThreads);
            if (*epi_fail) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * PAIR_N);
            const int row = mb * PAIR_M + (int)rank * HALF + 32 * q + lane;
            if constexpr (MODE == GEMM_TWELL_RELU)
                epi_twell_row<PAIR_N, CAP>(tbase, row, rowsA, nb, a, bias_sm);
            else
                epi_dense_row<PAIR_N>(tbase, row, rowsA, nb, a, bias_sm, s_col, 2 * mb + (int)rank, q, et);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * (uint32_t)acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (*epi_fail) fail(a.status, abort_flag);
    }

    // Neither CTA deallocates or exits while the pair's MMAs, loads or
    // arrivals may still touch the other's tensor or shared memory.
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------ tensor maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [rows, K] bf16 row-major, box = 64 (K) x box_rows, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int K, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int STAGES, int CAP = BN, int KSUB = 1>
cudaError_t run(const uint16_t* A, const uint16_t* B, const GemmArgs& a, int tok0, int sm_count, cudaStream_t s)
{
    using L = Layout<BN, STAGES, KSUB>;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, a.rowsA, a.K, BM) || !make_map(&mb, B, a.rowsB, a.K, BN)) return cudaErrorInvalidValue;
    auto kern = k_gemm_tc<BN, MODE, STAGES, CAP, KSUB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    const int tiles = ((a.rowsA + BM - 1) / BM) * ((a.rowsB + BN - 1) / BN);
    const int grid = tiles < sm_count ? tiles : sm_count;
    count_launches(1);
    kern<<<grid, 192, L::TOTAL, s>>>(ma, mb, a, tok0);
    return cudaGetLastError();
}

// Clusters of two that can be resident at once for this kernel (0 = none).
// [K, mn] bf16 row-major (an MN-major operand), box = 64 (MN) x 64 (K), 128-byte swizzle, zero fill.
bool make_map_mn(CUtensorMap* m, const void* ptr, int mn, int K)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)mn, (cuuint64_t)K};
    cuuint64_t strides[1] = {(cuuint64_t)mn * 2};
    cuuint32_t box[2] = {(cuuint32_t)kMnBox, (cuuint32_t)BK};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int STAGES, int CAP, bool A_MN, bool B_MN>
int pair_capacity(cudaLaunchConfig_t cfg)
{
    static int cached[64] = {0};
    static bool known[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!known[dev]) {
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pair<MODE, STAGES, CAP, A_MN, B_MN>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        cached[dev] = n;
        known[dev] = true;
    }
    return cached[dev];
}

// Launches the pair kernel; *launched = false (and nothing enqueued) when no
// cluster of two fits, so the caller can take the single-CTA kernel.
template <int MODE, int STAGES, int CAP = PAIR_N, bool A_MN = false, bool B_MN = false>
cudaError_t run_pair(const uint16_t* A, const uint16_t* B, const GemmArgs& a, cudaStream_t s, bool* launched)
{
    using L = PairLayout<STAGES>;
    *launched = false;
    auto kern = k_gemm_pair<MODE, STAGES, CAP, A_MN, B_MN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = L::TOTAL;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int cap = pair_capacity<MODE, STAGES, CAP, A_MN, B_MN>(cfg);
    if (cap <= 0) return cudaSuccess;
    CUtensorMap ma, mb;
    const bool ok_a = A_MN ? make_map_mn(&ma, A, a.rowsA, a.K) : make_map(&ma, A, a.rowsA, a.K, HALF);
    const bool ok_b = B_MN ? make_map_mn(&mb, B, a.rowsB, a.K) : make_map(&mb, B, a.rowsB, a.K, HALF);
    if (!ok_a || !ok_b) return cudaErrorInvalidValue;
    const int tiles = ((a.rowsA + PAIR_M - 1) / PAIR_M) * ((a.rowsB + PAIR_N - 1) / PAIR_N);
    cfg.gridDim = dim3(2 * (tiles < cap ? tiles : cap), 1, 1);
    count_launches(1);
    *launched = true;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, a);
}

// Row-wise epilogues: 256 x 256 tiles on CTA pairs when there are more than
// 128 rows, else (or without room for a cluster of two) 128 x 256 tiles on
// single CTAs.
template <int MODE, int CAP>
cudaError_t launch_row_wise(const uint16_t* A, const uint16_t* B, const GemmArgs& a, int sm_count, cudaStream_t s)
{
    if (a.rowsA > HALF) {
        bool launched = false;
        const cudaError_t e = run_pair<MODE, 6, CAP>(A, B, a, s, &launched);
        if (e != cudaSuccess || launched) return e;
    }
    return run<256, MODE, 4, CAP>(A, B, a, 0, sm_count, s);
}

}  // namespace

int gemm_block_n(int mode, int rowsB)
{
    if (mode == GEMM_GATE_SWAP) return rowsB <= 16 ? 16 : rowsB <= 32 ? 32 : 64;
    return 256;
}

cudaError_t launch_gemm(int mode, const uint16_t* A, const uint16_t* B, const GemmArgs& a, int sm_count,
                        cudaStream_t s)
{
    switch (mode) {
        case GEMM_TWELL_RELU:
            // Staging segments of 256, 64 or 32 entries (compile-time strides).
            switch (a.stage_cap) {
                case 256: return launch_row_wise<GEMM_TWELL_RELU, 256>(A, B, a, sm_count, s);
                case 64: return launch_row_wise<GEMM_TWELL_RELU, 64>(A, B, a, sm_count, s);
                case 32: return launch_row_wise<GEMM_TWELL_RELU, 32>(A, B, a, sm_count, s);
                default: return cudaErrorInvalidValue;
            }
        case GEMM_DENSE: {
            if (!a.a_mn && !a.b_mn) return launch_row_wise<GEMM_DENSE, 256>(A, B, a, sm_count, s);
            // MN-major operands: CTA pairs only
            bool launched = false;
            cudaError_t e;
            if (a.a_mn && a.b_mn)
                e = run_pair<GEMM_DENSE, 6, PAIR_N, true, true>(A, B, a, s, &launched);
            else if (a.b_mn)
                e = run_pair<GEMM_DENSE, 6, PAIR_N, false, true>(A, B, a, s, &launched);
            else
                e = run_pair<GEMM_DENSE, 6, PAIR_N, true, false>(A, B, a, s, &launched);
            if (e != cudaSuccess) return e;
            return launched ? cudaSuccess : cudaErrorNotSupported;
        }
        case GEMM_GATE_SWAP: {
            // B = x: token chunks of at most 64 rows, each a separate launch.
            const int bn = gemm_block_n(mode, a.rowsB);
            for (int t0 = 0; t0 < a.rowsB; t0 += 64) {
                GemmArgs c = a;
                c.rowsB = a.rowsB - t0 < 64 ? a.rowsB - t0 : 64;
                const uint16_t* Bc = B + (size_t)t0 * a.K;
                cudaError_t e;
                const int num_kb = (a.K + BK - 1) / BK;
                if (bn == 16 && num_kb % 4 == 0)
                    // four consecutive k-blocks per stage: 512 contiguous bytes of
                    // each W_gate row per stage
                    e = run<16, GEMM_GATE_SWAP, 3, 16, 4>(A, Bc, c, t0, sm_count, s);
                else if (bn == 16)
                    e = run<16, GEMM_GATE_SWAP, 11>(A, Bc, c, t0, sm_count, s);
                else if (bn == 32 && num_kb % 2 == 0)
                    e = run<32, GEMM_GATE_SWAP, 5, 32, 2>(A, Bc, c, t0, sm_count, s);
                else if (bn == 32)
                    e = run<32, GEMM_GATE_SWAP, 8>(A, Bc, c, t0, sm_count, s);
                else if (num_kb % 2 == 0)
                    e = run<64, GEMM_GATE_SWAP, 4, 64, 2>(A, Bc, c, t0, sm_count, s);
                else
                    e = run<64, GEMM_GATE_SWAP, 8>(A, Bc, c, t0, sm_count, s);
                if (e != cudaSuccess) return e;
            }
            return cudaSuccess;
        }
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace twell
