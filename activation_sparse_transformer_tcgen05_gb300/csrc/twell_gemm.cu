// twell_gemm.cu — persistent tcgen05 GEMM with a TwELL-emitting epilogue.
//
// D = A B^T with A [rowsA, K] and B [rowsB, K] bf16, both K-major, fp32
// accumulation in tensor memory. The pages build TwELL "directly in the
// epilogue of highly optimised dense matmul kernels", with no separate
// conversion kernel and no synchronisation between CTAs ("Sparser, Faster,
// Lighter Transformer Language Models", Resumo Técnico §2, "Formato de Dados
// TwELL"). Here each CTA compacts its own 128 x BN output tile independently:
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

template <int BN, int STAGES>
struct Layout {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BIAS_OFF = (MISC_OFF + 16 + 15) & ~15;
    static constexpr int BIAS_BYTES = 4 * (BN > BM ? BN : BM);
    static constexpr int MASK_OFF = BIAS_OFF + BIAS_BYTES;
    static constexpr int MASK_BYTES = 64 * 4 * 4;
    static constexpr int TOTAL = MASK_OFF + MASK_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                        : (2 * BN <= 256) ? 256 : 512;
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned");
};

__device__ __forceinline__ void fail(int32_t* status, volatile int* abort_flag)
{
    set_error(status, TWELL_ERR_TIMEOUT);
    *abort_flag = 1;
}

template <int BN, int MODE, int STAGES>
__global__ void __launch_bounds__(192, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs a, int tok0)
{
    using L = Layout<BN, STAGES>;
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

    const int num_m = (a.rowsA + BM - 1) / BM;
    const int num_n = (a.rowsB + BN - 1) / BN;
    const int num_kb = (a.K + BK - 1) / BK;
    const int num_tiles = num_m * num_n;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int mb = tile % num_m, nb = tile / num_m;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
                    tma_load_2d(sa, &tmA, kb * BK, mb * BM, &full[stage]);
                    tma_load_2d(sa + L::A_BYTES, &tmB, kb * BK, nb * BN, &full[stage]);
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
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
                    const uint64_t adesc = sw128_kmajor_desc(sa);
                    const uint64_t bdesc = sw128_kmajor_desc(sa + L::A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC, (kb | k) != 0);
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
                const int row = mb * BM + 32 * q + lane;
                const bool row_ok = row < a.rowsA;
                uint32_t* st = a.stage + ((size_t)(row_ok ? row : 0) * a.NB + nb) * BN;
                int cnt = 0;
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32_wait(tbase + ch * 32, v);
                    if (row_ok) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const float p = __uint_as_float(v[c]) + bias_sm[ch * 32 + c];
                            if (p > 0.f) {
                                const uint32_t hb = f32_to_bf16_bits(p);
                                if (hb != 0u) st[cnt++] = (hb << 16) | (uint32_t)(ch * 32 + c);
                            }
                        }
                    }
                }
                if (row_ok) {
                    a.stage_cnt[(size_t)row * a.NB + nb] = cnt;
                    if (cnt) atomicAdd(&a.nnz[row], cnt);
                }
            } else if constexpr (MODE == GEMM_GATE_SWAP) {
                const int j = mb * BM + 32 * q + lane;  // hidden unit
                const bool j_ok = j < a.rowsA;
                const float bj = j_ok ? a.bias[j] : 0.f;
                const int ntok = min(BN, a.rowsB);
                uint32_t v[BN];
                if constexpr (BN == 16) {
                    uint32_t (&v16)[16] = *reinterpret_cast<uint32_t(*)[16]>(v);
                    tmem_ld16_wait(tbase, v16);
                } else {
#pragma unroll
                    for (int ch = 0; ch < BN / 32; ++ch) {
                        uint32_t (&v32)[32] = *reinterpret_cast<uint32_t(*)[32]>(v + ch * 32);
                        tmem_ld32_wait(tbase + ch * 32, v32);
                    }
                }
#pragma unroll
                for (int t = 0; t < BN; ++t) {
                    if (t < ntok) {
                        const bool act = j_ok && (__uint_as_float(v[t]) + bj > 0.f);
                        const uint32_t m = __ballot_sync(0xffffffffu, act);
                        if (lane == 0) s_mask[t * 4 + q] = m;
                    }
                }
                named_bar_sync(1, kEpiThreads);
                const uint32_t lt = lanemask_lt();
#pragma unroll
                for (int t = 0; t < BN; ++t) {
                    if (t < ntok) {
                        const uint32_t mq = s_mask[t * 4 + q];
                        if ((mq >> lane) & 1u) {
                            int before = __popc(mq & lt);
                            for (int qq = 0; qq < q; ++qq) before += __popc(s_mask[t * 4 + qq]);
                            const float g = __uint_as_float(v[t]) + bj;
                            a.gstage[((size_t)(tok0 + t) * a.NB + mb) * BM + before] =
                                make_uint2((uint32_t)j, __float_as_uint(g));
                        }
                        if (et == 0) {
                            const int total = __popc(s_mask[t * 4 + 0]) + __popc(s_mask[t * 4 + 1]) +
                                              __popc(s_mask[t * 4 + 2]) + __popc(s_mask[t * 4 + 3]);
                            a.stage_cnt[(size_t)(tok0 + t) * a.NB + mb] = total;
                            if (total) atomicAdd(&a.nnz[tok0 + t], total);
                        }
                    }
                }
            } else {  // GEMM_DENSE
                const int row = mb * BM + 32 * q + lane;
                const bool row_ok = row < a.rowsA;
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32_wait(tbase + ch * 32, v);
                    if (row_ok) {
#pragma unroll
                        for (int g8 = 0; g8 < 4; ++g8) {
                            const int col = nb * BN + ch * 32 + g8 * 8;
                            if (col < a.rowsB) {
                                float f[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    f[e] = __uint_as_float(v[g8 * 8 + e]) + bias_sm[ch * 32 + g8 * 8 + e];
                                    if (a.relu) f[e] = fmaxf(f[e], 0.f);
                                }
                                uint4 o;
                                o.x = pack_bf16x2(f[0], f[1]);
                                o.y = pack_bf16x2(f[2], f[3]);
                                o.z = pack_bf16x2(f[4], f[5]);
                                o.w = pack_bf16x2(f[6], f[7]);
                                *reinterpret_cast<uint4*>(a.out + (size_t)row * a.ldo + col) = o;
                            }
                        }
                    }
                }
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

template <int BN, int MODE, int STAGES>
cudaError_t run(const uint16_t* A, const uint16_t* B, const GemmArgs& a, int tok0, int sm_count, cudaStream_t s)
{
    using L = Layout<BN, STAGES>;
    CUtensorMap ma, mb;
    if (!make_map(&ma, A, a.rowsA, a.K, BM) || !make_map(&mb, B, a.rowsB, a.K, BN)) return cudaErrorInvalidValue;
    auto kern = k_gemm_tc<BN, MODE, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    const int tiles = ((a.rowsA + BM - 1) / BM) * ((a.rowsB + BN - 1) / BN);
    const int grid = tiles < sm_count ? tiles : sm_count;
    count_launches(1);
    kern<<<grid, 192, L::TOTAL, s>>>(ma, mb, a, tok0);
    return cudaGetLastError();
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
            return run<256, GEMM_TWELL_RELU, 4>(A, B, a, 0, sm_count, s);
        case GEMM_DENSE:
            return run<256, GEMM_DENSE, 4>(A, B, a, 0, sm_count, s);
        case GEMM_GATE_SWAP: {
            // B = x: token chunks of at most 64 rows, each a separate launch.
            const int bn = gemm_block_n(mode, a.rowsB);
            for (int t0 = 0; t0 < a.rowsB; t0 += 64) {
                GemmArgs c = a;
                c.rowsB = a.rowsB - t0 < 64 ? a.rowsB - t0 : 64;
                const uint16_t* Bc = B + (size_t)t0 * a.K;
                cudaError_t e;
                if (bn == 16)
                    e = run<16, GEMM_GATE_SWAP, 11>(A, Bc, c, t0, sm_count, s);
                else if (bn == 32)
                    e = run<32, GEMM_GATE_SWAP, 8>(A, Bc, c, t0, sm_count, s);
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
