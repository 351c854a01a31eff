// twell_sparse.cu — TwELL construction, sparse products and the sparse backward.
//
// The method ("Sparser, Faster, Lighter Transformer Language Models", Resumo
// Técnico §2 Metodologia) packs the ReLU hidden matrix into TwELL and runs the
// down-projection and the training kernels only over the stored entries. These
// are the CUDA-core kernels of that path: every one is a gather over rows of a
// dense bf16 matrix (W_down, W_up, x or dy) named by TwELL indices, with fp32
// accumulation. Work is split so that a warp's 32 lanes read one 512-byte
// stretch of a gathered row with 128-bit loads; all reductions run in a fixed
// order, so results are bit-reproducible.
#include "sparse_common.cuh"

namespace twell {

std::atomic<long long> g_kernel_launches{0};
KernelTimer g_timer{0, nullptr, nullptr};

namespace {

// ------------------------------------------------------------ construction --

// nnz[r] = number of entries of row r of a dense bf16 matrix that are not +-0.
__global__ void k_count_dense(const uint16_t* __restrict__ h, int ldh, TwellView tw, const int32_t* status)
{
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= tw.M || has_error(status)) return;
    const uint16_t* row = h + (size_t)r * ldh;
    int c = 0;
    for (int j = lane * 8; j < tw.F; j += 256) {
        const uint4 q = ldg16(row + j);
        c += nz_bf16(q.x) + nz_bf16(q.x >> 16) + nz_bf16(q.y) + nz_bf16(q.y >> 16) + nz_bf16(q.z) +
             nz_bf16(q.z >> 16) + nz_bf16(q.w) + nz_bf16(q.w >> 16);
    }
    c = warp_sum_i(c);
    if (lane == 0) tw.nnz[r] = c;
}

// One block of 1024 threads: K[t] = max nnz over tile t (a warp per tile), then
// off[] = exclusive prefix of rows(t) * K[t]; flags a capacity overflow.
__global__ void __launch_bounds__(1024) k_tile_layout(TwellView tw, int32_t* status)
{
    __shared__ int64_t s_chunk[1024];
    __shared__ int64_t s_warp[32];
    __shared__ int64_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (has_error(status)) return;
    if (tid == 0) {
        s_carry = 0;
        tw.off[0] = 0;
    }
    __syncthreads();
    for (int t0 = 0; t0 < tw.n_tiles; t0 += 1024) {
        const int chunk = min(1024, tw.n_tiles - t0);
        for (int tt = warp; tt < chunk; tt += 32) {
            const int t = t0 + tt, r0 = t * tw.T, rows = min(tw.T, tw.M - r0);
            int mx = 0;
            for (int i = lane; i < rows; i += 32) mx = max(mx, tw.nnz[r0 + i]);
            mx = warp_max_i(mx);
            if (lane == 0) {
                tw.K[t] = mx;
                s_chunk[tt] = (int64_t)rows * mx;
            }
        }
        __syncthreads();
        int64_t v = tid < chunk ? s_chunk[tid] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) s_warp[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int64_t w = s_warp[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int64_t n = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += n;
            }
            s_warp[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int64_t incl = v + (warp > 0 ? s_warp[warp - 1] : 0);
        if (tid < chunk) tw.off[t0 + tid + 1] = s_carry + incl;
        __syncthreads();
        if (tid == 0) s_carry += s_warp[31];
        __syncthreads();
    }
    if (tid == 0 && s_carry > tw.cap) set_error(status, TWELL_ERR_CAPACITY);
}

// Slots of row r (a warp) from a dense bf16 matrix: warp prefix-sum order keeps
// the columns ascending; padding (-1, +0) after the row's entries.
__global__ void k_fill_dense(const uint16_t* __restrict__ h, int ldh, TwellView tw, const int32_t* status)
{
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= tw.M || has_error(status) || over_capacity(tw)) return;
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    const uint16_t* row = h + (size_t)r * ldh;
    int pos = 0;
    for (int j0 = 0; j0 < tw.F; j0 += 256) {
        const int j = j0 + lane * 8;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (j < tw.F) q = ldg16(row + j);
        const uint32_t e[4] = {q.x, q.y, q.z, q.w};
        int c = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) c += nz_bf16(e[k]) + nz_bf16(e[k] >> 16);
        const int incl = warp_incl_scan(c, lane);
        int64_t p = base + pos + (incl - c);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t hv = (e[k >> 1] >> ((k & 1) * 16)) & 0xffffu;
            if (nz_bf16(hv)) {
                tw.idx[p] = j + k;
                tw.val[p] = (uint16_t)hv;
                ++p;
            }
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int k = pos + lane; k < Kt; k += 32) {
        tw.idx[base + k] = -1;
        tw.val[base + k] = 0;
    }
}

// Slots of row r (a warp) from the up-projection epilogue's staging: the row's
// column blocks are concatenated in block order (each block's entries are
// already ascending), then padded. Blocks go 64 at a time (two per lane), and
// the first four entries of both of a lane's blocks are loaded before any is
// stored, so that at ~1 % density (2.6 entries per block) a row costs two
// dependent round trips instead of one per entry.
__device__ __forceinline__ void fill_row_staged(const uint32_t* __restrict__ stage,
                                                const int32_t* __restrict__ stage_cnt, int NB, int nb_end, int BN,
                                                int stride, const TwellView& tw, int r, int64_t base, int Kt, int lane)
{
    int pos = 0;
    for (int nb0 = 0; nb0 < nb_end; nb0 += 64) {
        int c[2], incl[2];
        const uint32_t* src[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nb = nb0 + 32 * h + lane;
            c[h] = nb < nb_end ? stage_cnt[(size_t)r * NB + nb] : 0;
            src[h] = stage + ((size_t)r * NB + nb) * stride;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) incl[h] = warp_incl_scan(c[h], lane);
        const int tot0 = __shfl_sync(0xffffffffu, incl[0], 31);
        uint32_t w[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) w[h][q] = q < c[h] ? src[h][q] : 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nb = nb0 + 32 * h + lane;
            const int64_t p = base + pos + (h ? tot0 : 0) + (incl[h] - c[h]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q < c[h]) {
                    tw.idx[p + q] = nb * BN + (int)(w[h][q] & 0xffffu);
                    tw.val[p + q] = (uint16_t)(w[h][q] >> 16);
                }
            }
            for (int e = 4; e < c[h]; ++e) {  // denser blocks
                const uint32_t v = src[h][e];
                tw.idx[p + e] = nb * BN + (int)(v & 0xffffu);
                tw.val[p + e] = (uint16_t)(v >> 16);
            }
        }
        pos += tot0 + __shfl_sync(0xffffffffu, incl[1], 31);
    }
    for (int k = pos + lane; k < Kt; k += 32) {
        tw.idx[base + k] = -1;
        tw.val[base + k] = 0;
    }
}

// A warp per row. With ov_pos (hybrid format), rows routed to the dense
// overflow block (ov_pos[r] >= 0) are left empty here: padding only.
__global__ void k_fill_staged_relu(const uint32_t* __restrict__ stage, const int32_t* __restrict__ stage_cnt, int NB,
                                   int BN, int stride, TwellView tw, const int32_t* __restrict__ ov_pos,
                                   const int32_t* status)
{
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= tw.M || has_error(status) || over_capacity(tw)) return;
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    const int nb_end = (ov_pos && ov_pos[r] >= 0) ? 0 : NB;
    fill_row_staged(stage, stage_cnt, NB, nb_end, BN, stride, tw, r, base, Kt, lane);
}

// Layout and fill of the ReLU TwELL in one launch (n_tiles <= kFusedFillMaxTiles):
// every block computes the tile widths K[t] (max nnz over the tile's rows,
// read from L2) and their compact offsets in shared memory, then fills the
// slots of its own rows_per_block rows as k_fill_staged_relu does (a warp per
// row). Block 0 writes K[] and off[] and reports a capacity overflow; every
// block sees the same total and skips the fill then. This replaces the
// single-block k_tile_layout and its dependent launch.
constexpr int kFusedFillMaxTiles = 2048;

__global__ void __launch_bounds__(1024) k_layout_fill_relu(const uint32_t* __restrict__ stage,
                                                           const int32_t* __restrict__ stage_cnt, int NB, int BN,
                                                           int stride, TwellView tw, int rows_per_block,
                                                           int32_t* status)
{
    __shared__ int s_K[kFusedFillMaxTiles];
    __shared__ long long s_off[kFusedFillMaxTiles + 1];
    __shared__ long long s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (has_error(status)) return;
    const int nt = tw.n_tiles;
    for (int t = warp; t < nt; t += 32) {
        const int r0 = t * tw.T, rows = min(tw.T, tw.M - r0);
        int mx = 0;
        for (int i = lane; i < rows; i += 32) mx = max(mx, tw.nnz[r0 + i]);
        mx = warp_max_i(mx);
        if (lane == 0) s_K[t] = mx;
    }
    __syncthreads();
    // exclusive prefix of rows(t) * K[t]: thread i sums tiles 2i, 2i + 1
    long long v0 = 0, v1 = 0;
    const int t0 = 2 * tid;
    if (t0 < nt) v0 = (long long)min(tw.T, tw.M - t0 * tw.T) * s_K[t0];
    if (t0 + 1 < nt) v1 = (long long)min(tw.T, tw.M - (t0 + 1) * tw.T) * s_K[t0 + 1];
    long long incl = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    long long before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    const long long excl = before + incl - (v0 + v1);
    if (t0 < nt) s_off[t0] = excl;
    if (t0 + 1 < nt) s_off[t0 + 1] = excl + v0;
    if (tid == 0) {
        long long total = 0;
        for (int w = 0; w < 32; ++w) total += s_warp[w];
        s_off[nt] = total;
    }
    __syncthreads();
    const bool over = s_off[nt] > tw.cap;
    if (blockIdx.x == 0) {
        for (int t = tid; t <= nt; t += blockDim.x) {
            if (t < nt) tw.K[t] = s_K[t];
            tw.off[t] = s_off[t];
        }
        if (tid == 0 && over) set_error(status, TWELL_ERR_CAPACITY);
    }
    if (over) return;  // uniform: every block computed the same layout
    const int r_begin = blockIdx.x * rows_per_block, r_end = min(tw.M, r_begin + rows_per_block);
    for (int r = r_begin + warp; r < r_end; r += 32) {
        const int t = r / tw.T, Kt = s_K[t];
        const int64_t base = s_off[t] + (int64_t)(r - t * tw.T) * Kt;
        fill_row_staged(stage, stage_cnt, NB, NB, BN, stride, tw, r, base, Kt, lane);
    }
}

// Same for the gate staging: entries (global column, fp32 gate value). The
// values go to gval[slot]; val[] is written later by the gated-up kernel.
__global__ void k_fill_staged_gate(const uint2* __restrict__ stage, const int32_t* __restrict__ stage_cnt, int NB,
                                   int BM, TwellView tw, float* gval, const int32_t* status)
{
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= tw.M || has_error(status) || over_capacity(tw)) return;
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    int pos = 0;
    for (int nb0 = 0; nb0 < NB; nb0 += 32) {
        const int nb = nb0 + lane;
        const int c = nb < NB ? stage_cnt[(size_t)r * NB + nb] : 0;
        const int incl = warp_incl_scan(c, lane);
        const int64_t p = base + pos + (incl - c);
        const uint2* src = stage + ((size_t)r * NB + nb) * BM;
        for (int e = 0; e < c; ++e) {
            const uint2 w = src[e];
            tw.idx[p + e] = (int)w.x;
            gval[p + e] = __uint_as_float(w.y);
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    for (int k = pos + lane; k < Kt; k += 32) {
        tw.idx[base + k] = -1;
        tw.val[base + k] = 0;
        gval[base + k] = 0.f;
    }
}

// ------------------------------------------------- hybrid (ELL + dense) --
//
// "Sparser, Faster, Lighter Transformer Language Models", Resumo Técnico §2,
// "Formato Híbrido para Treinamento": rows are partitioned dynamically; rows
// within the ELL capacity stay in the compact format, rows with more nonzeros
// (overflow) go to a dense backup matrix. Here: a row with nnz > C is an
// overflow row. Its TwELL row is empty (nnz 0, so the TwELL kernels need no
// change) and its whole hidden row is written densely to the next row of the
// overflow block, rows in ascending order.

// One block of 1024 threads: overflow flags (nnz[r] > C), their ascending
// positions, the row list and count; nnz of overflow rows set to 0 so that the
// tile layout that follows sizes the TwELL on the remaining rows only.
__global__ void __launch_bounds__(1024) k_overflow_rows(TwellView tw, int C, int cap_rows, int32_t* __restrict__ ov_pos,
                                                        int32_t* __restrict__ ov_rows, int32_t* __restrict__ n_rows,
                                                        int32_t* status)
{
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (has_error(status)) return;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int r0 = 0; r0 < tw.M; r0 += 1024) {
        const int r = r0 + tid;
        const bool in = r < tw.M;
        const int n = in ? tw.nnz[r] : 0;
        const int f = (in && n > C) ? 1 : 0;
        const int incl = warp_incl_scan(f, lane);
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int w = s_warp[lane];
            s_warp[lane] = warp_incl_scan(w, lane);
        }
        __syncthreads();
        const int pos = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + incl - f;
        if (in) {
            ov_pos[r] = f ? pos : -1;
            if (f) {
                if (pos < cap_rows) ov_rows[pos] = r;
                tw.nnz[r] = 0;
            }
        }
        __syncthreads();
        if (tid == 0) s_carry += s_warp[31];
        __syncthreads();
    }
    if (tid == 0) {
        *n_rows = min(s_carry, cap_rows);
        if (s_carry > cap_rows) set_error(status, TWELL_ERR_CAPACITY);
    }
}

// Block i writes overflow row i: zeros over all F columns, then the row's
// staged entries at their columns. F % 8 == 0 (16-byte rows of 8 bf16).
__global__ void __launch_bounds__(256) k_overflow_dense(const uint32_t* __restrict__ stage,
                                                        const int32_t* __restrict__ stage_cnt, int NB, int BN, int F,
                                                        const int32_t* __restrict__ ov_rows,
                                                        const int32_t* __restrict__ n_rows, uint16_t* __restrict__ dense,
                                                        const int32_t* status)
{
    const int i = blockIdx.x;
    if (has_error(status) || i >= *n_rows) return;
    const int r = ov_rows[i];
    uint16_t* drow = dense + (size_t)i * F;
    for (int c = threadIdx.x * 8; c < F; c += blockDim.x * 8)
        *reinterpret_cast<uint4*>(drow + c) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int nb = warp; nb < NB; nb += nw) {
        const int c = stage_cnt[(size_t)r * NB + nb];
        const uint32_t* src = stage + ((size_t)r * NB + nb) * BN;
        for (int e = lane; e < c; e += 32) {
            const uint32_t w = src[e];
            drow[nb * BN + (int)(w & 0xffffu)] = (uint16_t)(w >> 16);
        }
    }
}

// Layout and fill without a separate layout pass, for small problems (M * NB <= kSmallFillMax
// staging blocks, M <= 1024): the per-(row, block) counts go to shared memory
// with one coalesced load, rows' nnz and block prefixes, tile widths and offsets
// are computed there, and every thread then copies the entries of its (row,
// block) pairs and writes padding. This replaces k_tile_layout + the warp-per-row
// fill, whose dependent global round trips dominate at decode sizes.
constexpr int kSmallFillMax = 8192;

template <typename Entry>
__global__ void __launch_bounds__(1024) k_layout_fill_small(const Entry* __restrict__ stage,
                                                            const int32_t* __restrict__ stage_cnt, int NB, int BW,
                                                            int stride, TwellView tw, float* gval, int32_t* status)
{
    __shared__ int s_cnt[kSmallFillMax];  // per (row, block): count, then exclusive prefix within the row
    __shared__ int s_nnz[1024];
    __shared__ long long s_off[1025];
    __shared__ int s_K[1024];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (has_error(status)) return;
    const int M = tw.M, total = M * NB;
    for (int i = tid; i < total; i += 1024) s_cnt[i] = stage_cnt[i];
    __syncthreads();
    // per-row exclusive prefix over blocks and nnz (a warp per row)
    for (int r = warp; r < M; r += 32) {
        int carry = 0;
        for (int nb0 = 0; nb0 < NB; nb0 += 32) {
            const int nb = nb0 + lane;
            const int c = nb < NB ? s_cnt[r * NB + nb] : 0;
            const int incl = warp_incl_scan(c, lane);
            if (nb < NB) s_cnt[r * NB + nb] = carry + incl - c;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            s_nnz[r] = carry;
            if (blockIdx.x == 0) tw.nnz[r] = carry;
        }
    }
    __syncthreads();
    // tile widths and offsets (one thread; at most 1024 tiles of at most 1024 rows in total).
    // Every block computes the same layout; block 0 writes it out.
    if (tid == 0) {
        long long off = 0;
        for (int t = 0; t < tw.n_tiles; ++t) {
            const int r0 = t * tw.T, rows = min(tw.T, M - r0);
            int mx = 0;
            for (int i = 0; i < rows; ++i) mx = max(mx, s_nnz[r0 + i]);
            s_K[t] = mx;
            s_off[t] = off;
            if (blockIdx.x == 0) {
                tw.K[t] = mx;
                tw.off[t] = off;
            }
            off += (long long)rows * mx;
        }
        s_off[tw.n_tiles] = off;
        if (blockIdx.x == 0) {
            tw.off[tw.n_tiles] = off;
            if (off > tw.cap) set_error(status, TWELL_ERR_CAPACITY);
        }
    }
    __syncthreads();
    if (s_off[tw.n_tiles] > tw.cap) return;
    // entries: (row, block) pairs spread over the blocks
    for (int i = blockIdx.x * 1024 + tid; i < total; i += gridDim.x * 1024) {
        const int r = i / NB, nb = i - r * NB;
        const int t = r / tw.T;
        const long long base = s_off[t] + (long long)(r - t * tw.T) * s_K[t] + s_cnt[i];
        const int c = stage_cnt[i];
        const Entry* src = stage + (size_t)i * stride;
        for (int e = 0; e < c; ++e) {
            const Entry w = src[e];
            if constexpr (sizeof(Entry) == 8) {
                tw.idx[base + e] = (int)w.x;
                gval[base + e] = __uint_as_float(w.y);
            } else {
                tw.idx[base + e] = nb * BW + (int)(w & 0xffffu);
                tw.val[base + e] = (uint16_t)(w >> 16);
            }
        }
    }
    // padding: rows spread over the blocks' warps
    for (int r = blockIdx.x * 32 + warp; r < M; r += gridDim.x * 32) {
        const int t = r / tw.T;
        const long long base = s_off[t] + (long long)(r - t * tw.T) * s_K[t];
        for (int k = s_nnz[r] + lane; k < s_K[t]; k += 32) {
            tw.idx[base + k] = -1;
            tw.val[base + k] = 0;
            if constexpr (sizeof(Entry) == 8) gval[base + k] = 0.f;
        }
    }
}

// Gated up products, one warp per stored slot over a persistent grid:
// val[slot] = bf16(relu(g) * (x[r] . W_up[j])), g = gval[slot]. Slots are
// visited in tile order; a slot's row and position come from off[] / K[].
__global__ void __launch_bounds__(kWarps * 32) k_gated_up_slots(TwellView tw, const uint16_t* __restrict__ x,
                                                                const uint16_t* __restrict__ W_up, int d,
                                                                const float* __restrict__ gval,
                                                                const int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * kWarps;
    if (has_error(status) || over_capacity(tw)) return;
    const long long S = tw.off[tw.n_tiles];
    int t = 0;
    for (long long s = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); s < S; s += nwarps) {
        while (tw.off[t + 1] <= s) ++t;  // slots only grow, so the tile index only advances
        const int Kt = tw.K[t];
        const long long rel = s - tw.off[t];
        const int i = (int)(rel / Kt), k = (int)(rel - (long long)i * Kt);
        const int r = t * tw.T + i;
        if (k >= tw.nnz[r]) continue;  // padding
        const int j = tw.idx[s];
        const uint16_t* xr = x + (size_t)r * d + lane * 8;
        const uint16_t* wr = W_up + (size_t)j * d + lane * 8;
        float acc = 0.f;
        // 8 chunks of 256 columns in flight at a time
        for (int c0 = 0; c0 < d; c0 += 8 * 256) {
            uint4 a[8], w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + q * 256;
                const bool ok = c + lane * 8 < d;
                a[q] = ok ? ldg16(xr + c) : make_uint4(0, 0, 0, 0);
                w[q] = ok ? ldg16(wr + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) acc += dot8_bf16(a[q], w[q]);
        }
        acc = warp_sum_f(acc);
        if (lane == 0) tw.val[s] = f32_to_bf16_bits(fmaxf(gval[s], 0.f) * acc);
    }
}

// -------------------------------------------------------- sparse products --

// y[r, cols] = sum_k v[r,k] W[idx[r,k], cols] for one (row, 256-column group)
// task. SPLIT warps share a task, each taking a contiguous share of the row's
// entries; their partial sums are added in warp order through shared memory.
template <int SPLIT>
__global__ void __launch_bounds__((SPLIT > kWarps ? SPLIT : kWarps) * 32) k_spmm_rows(
    TwellView tw, const float* __restrict__ vals_f32, const uint16_t* __restrict__ W, int d,
    uint16_t* __restrict__ y, const int32_t* status)
{
    constexpr int BW = SPLIT > kWarps ? SPLIT : kWarps;  // warps per block
    __shared__ float red[SPLIT > 1 ? BW : 1][SPLIT > 1 ? 256 : 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = (d + 255) >> 8;
    const int64_t task = (int64_t)blockIdx.x * (BW / SPLIT) + warp / SPLIT;
    const int sub = warp % SPLIT;
    if (has_error(status) || over_capacity(tw)) return;  // uniform across the block
    const int r = (int)(task / ngroups), g = (int)(task % ngroups);
    const bool task_ok = r < tw.M;
    const int c0 = g * 256 + lane * 8;
    const bool col_ok = task_ok && c0 < d;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    if (task_ok) {
        int Kt;
        const int64_t base = row_base(tw, r, &Kt);
        const int n = tw.nnz[r];
        const int per = (n + SPLIT - 1) / SPLIT;
        const int kb = min(n, sub * per), ke = min(n, kb + per);
        const uint16_t* Wc = W + c0;
        for (int k0 = kb; k0 < ke; k0 += 32) {
            const int m = min(32, ke - k0);
            int jl = 0;
            float vl = 0.f;
            uint32_t vb = 0;
            if (lane < m) {
                jl = tw.idx[base + k0 + lane];
                if (vals_f32)
                    vl = vals_f32[base + k0 + lane];
                else
                    vb = tw.val[base + k0 + lane];
            }
            int u = 0;
            for (; u + 4 <= m; u += 4) {
                uint4 w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int jj = __shfl_sync(0xffffffffu, jl, u + q);
                    w[q] = col_ok ? ldg16(Wc + (size_t)jj * d) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (vals_f32)
                        fma8(acc, __shfl_sync(0xffffffffu, vl, u + q), w[q]);
                    else
                        fma8_bf16(acc, __shfl_sync(0xffffffffu, vb, u + q), w[q]);
                }
            }
            for (; u < m; ++u) {
                const int jj = __shfl_sync(0xffffffffu, jl, u);
                const uint4 w = col_ok ? ldg16(Wc + (size_t)jj * d) : make_uint4(0, 0, 0, 0);
                if (vals_f32)
                    fma8(acc, __shfl_sync(0xffffffffu, vl, u), w);
                else
                    fma8_bf16(acc, __shfl_sync(0xffffffffu, vb, u), w);
            }
        }
    }
    if constexpr (SPLIT > 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
        __syncthreads();
        if (sub != 0) return;
        for (int s2 = 1; s2 < SPLIT; ++s2) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += red[warp + s2][lane * 8 + e];
        }
    }
    if (col_ok) {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(y + (size_t)r * d + c0) = o;
    }
}

// acc[0..7] += v * (8 bf16 in w), fp32 v: the widened pairs go through the
// packed fma.rn.f32x2 (two fp32 FMAs per instruction, each rounded like fmaf),
// which issues half as many FMA instructions as fma8.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float x0, float x1, float v)
{
    asm("{\n.reg .b64 acc, xx, vv;\n"
        "mov.b64 acc, {%0, %1};\n"
        "mov.b64 xx, {%2, %3};\n"
        "mov.b64 vv, {%4, %4};\n"
        "fma.rn.f32x2 acc, xx, vv, acc;\n"
        "mov.b64 {%0, %1}, acc;\n}\n"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1), "f"(v));
}

__device__ __forceinline__ void fma8x2(float (&acc)[8], float v, const uint4& w)
{
    ffma2(acc[0], acc[1], bf16_lo(w.x), bf16_hi(w.x), v);
    ffma2(acc[2], acc[3], bf16_lo(w.y), bf16_hi(w.y), v);
    ffma2(acc[4], acc[5], bf16_lo(w.z), bf16_hi(w.z), v);
    ffma2(acc[6], acc[7], bf16_lo(w.w), bf16_hi(w.w), v);
}

// Where a gather's entry lists come from:
//   SRC_TWELL  task row r of the TwELL: its stored slots, indices = columns j,
//              values = val (bf16) or an fp32 array indexed by slot;
//   SRC_CSC    task unit j of the column lists: entries colptr[j] ..
//              colptr[j+1], indices = rows r (crow), values = cval (bf16 h) or
//              cdpre (fp32).
enum GatherSrc { SRC_TWELL = 0, SRC_CSC = 1 };

struct GatherArgs {
    TwellView tw;
    const int32_t* colptr;  // SRC_CSC
    const int32_t* eidx;    // SRC_CSC: entry indices (crow)
    const uint16_t* vb;     // bf16 values (TwELL val or cval), or null
    const float* vf;        // fp32 values (by slot or by list position), or null
    const uint16_t* W;      // gathered matrix, rows of d bf16
    int d;
    uint16_t* out_bf16;     // output rows of d: bf16 ...
    float* out_f32;         //   ... or fp32
    float* rowsum;          // SRC_CSC with fp32 values: sum of each list's values (db), or null
};

// out[t, :] = sum over task t's entries e of v_e W[i_e, :], fp32 accumulation
// in entry order. Column-group-major: warp task (column group g of CH x 256
// columns, task row t) with index g * ntasks + t, so that at any time the grid
// works through one group's slice of W (rows x CH x 256 bf16, 8 or 16 MB at
// 16384 rows) and that slice stays in L2, whatever the size of W. Lane l holds
// columns 256 CH g + 256 c + 8 l .. +7 of chunk c; entries come 4 at a time
// (4 CH 128-bit loads in flight per lane).
// Small blocks balance the last wave: 4 warps finish 1-3 % sooner than 8 at
// the training size, 2 warps another ~1 % (weight gradients). 28 warps per SM
// (72 registers, a few bytes spilled on the tail path) instead of the 24 that
// 80 registers allow keep more rows' loads in flight: 3-4 % faster; 32 warps
// (64 registers) spill in the main loop and are slower.
constexpr int kGatherWarps = 2;

template <int CH, int SRC>
__global__ void __launch_bounds__(kGatherWarps * 32, 14) k_gather(GatherArgs ga, const int32_t* status)
{
    constexpr int GW = 256 * CH;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t task = (int64_t)blockIdx.x * kGatherWarps + warp;
    const TwellView& tw = ga.tw;
    if (has_error(status) || over_capacity(tw)) return;  // uniform across the block
    const int ntasks = SRC == SRC_TWELL ? tw.M : tw.F;
    const int g = (int)(task / ntasks), t = (int)(task % ntasks);
    const int d = ga.d;
    if (g * GW >= d) return;
    int c0[CH];
    bool ok[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        c0[c] = g * GW + c * 256 + lane * 8;
        ok[c] = c0[c] < d;
    }
    float acc[CH][8];
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;
    int64_t base;
    int n;
    const int32_t* eidx;
    if (SRC == SRC_TWELL) {
        int Kt;
        base = row_base(tw, t, &Kt);
        n = tw.nnz[t];
        eidx = tw.idx;
    } else {
        base = ga.colptr[t];
        n = ga.colptr[t + 1] - (int)base;
        eidx = ga.eidx;
    }
    const bool f32v = ga.vf != nullptr;
    const uint16_t* W = ga.W;
    float vsum = 0.f;
    for (int k0 = 0; k0 < n; k0 += 32) {
        const int m = min(32, n - k0);
        int jl = 0;
        float vl = 0.f;
        uint32_t vbl = 0;
        if (lane < m) {
            jl = eidx[base + k0 + lane];
            if (f32v)
                vl = ga.vf[base + k0 + lane];
            else
                vbl = ga.vb[base + k0 + lane];
        }
        vsum += vl;
        int u = 0;
        for (; u + 4 <= m; u += 4) {
            uint4 w[4][CH];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jj = __shfl_sync(0xffffffffu, jl, u + q);
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    w[q][c] = ok[c] ? ldg16(W + (size_t)jj * d + c0[c]) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (f32v) {
                    const float v = __shfl_sync(0xffffffffu, vl, u + q);
#pragma unroll
                    for (int c = 0; c < CH; ++c) fma8x2(acc[c], v, w[q][c]);
                } else {
                    const uint32_t v = __shfl_sync(0xffffffffu, vbl, u + q);
#pragma unroll
                    for (int c = 0; c < CH; ++c) fma8_bf16(acc[c], v, w[q][c]);
                }
            }
        }
        for (; u < m; ++u) {
            const int jj = __shfl_sync(0xffffffffu, jl, u);
            uint4 w[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c) w[c] = ok[c] ? ldg16(W + (size_t)jj * d + c0[c]) : make_uint4(0, 0, 0, 0);
            if (f32v) {
                const float v = __shfl_sync(0xffffffffu, vl, u);
#pragma unroll
                for (int c = 0; c < CH; ++c) fma8x2(acc[c], v, w[c]);
            } else {
                const uint32_t v = __shfl_sync(0xffffffffu, vbl, u);
#pragma unroll
                for (int c = 0; c < CH; ++c) fma8_bf16(acc[c], v, w[c]);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        if (!ok[c]) continue;
        if (ga.out_f32) {
            float4* o = reinterpret_cast<float4*>(ga.out_f32 + (size_t)t * d + c0[c]);
            o[0] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
            o[1] = make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
        } else {
            uint4 o;
            o.x = pack_bf16x2(acc[c][0], acc[c][1]);
            o.y = pack_bf16x2(acc[c][2], acc[c][3]);
            o.z = pack_bf16x2(acc[c][4], acc[c][5]);
            o.w = pack_bf16x2(acc[c][6], acc[c][7]);
            *reinterpret_cast<uint4*>(ga.out_bf16 + (size_t)t * d + c0[c]) = o;
        }
    }
    if (SRC == SRC_CSC && ga.rowsum && g == 0) {
        vsum = warp_sum_f(vsum);  // lanes' partial sums in a fixed butterfly order
        if (lane == 0) ga.rowsum[t] = vsum;
    }
}

// Backward SDDMM over column slices of NCH x 256 columns: warp task (slice s,
// row r), task = s * M + r (slice-major, so one slice of W_down stays in L2).
// The lane holds its 8 NCH columns of dy[r] in registers; the row's entries
// go in half-batches of 16, two at a time (2 NCH 128-bit loads in flight per
// lane), each lane forming its columns' share of both dot products;
// transpose_reduce16 then leaves entry u's slice sum in lane u, written to
// part[s * cap + slot]. k_sddmm_combine_scatter adds the slices in order.
// Blocks of 4 warps, seven per SM (72 registers): against 32-entry batches in
// 8-warp blocks at 80 registers, 6 % faster at the training size.
constexpr int kSddmmWarps = 4;

template <int NCH>
__global__ void __launch_bounds__(kSddmmWarps * 32, 7)
    k_sddmm_slices(TwellView tw, const uint16_t* __restrict__ dy, const uint16_t* __restrict__ W, int d, int nslices,
                   float* __restrict__ part, const int32_t* status)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t task = (int64_t)blockIdx.x * kSddmmWarps + warp;
    if (has_error(status) || over_capacity(tw)) return;  // uniform across the block
    const int sl = (int)(task / tw.M), r = (int)(task % tw.M);
    if (sl >= nslices) return;
    int col[NCH];
    bool ok[NCH];
    uint4 a[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        col[c] = (sl * NCH + c) * 256 + lane * 8;
        ok[c] = col[c] < d;
        a[c] = ok[c] ? ldg16(dy + (size_t)r * d + col[c]) : make_uint4(0, 0, 0, 0);
    }
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    const int n = tw.nnz[r];
    float* out = part + (size_t)sl * (size_t)tw.cap + base;
    for (int k0 = 0; k0 < n; k0 += 32) {
        const int m = min(32, n - k0);
        const int jl = tw.idx[base + k0 + (lane < m ? lane : 0)];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int mh = m - 16 * h;  // entries of this half (warp-uniform)
            if (mh <= 0) break;
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
                if (u < mh) {
                    const int e = 16 * h + u;
                    const int j0 = __shfl_sync(0xffffffffu, jl, e);
                    const int j1 = __shfl_sync(0xffffffffu, jl, e + 1 < m ? e + 1 : e);
                    uint4 w0[NCH], w1[NCH];
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        w0[c] = ok[c] ? ldg16(W + (size_t)j0 * d + col[c]) : make_uint4(0, 0, 0, 0);
                        w1[c] = ok[c] ? ldg16(W + (size_t)j1 * d + col[c]) : make_uint4(0, 0, 0, 0);
                    }
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        s0 += dot8_bf16(a[c], w0[c]);
                        s1 += dot8_bf16(a[c], w1[c]);
                    }
                    v[u] = s0;
                    v[u + 1] = u + 1 < mh ? s1 : 0.f;
                } else {
                    v[u] = 0.f;
                    v[u + 1] = 0.f;
                }
            }
            transpose_reduce16(v, lane);
            if (lane < min(16, mh)) out[k0 + 16 * h + lane] = v[0];
        }
    }
}

// Gated up products, row-parallel: for stored entry (r, k) with column j,
// s = A[r] . W[j] and val[slot] = bf16(relu(g) * s), g = gval[slot]. WPR warps
// share a row, entry k going to warp k % WPR; a row's A slice stays in
// registers (NCH chunks of 256 columns, 8 per lane).
template <int NCH>
__global__ void __launch_bounds__(kWarps * 32) k_row_dots(TwellView tw, const uint16_t* __restrict__ A,
                                                          const uint16_t* __restrict__ W, int d, int wpr,
                                                          const float* __restrict__ gval, const int32_t* status)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * (kWarps / wpr) + warp / wpr;
    const int sub = warp % wpr;
    if (r >= tw.M || has_error(status) || over_capacity(tw)) return;
    uint4 a[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const int c = ch * 256 + lane * 8;
        a[ch] = c < d ? ldg16(A + (size_t)r * d + c) : make_uint4(0, 0, 0, 0);
    }
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    const int n = tw.nnz[r];
    // entries of this warp: k = sub + wpr * q, q = 0, 1, ...
    const int nq = n > sub ? (n - sub + wpr - 1) / wpr : 0;
    for (int q0 = 0; q0 < nq; q0 += 32) {
        const int m = min(32, nq - q0);
        const int kl = sub + wpr * (q0 + lane);
        const int jl = lane < m ? tw.idx[base + kl] : 0;
        float res = 0.f;
        int u = 0;
        for (; u + 2 <= m; u += 2) {
            const int ja = __shfl_sync(0xffffffffu, jl, u), jb = __shfl_sync(0xffffffffu, jl, u + 1);
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                const int c = ch * 256 + lane * 8;
                if (c < d) {
                    const uint4 wa = ldg16(W + (size_t)ja * d + c);
                    const uint4 wb = ldg16(W + (size_t)jb * d + c);
                    sa += dot8(a[ch], wa);
                    sb += dot8(a[ch], wb);
                }
            }
            sa = warp_sum_f(sa);
            sb = warp_sum_f(sb);
            if (lane == u) res = sa;
            if (lane == u + 1) res = sb;
        }
        if (u < m) {
            const int ja = __shfl_sync(0xffffffffu, jl, u);
            float sa = 0.f;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                const int c = ch * 256 + lane * 8;
                if (c < d) sa += dot8(a[ch], ldg16(W + (size_t)ja * d + c));
            }
            sa = warp_sum_f(sa);
            if (lane == u) res = sa;
        }
        if (lane < m) {
            const int64_t s = base + kl;
            tw.val[s] = f32_to_bf16_bits(fmaxf(gval[s], 0.f) * res);
        }
    }
}

// ------------------------------------------------------------- CSC build ----
//
// Column lists of the stored entries, rows ascending inside each column, built
// without atomics on global memory: row blocks of 64 rows record, per column,
// a 64-bit mask of the rows that hold it; a column-wise scan of the mask
// popcounts gives each (block, column) its start, and an entry's position is
// colptr[j] + start[b][j] + popcount of the mask bits below its row.

constexpr int kCscRows = 64;

__global__ void __launch_bounds__(256) k_csc_mask(TwellView tw, int col_range,
                                                  unsigned long long* __restrict__ masks, const int32_t* status)
{
    extern __shared__ unsigned long long s_mask[];  // [col_range]
    const int b = blockIdx.x;
    const int jlo = blockIdx.y * col_range, jhi = min(tw.F, jlo + col_range);
    if (has_error(status)) return;
    for (int j = threadIdx.x; j < jhi - jlo; j += blockDim.x) s_mask[j] = 0ull;
    __syncthreads();
    const int r0 = b * kCscRows, r1 = min(tw.M, r0 + kCscRows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = r0 + warp; r < r1; r += blockDim.x >> 5) {
        int Kt;
        const int64_t base = row_base(tw, r, &Kt);
        const int n = tw.nnz[r];
        const unsigned long long bit = 1ull << (r - r0);
        for (int k = lane; k < n; k += 32) {
            const int j = tw.idx[base + k];
            if (j >= jlo && j < jhi) atomicOr(&s_mask[j - jlo], bit);
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < jhi - jlo; j += blockDim.x) masks[(size_t)b * tw.F + jlo + j] = s_mask[j];
}

// 32 columns per block: start[b][j] = sum over blocks b' < b of popc(mask[b'][j]);
// colcnt[j] = total over all blocks.
__global__ void __launch_bounds__(1024) k_csc_colscan(const unsigned long long* __restrict__ masks, int row_blocks,
                                                      int F, int32_t* __restrict__ start, int32_t* __restrict__ colcnt,
                                                      const int32_t* status)
{
    __shared__ int s_cnt[32][33];
    __shared__ int s_carry[32];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 32
    const int j = blockIdx.x * 32 + tx;
    if (has_error(status)) return;
    if (ty == 0) s_carry[tx] = 0;
    __syncthreads();
    for (int b0 = 0; b0 < row_blocks; b0 += 32) {
        const int b = b0 + ty;
        s_cnt[ty][tx] = (b < row_blocks && j < F) ? __popcll(masks[(size_t)b * F + j]) : 0;
        __syncthreads();
        // warp ty scans column (blockIdx.x*32 + ty) over the 32 blocks (lane = block)
        const int v = s_cnt[tx][ty];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (tx >= o) incl += n;
        }
        const int jj = blockIdx.x * 32 + ty;
        const int bb = b0 + tx;
        const int carry = s_carry[ty];
        if (jj < F && bb < row_blocks) start[(size_t)bb * F + jj] = carry + incl - v;
        __syncthreads();
        if (tx == 31) s_carry[ty] = carry + incl;
        __syncthreads();
    }
    if (ty == 0 && j < F) colcnt[j] = s_carry[tx];
}

// Single block: ptr[0..n] = exclusive prefix of cnt[0..n). Each thread scans
// a run of consecutive elements; the run totals are scanned across the block.
__global__ void __launch_bounds__(1024) k_scan_i32(const int32_t* __restrict__ cnt, int n, int32_t* __restrict__ ptr,
                                                   const int32_t* status)
{
    __shared__ int s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (has_error(status)) return;
    const int per = (n + 1023) / 1024;
    const int i0 = tid * per;
    int local = 0;
    for (int k = 0; k < per; ++k)
        if (i0 + k < n) local += cnt[i0 + k];
    const int incl = warp_incl_scan(local, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) s_warp[lane] = warp_incl_scan(s_warp[lane], lane);
    __syncthreads();
    int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int k = 0; k < per; ++k) {
        if (i0 + k < n) {
            ptr[i0 + k] = run;
            run += cnt[i0 + k];
        }
    }
    if (tid == 1023) ptr[n] = run;
}

// The SDDMM's last step and the column lists' scatter in one pass, a warp per
// row: dpre[slot] = (part[0][slot] + part[1][slot] + ...) + l1 on the stored
// slots of row r (slices added in order), 0 on its padding; and each stored
// entry goes to its place in its column's list with its row, its h and its
// dpre, so that the weight-gradient gathers read them with coalesced loads.
// An entry's place is colptr[j] + start[b][j] + the popcount of the mask
// bits below its row.
__global__ void __launch_bounds__(kWarps * 32) k_sddmm_combine_scatter(
    TwellView tw, const float* __restrict__ part, int nslices, float l1, float* __restrict__ dpre,
    const unsigned long long* __restrict__ masks, const int32_t* __restrict__ start,
    const int32_t* __restrict__ colptr, int32_t* __restrict__ crow, uint16_t* __restrict__ cval,
    float* __restrict__ cdpre, const int32_t* status)
{
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= tw.M || has_error(status) || over_capacity(tw)) return;
    int Kt;
    const int64_t base = row_base(tw, r, &Kt);
    const int n = tw.nnz[r];
    const int b = r / kCscRows;
    const unsigned long long below = (1ull << (r - b * kCscRows)) - 1ull;
    for (int k = lane; k < Kt; k += 32) {
        const int64_t slot = base + k;
        float v = 0.f;
        if (k < n) {
            v = part[slot];
            for (int sl = 1; sl < nslices; ++sl) v += part[(size_t)sl * (size_t)tw.cap + slot];
            v += l1;
            const int j = tw.idx[slot];
            const size_t bj = (size_t)b * tw.F + j;
            const int pos = colptr[j] + start[bj] + __popcll(masks[bj] & below);
            crow[pos] = r;
            cval[pos] = tw.val[slot];
            cdpre[pos] = v;
        }
        dpre[slot] = v;
    }
}


}  // namespace

// ------------------------------------------------------------- launchers ----

cudaError_t launch_count_dense(const uint16_t* h, int ldh, const TwellView& tw, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_count_dense<<<grid_for_warps(tw.M), kWarps * 32, 0, s>>>(h, ldh, tw, status);
    return cudaGetLastError();
}

cudaError_t launch_tile_layout(const TwellView& tw, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_tile_layout<<<1, 1024, 0, s>>>(tw, status);
    return cudaGetLastError();
}

cudaError_t launch_fill_dense(const uint16_t* h, int ldh, const TwellView& tw, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_fill_dense<<<grid_for_warps(tw.M), kWarps * 32, 0, s>>>(h, ldh, tw, status);
    return cudaGetLastError();
}

cudaError_t launch_fill_staged_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int stride,
                                    const TwellView& tw, const int32_t* ov_pos, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_fill_staged_relu<<<grid_for_warps(tw.M), kWarps * 32, 0, s>>>(stage, stage_cnt, NB, BN, stride, tw, ov_pos,
                                                                     status);
    return cudaGetLastError();
}

bool fused_fill_ok(int n_tiles) { return n_tiles <= kFusedFillMaxTiles; }

cudaError_t launch_layout_fill_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int stride,
                                    const TwellView& tw, int sm_count, int32_t* status, cudaStream_t s)
{
    if (!fused_fill_ok(tw.n_tiles)) return cudaErrorInvalidValue;
    // one block per SM, each filling a contiguous share of the rows
    const int blocks = sm_count > 0 ? sm_count : 1;
    const int rows_per_block = (tw.M + blocks - 1) / blocks;
    const int grid = (tw.M + rows_per_block - 1) / rows_per_block;
    count_launches(1);
    k_layout_fill_relu<<<grid, 1024, 0, s>>>(stage, stage_cnt, NB, BN, stride, tw, rows_per_block, status);
    return cudaGetLastError();
}

cudaError_t launch_overflow_rows(const TwellView& tw, int C, int cap_rows, int32_t* ov_pos, int32_t* ov_rows,
                                 int32_t* n_rows, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_overflow_rows<<<1, 1024, 0, s>>>(tw, C, cap_rows, ov_pos, ov_rows, n_rows, status);
    return cudaGetLastError();
}

cudaError_t launch_overflow_dense(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN, int F,
                                  const int32_t* ov_rows, const int32_t* n_rows, int cap_rows, uint16_t* dense,
                                  const int32_t* status, cudaStream_t s)
{
    if (cap_rows <= 0) return cudaSuccess;
    count_launches(1);
    k_overflow_dense<<<cap_rows, 256, 0, s>>>(stage, stage_cnt, NB, BN, F, ov_rows, n_rows, dense, status);
    return cudaGetLastError();
}

cudaError_t launch_fill_staged_gate(const uint2* stage, const int32_t* stage_cnt, int NB, int BM,
                                    const TwellView& tw, float* gval, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    k_fill_staged_gate<<<grid_for_warps(tw.M), kWarps * 32, 0, s>>>(stage, stage_cnt, NB, BM, tw, gval, status);
    return cudaGetLastError();
}

// Column-group-major gather over TwELL rows or column lists (k_gather), two
// 256-column chunks per lane when d has them.
static cudaError_t launch_gather(int src, const GatherArgs& ga, int ntasks, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    const int ch = ga.d > 256 ? 2 : 1;
    const int64_t tasks = (int64_t)ntasks * ((ga.d + 256 * ch - 1) / (256 * ch));
    const unsigned grid = (unsigned)((tasks + kGatherWarps - 1) / kGatherWarps);
    if (ch == 2) {
        if (src == SRC_TWELL)
            k_gather<2, SRC_TWELL><<<grid, kGatherWarps * 32, 0, s>>>(ga, status);
        else
            k_gather<2, SRC_CSC><<<grid, kGatherWarps * 32, 0, s>>>(ga, status);
    } else {
        if (src == SRC_TWELL)
            k_gather<1, SRC_TWELL><<<grid, kGatherWarps * 32, 0, s>>>(ga, status);
        else
            k_gather<1, SRC_CSC><<<grid, kGatherWarps * 32, 0, s>>>(ga, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_spmm_rows(const TwellView& tw, const float* vals_f32, const uint16_t* W, int d, uint16_t* y,
                             int32_t* status, cudaStream_t s)
{
    if (tw.M >= 256) {
        GatherArgs ga{};
        ga.tw = tw;
        ga.vb = vals_f32 ? nullptr : tw.val;
        ga.vf = vals_f32;
        ga.W = W;
        ga.d = d;
        ga.out_bf16 = y;
        return launch_gather(SRC_TWELL, ga, tw.M, status, s);
    }
    // few rows: 16 warps share each (row, 256-column group) task
    const int64_t tasks = (int64_t)tw.M * ((d + 255) / 256);
    count_launches(1);
    k_spmm_rows<16><<<(unsigned)tasks, 16 * 32, 0, s>>>(tw, vals_f32, W, d, y, status);
    return cudaGetLastError();
}

static cudaError_t launch_row_dots(const TwellView& tw, const uint16_t* A, const uint16_t* W, int d,
                                   const float* gval, int32_t* status, cudaStream_t s)
{
    const int nch = (d + 255) / 256;
    const int wpr = tw.M >= 256 ? 1 : kWarps;
    const unsigned grid = (unsigned)(((int64_t)tw.M * wpr + kWarps - 1) / kWarps);
    count_launches(1);
#define TWELL_ROWDOT_CASE(N)                                                                      \
    case N:                                                                                       \
        k_row_dots<N><<<grid, kWarps * 32, 0, s>>>(tw, A, W, d, wpr, gval, status); \
        break;
    switch (nch) {
        TWELL_ROWDOT_CASE(1)
        TWELL_ROWDOT_CASE(2)
        TWELL_ROWDOT_CASE(3)
        TWELL_ROWDOT_CASE(4)
        TWELL_ROWDOT_CASE(5)
        TWELL_ROWDOT_CASE(6)
        TWELL_ROWDOT_CASE(7)
        TWELL_ROWDOT_CASE(8)
        TWELL_ROWDOT_CASE(12)
        TWELL_ROWDOT_CASE(16)
        default:
            if (nch <= 12) {
                k_row_dots<12><<<grid, kWarps * 32, 0, s>>>(tw, A, W, d, wpr, gval, status);
            } else if (nch <= 16) {
                k_row_dots<16><<<grid, kWarps * 32, 0, s>>>(tw, A, W, d, wpr, gval, status);
            } else {
                return cudaErrorInvalidValue;
            }
    }
#undef TWELL_ROWDOT_CASE
    return cudaGetLastError();
}

int sddmm_slices(int d) { return (d + 1023) / 1024; }

cudaError_t launch_sddmm_slices(const TwellView& tw, const uint16_t* dy, const uint16_t* W, int d, float* part,
                                int32_t* status, cudaStream_t s)
{
    // slices of up to four 256-column chunks (1024 columns)
    const int nch_total = (d + 255) / 256;
    const int nch = nch_total < 4 ? nch_total : 4;
    const int nsl = (nch_total + nch - 1) / nch;
    if (nsl > sddmm_slices(d)) return cudaErrorInvalidValue;
    const int64_t tasks = (int64_t)tw.M * nsl;
    count_launches(1);
    switch (nch) {
        case 1: k_sddmm_slices<1><<<(unsigned)((tasks + kSddmmWarps - 1) / kSddmmWarps), kSddmmWarps * 32, 0, s>>>(tw, dy, W, d, nsl, part, status); break;
        case 2: k_sddmm_slices<2><<<(unsigned)((tasks + kSddmmWarps - 1) / kSddmmWarps), kSddmmWarps * 32, 0, s>>>(tw, dy, W, d, nsl, part, status); break;
        case 3: k_sddmm_slices<3><<<(unsigned)((tasks + kSddmmWarps - 1) / kSddmmWarps), kSddmmWarps * 32, 0, s>>>(tw, dy, W, d, nsl, part, status); break;
        default: k_sddmm_slices<4><<<(unsigned)((tasks + kSddmmWarps - 1) / kSddmmWarps), kSddmmWarps * 32, 0, s>>>(tw, dy, W, d, nsl, part, status); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_gated_up(const TwellView& tw, const uint16_t* x, const uint16_t* W_up, int d, const float* gval,
                            int32_t* status, cudaStream_t s)
{
    if (tw.M <= 256 || (d + 255) / 256 > 16) {
        // few rows: spread the slots over the whole GPU, a warp per slot (also
        // for d_model beyond the 16 chunks the row-parallel kernel holds)
        count_launches(1);
        k_gated_up_slots<<<2 * 152, kWarps * 32, 0, s>>>(tw, x, W_up, d, gval, status);
        return cudaGetLastError();
    }
    return launch_row_dots(tw, x, W_up, d, gval, status, s);
}

bool small_fill_ok(int M, int NB) { return M <= 1024 && (long long)M * NB <= kSmallFillMax; }

cudaError_t launch_layout_fill_small_gate(const uint2* stage, const int32_t* stage_cnt, int NB, int BM,
                                          const TwellView& tw, float* gval, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    const int nblk = (tw.M * NB + 1023) / 1024;
    k_layout_fill_small<uint2><<<nblk, 1024, 0, s>>>(stage, stage_cnt, NB, BM, BM, tw, gval, status);
    return cudaGetLastError();
}

cudaError_t launch_layout_fill_small_relu(const uint32_t* stage, const int32_t* stage_cnt, int NB, int BN,
                                          int stride, const TwellView& tw, int32_t* status, cudaStream_t s)
{
    count_launches(1);
    const int nblk = (tw.M * NB + 1023) / 1024;
    k_layout_fill_small<uint32_t><<<nblk, 1024, 0, s>>>(stage, stage_cnt, NB, BN, stride, tw, nullptr, status);
    return cudaGetLastError();
}

void csc_plan(int M, int F, int* row_blocks, int* rows_per_block)
{
    (void)F;
    *rows_per_block = kCscRows;
    *row_blocks = (M + kCscRows - 1) / kCscRows;
}

cudaError_t launch_csc_lists(const TwellView& tw, const CscWork& w, int32_t* status, cudaStream_t s)
{
    // split the columns so that the mask pass has at least two blocks per SM
    int splits = (2 * 152 + w.row_blocks - 1) / w.row_blocks;
    splits = splits < 1 ? 1 : splits;
    int col_range = (tw.F + splits - 1) / splits;
    col_range = (col_range + 31) / 32 * 32;
    if (col_range < 256) col_range = 256;
    if (col_range > 16384) col_range = 16384;  // shared-memory masks: 128 KB at most
    const int ny = (tw.F + col_range - 1) / col_range;
    const size_t smem = (size_t)col_range * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(k_csc_mask, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    count_launches(3);
    k_csc_mask<<<dim3(w.row_blocks, ny), 256, smem, s>>>(tw, col_range, w.masks, status);
    k_csc_colscan<<<(tw.F + 31) / 32, 1024, 0, s>>>(w.masks, w.row_blocks, tw.F, w.start, w.colcnt, status);
    k_scan_i32<<<1, 1024, 0, s>>>(w.colcnt, tw.F, w.colptr, status);
    return cudaGetLastError();
}

cudaError_t launch_sddmm_combine_scatter(const TwellView& tw, int d, const float* part, float l1, float* dpre,
                                         const CscWork& w, int32_t* status, cudaStream_t s)
{
    const int nch_total = (d + 255) / 256;
    const int nch = nch_total < 4 ? nch_total : 4;
    const int nsl = (nch_total + nch - 1) / nch;
    count_launches(1);
    k_sddmm_combine_scatter<<<grid_for_warps(tw.M), kWarps * 32, 0, s>>>(tw, part, nsl, l1, dpre, w.masks, w.start,
                                                                           w.colptr, w.crow, w.cval, w.cdpre, status);
    return cudaGetLastError();
}

cudaError_t launch_wgrad(const TwellView& tw, const CscWork& w, const float* dpre, const uint16_t* x,
                         const uint16_t* dy, int d, float* dW_up, float* dW_down, float* db, int32_t* status,
                         cudaStream_t s)
{
    (void)dpre;  // carried in the column lists
    // dW_down[j] = sum h dy[r] over column j's entries, then dW_up[j] = sum
    // dpre x[r] and db[j] = sum dpre: two gathers of one matrix each (measured
    // faster than one pass gathering x and dy together: 2.77 ms at 16384 x
    // 4096 x 16384, and 3.2-3.8 ms for the unit-major orders)
    GatherArgs ga{};
    ga.tw = tw;
    ga.colptr = w.colptr;
    ga.eidx = w.crow;
    ga.d = d;
    ga.vb = w.cval;
    ga.W = dy;
    ga.out_f32 = dW_down;
    cudaError_t e = launch_gather(SRC_CSC, ga, tw.F, status, s);
    if (e != cudaSuccess) return e;
    ga.vb = nullptr;
    ga.vf = w.cdpre;
    ga.W = x;
    ga.out_f32 = dW_up;
    ga.rowsum = db;
    return launch_gather(SRC_CSC, ga, tw.F, status, s);
}

}  // namespace twell
