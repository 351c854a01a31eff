/*
 * twell_oracle.c — CPU oracle for the TwELL activation-sparse feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this file's library. The product
 * (the CUDA library and its Python binding) never calls it and shares no code,
 * header or table with it.
 *
 * Plain loops, fp64 accumulation, no blocking or reordering beyond what each
 * definition states. Every function cites the passage it follows; the method's
 * source is "Sparser, Faster, Lighter Transformer Language Models" (gist.science
 * summary of arXiv 2603.23198, Resumo Técnico §2 Metodologia). The TwELL layout
 * is stated in full above oracle_twell_layout and oracle_twell_fill.
 *
 * bf16 values travel as uint16 bit patterns. Rounding to bf16 is round to
 * nearest, ties to even, with no flush-to-zero.
 *
 * Pins (tests under tests/test_oracle_*.py): pack/unpack round trip, per-tile
 * width == max row count, compact offsets, T=1 and T>=M special cases, brute
 * force on tiny inputs, exact results on integer-valued inputs, agreement of the
 * dense forward with numpy's matmul, sparse product == dense product, hidden
 * density against the closed form 1 - Phi(-b), and gradients against central
 * finite differences and against torch autograd.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 ---- */

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even from the definition: keep the top 16 bits, look at the
 * 16 dropped bits, round up when they exceed half an ulp or equal half an ulp
 * with an odd kept part. A carry out of the mantissa moves into the exponent,
 * which is the correct overflow to infinity. NaN stays a (quiet) NaN. */
static uint16_t float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

static double bf(uint16_t b) { return (double)bf16_to_float(b); }

/* A bf16 entry of h is active when it is not +0 or -0 (NaN counts as active). */
static int bf16_nonzero(uint16_t b) { return (b & 0x7fffu) != 0u; }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_round_bf16(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16(in[i]);
}

/* ------------------------------------------------------------- forward ---- */

/*
 * Dense forward of the layer for the listed token rows (Resumo Técnico §2,
 * "Técnicas de Treinamento": a ReLU feed-forward layer; "Kernels de Inferência":
 * the gated variant whose gate activations drive the sparse iteration).
 *
 *   ReLU : pre[r,j] = float(sum_k x[r,k] W_up[j,k]) + b[j]   (bias added in fp32)
 *          h[r,j]   = bf16(pre)  if pre > 0, else +0
 *          active   = h != 0
 *   Gated: pre[r,j] = float(sum_k x[r,k] W_gate[j,k]) + b[j]
 *          u[r,j]   = float(sum_k x[r,k] W_up[j,k])
 *          h[r,j]   = bf16(float(pre * u)) if pre > 0, else +0
 *          active   = pre > 0
 *   y[r,c] = sum_j h[r,j] W_down[j,c]   (fp64, returned unrounded)
 *
 * Inputs are bf16 bits; weights are [F, d] row-major. Outputs are indexed by
 * position in `rows` (row i of an output belongs to token rows[i]). pre_out,
 * u_out, active_out, y_out may be NULL.
 */
void oracle_ffn_fwd_rows(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate,
                         const float* b, const uint16_t* W_down, int M, int d, int F,
                         const int32_t* rows, int nrows,
                         float* pre_out, float* u_out, uint16_t* h_out,
                         uint8_t* active_out, double* y_out)
{
    (void)M;
    const uint16_t* W_pre = W_gate ? W_gate : W_up;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const int64_t r = rows[i];
        const uint16_t* xr = x + r * d;
        uint16_t* hr = h_out + (int64_t)i * F;
        for (int j = 0; j < F; ++j) {
            double s = 0.0;
            for (int k = 0; k < d; ++k) s += bf(xr[k]) * bf(W_pre[(int64_t)j * d + k]);
            float pre = (float)s + b[j];
            int active;
            uint16_t h;
            float u = 0.0f;
            if (W_gate) {
                double su = 0.0;
                for (int k = 0; k < d; ++k) su += bf(xr[k]) * bf(W_up[(int64_t)j * d + k]);
                u = (float)su;
                active = pre > 0.0f;
                h = active ? float_to_bf16((float)((double)pre * (double)u)) : (uint16_t)0;
            } else {
                h = pre > 0.0f ? float_to_bf16(pre) : (uint16_t)0;
                active = bf16_nonzero(h);
            }
            hr[j] = h;
            if (pre_out) pre_out[(int64_t)i * F + j] = pre;
            if (u_out) u_out[(int64_t)i * F + j] = u;
            if (active_out) active_out[(int64_t)i * F + j] = (uint8_t)active;
        }
        if (y_out) {
            double* yr = y_out + (int64_t)i * d;
            for (int c = 0; c < d; ++c) yr[c] = 0.0;
            for (int j = 0; j < F; ++j) {
                if (hr[j] == 0) continue; /* a +0 term adds nothing */
                double hv = bf(hr[j]);
                for (int c = 0; c < d; ++c) yr[c] += hv * bf(W_down[(int64_t)j * d + c]);
            }
        }
    }
}

/* ------------------------------------------------------------ TwELL pack -- */

static int entry_active(const uint16_t* h, const uint8_t* active, int64_t at)
{
    return active ? active[at] != 0 : bf16_nonzero(h[at]);
}

/*
 * TwELL layout of h (Resumo Técnico §2, "Formato de Dados TwELL": horizontal
 * tiles, nonzeros and indices aligned locally inside each tile). Tiles are
 * bands of T consecutive token rows spanning all F columns; the last may be
 * short, rows(t) = min(T, M - t*T).
 *   nnz[r]   = number of active entries of row r
 *   K[t]     = max nnz[r] over the rows of tile t
 *   off[0]=0, off[t+1] = off[t] + rows(t) * K[t]
 * Returns off[n_tiles], the total slot count. `active` (may be NULL) overrides
 * the default active set h != 0 (used by the gated layer). ldh = row stride.
 */
int64_t oracle_twell_layout(const uint16_t* h, const uint8_t* active, int M, int F, int ldh,
                            int T, int32_t* nnz, int32_t* K, int64_t* off)
{
    const int n_tiles = (M + T - 1) / T;
    for (int r = 0; r < M; ++r) {
        int c = 0;
        for (int j = 0; j < F; ++j) c += entry_active(h, active, (int64_t)r * ldh + j);
        nnz[r] = c;
    }
    off[0] = 0;
    for (int t = 0; t < n_tiles; ++t) {
        int r0 = t * T;
        int rows = (M - r0 < T) ? (M - r0) : T;
        int kmax = 0;
        for (int i = 0; i < rows; ++i)
            if (nnz[r0 + i] > kmax) kmax = nnz[r0 + i];
        K[t] = kmax;
        off[t + 1] = off[t] + (int64_t)rows * kmax;
    }
    return off[n_tiles];
}

/*
 * TwELL slots: row i of tile t owns slots off[t] + i*K[t] + k (row-major inside
 * the tile),
 * k < K[t]; the first nnz[r] hold the active columns in ascending order with
 * their h values, the rest idx = -1, val = +0.
 */
void oracle_twell_fill(const uint16_t* h, const uint8_t* active, int M, int F, int ldh, int T,
                       const int32_t* K, const int64_t* off, int32_t* idx, uint16_t* val)
{
    const int n_tiles = (M + T - 1) / T;
    for (int t = 0; t < n_tiles; ++t) {
        int r0 = t * T;
        int rows = (M - r0 < T) ? (M - r0) : T;
        for (int i = 0; i < rows; ++i) {
            int64_t base = off[t] + (int64_t)i * K[t];
            int k = 0;
            for (int j = 0; j < F; ++j) {
                int64_t at = (int64_t)(r0 + i) * ldh + j;
                if (entry_active(h, active, at)) {
                    idx[base + k] = j;
                    val[base + k] = h[at];
                    ++k;
                }
            }
            for (; k < K[t]; ++k) {
                idx[base + k] = -1;
                val[base + k] = 0;
            }
        }
    }
}

/*
 * Checks a TwELL against the layout above and writes the dense matrix it encodes.
 * Returns 0 when valid, else a positive code naming the first violation:
 *   1 off[0] != 0     2 off not compact     3 K[t] != max nnz of the tile
 *   4 nnz out of range  5 stored idx out of [0,F)  6 idx not strictly ascending
 *   7 padding slot not (-1, +0)
 */
int oracle_twell_unpack(int M, int F, int T, const int32_t* nnz, const int32_t* K,
                        const int64_t* off, const int32_t* idx, const uint16_t* val,
                        uint16_t* h_out)
{
    const int n_tiles = (M + T - 1) / T;
    if (off[0] != 0) return 1;
    for (int64_t e = 0; e < (int64_t)M * F; ++e) h_out[e] = 0;
    for (int t = 0; t < n_tiles; ++t) {
        int r0 = t * T;
        int rows = (M - r0 < T) ? (M - r0) : T;
        if (off[t + 1] != off[t] + (int64_t)rows * K[t]) return 2;
        int kmax = 0;
        for (int i = 0; i < rows; ++i) {
            int n = nnz[r0 + i];
            if (n < 0 || n > F || n > K[t]) return 4;
            if (n > kmax) kmax = n;
            int64_t base = off[t] + (int64_t)i * K[t];
            for (int k = 0; k < K[t]; ++k) {
                int32_t j = idx[base + k];
                if (k < n) {
                    if (j < 0 || j >= F) return 5;
                    if (k > 0 && j <= idx[base + k - 1]) return 6;
                    h_out[(int64_t)(r0 + i) * F + j] = val[base + k];
                } else if (j != -1 || val[base + k] != 0) {
                    return 7;
                }
            }
        }
        if (kmax != K[t]) return 3;
    }
    return 0;
}

/* ------------------------------------------------------- sparse product --- */

/*
 * Sparse down-projection on the TwELL (Resumo Técnico §2, "Kernels de
 * Inferência": iterate only over the active neurons):
 *   y[r,c] = sum_{k < nnz[r]} val[r,k] * W[idx[r,k], c]   (fp64)
 * W is [F, d] bf16 row-major; y is [M, d] fp64.
 */
void oracle_twell_spmm(int M, int F, int T, const int32_t* nnz, const int32_t* K,
                       const int64_t* off, const int32_t* idx, const uint16_t* val,
                       const uint16_t* W, int d, double* y)
{
    (void)F;
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < M; ++r) {
        int t = r / T;
        int i = r - t * T;
        int64_t base = off[t] + (int64_t)i * K[t];
        double* yr = y + (int64_t)r * d;
        for (int c = 0; c < d; ++c) yr[c] = 0.0;
        for (int k = 0; k < nnz[r]; ++k) {
            double v = bf(val[base + k]);
            const uint16_t* wr = W + (int64_t)idx[base + k] * d;
            for (int c = 0; c < d; ++c) yr[c] += v * bf(wr[c]);
        }
    }
}

/* -------------------------------------------------------------- backward -- */

/*
 * Backward of L = <dy, y> + l1 * sum_{r,j} |h[r,j]| for the ReLU layer
 * y = h W_down, h = relu(x W_up^T + b) (Resumo Técnico §2, "Técnicas de
 * Treinamento": L1 on the ReLU activations; the gradient at h = 0 is taken 0,
 * matching the ReLU mask):
 *   dpre[r,j] = (sum_c dy[r,c] W_down[j,c] + l1) * [h[r,j] != 0]
 *   dx[r,:]   = sum_j dpre[r,j] W_up[j,:]
 *   dW_up[j,:]   = sum_r dpre[r,j] x[r,:]
 *   dW_down[j,:] = sum_r h[r,j] dy[r,:]
 *   db[j]        = sum_r dpre[r,j]
 * All operands fp64 (bf16 inputs are widened exactly by the caller); h is the
 * dense [M, F] hidden matrix the forward produced (h >= 0, so |h|' = 1 on the
 * active set).
 */
void oracle_ffn_bwd_rows(const double* x, const double* W_up, const double* W_down,
                         const double* h, const double* dy, double l1,
                         int M, int d, int F, const int32_t* rows, int nrows,
                         double* dpre_out, double* dx_out)
{
    (void)M; (void)x;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const int64_t r = rows[i];
        double* dp = dpre_out + (int64_t)i * F;
        for (int j = 0; j < F; ++j) {
            if (h[r * F + j] == 0.0) { dp[j] = 0.0; continue; }
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += dy[r * d + c] * W_down[(int64_t)j * d + c];
            dp[j] = s + l1;
        }
        if (dx_out) {
            double* dxr = dx_out + (int64_t)i * d;
            for (int c = 0; c < d; ++c) dxr[c] = 0.0;
            for (int j = 0; j < F; ++j) {
                if (dp[j] == 0.0) continue;
                for (int c = 0; c < d; ++c) dxr[c] += dp[j] * W_up[(int64_t)j * d + c];
            }
        }
    }
}

void oracle_ffn_bwd_cols(const double* x, const double* W_up, const double* W_down,
                         const double* h, const double* dy, double l1,
                         int M, int d, int F, const int32_t* cols, int ncols,
                         double* dWup_out, double* dWdown_out, double* db_out)
{
    (void)W_up;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < ncols; ++i) {
        const int64_t j = cols[i];
        double* gu = dWup_out + (int64_t)i * d;
        double* gd = dWdown_out + (int64_t)i * d;
        double gb = 0.0;
        for (int c = 0; c < d; ++c) { gu[c] = 0.0; gd[c] = 0.0; }
        for (int64_t r = 0; r < M; ++r) {
            double hv = h[r * F + j];
            if (hv == 0.0) continue;
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += dy[r * d + c] * W_down[j * d + c];
            double dp = s + l1;
            gb += dp;
            for (int c = 0; c < d; ++c) {
                gu[c] += dp * x[r * d + c];
                gd[c] += hv * dy[r * d + c];
            }
        }
        db_out[i] = gb;
    }
}

/*
 * The same loss evaluated entirely in fp64 with no rounding anywhere, for
 * finite-difference checks of the backward:
 *   pre = x W_up^T + b,  h = max(pre, 0),  y = h W_down,
 *   L = sum dy * y + l1 * sum h.
 * Writes h (fp64, [M, F]) when h_out is not NULL.
 */
double oracle_ffn_loss_f64(const double* x, const double* W_up, const double* b,
                           const double* W_down, const double* dy, double l1,
                           int M, int d, int F, double* h_out)
{
    double L = 0.0;
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t j = 0; j < F; ++j) {
            double s = b[j];
            for (int c = 0; c < d; ++c) s += x[r * d + c] * W_up[j * d + c];
            double hv = s > 0.0 ? s : 0.0;
            if (h_out) h_out[r * F + j] = hv;
            if (hv == 0.0) continue;
            L += l1 * hv;
            for (int c = 0; c < d; ++c) L += dy[r * d + c] * hv * W_down[j * d + c];
        }
    }
    return L;
}
