/*
 * bsmm_oracle.c -- plain, slow, obviously-correct CPU oracle for block-sparse
 * matrix multiplication.  TEST INFRASTRUCTURE ONLY: it exists to check the
 * CUDA library and may be used only by the tests, the package's smoke check
 * and the CPU-baseline leg of the benchmark.  The product path never calls it.
 *
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Source: the blocksparse README (openai/blocksparse, as mirrored on the
 * kiteco/blocksparse page), section "API Documentation: blocksparse.matmul":
 *   - BlocksparseMatMul(layout, block_size, feature_axis): layout is a 2-D 0/1
 *     array of blocks, block_size in {32,16,8}, feature_axis 1 means (N,C)
 *     activations and 0 means (C,N).
 *   - block_coord(block): the (c,k) layout coordinate of a block id.
 *   - w_shape: one bs x bs weight block per nonzero layout entry.
 *   - __call__(I, W): y = I . W with W the block-sparse (C x K) weight.
 *   - identity_init: identity initialisation of the weight blocks.
 *   - l2_normalize: weight normalisation of the block-sparse weight (and its
 *     gradient), near the end of this file.
 *   - SparseProj: gather / scatter projections over a one-to-one feature map (at
 *     the end of this file).
 *   - group_param_grads: the weight gradients of up to 8 timesteps sharing one
 *     weight are summed (cast32: in float32 or wider).
 * and its section "blocksparse.norms" for layer_norm (at the end of this file).
 *
 * Readings where the page is silent (each one also listed in the design notes):
 *   - block ids are assigned in row-major scan order of the layout
 *     (c outer, k inner);
 *   - weight block b at layout (c,k) holds W[c*bs+i][k*bs+j] at w[b][i][j];
 *   - identity_init sets blocks with c == k to the bs x bs identity and every
 *     other block to zero;
 *   - an output block column (row) with no nonzero block is zero.
 *
 * Everything is float64, row-major, no blocking or reordering of the sums
 * beyond the definition: each output is accumulated over its reduction index
 * in increasing order.  OpenMP only splits independent outputs across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of nonzero blocks of a layout. */
int64_t oracle_nnz(const uint8_t *L, int R, int S)
{
    int64_t n = 0;
    for (int64_t i = 0; i < (int64_t)R * S; ++i)
        n += L[i] != 0;
    return n;
}

/* Block-id map: bid[c*S+k] = id of block (c,k) in row-major scan order, or -1. */
static int32_t *block_id_map(const uint8_t *L, int R, int S)
{
    int32_t *bid = (int32_t *)malloc(sizeof(int32_t) * (size_t)R * (size_t)S);
    int32_t next = 0;
    for (int c = 0; c < R; ++c)
        for (int k = 0; k < S; ++k)
            bid[(size_t)c * S + k] = L[(size_t)c * S + k] ? next++ : -1;
    return bid;
}

/*
 * Lookup tables, built by naive scans.
 *   coord[2b], coord[2b+1]       = (c, k) of block b            (block_coord)
 *   col_ptr[k] .. col_ptr[k+1]   = entries of output block column k,
 *   col_ent[2e], col_ent[2e+1]   = (b, c), c increasing
 *   row_ptr[c] .. row_ptr[c+1]   = entries of input block row c,
 *   row_ent[e]                   = k, k increasing (the block id is e itself)
 */
void oracle_luts(const uint8_t *L, int R, int S,
                 int32_t *row_ptr, int32_t *row_ent,
                 int32_t *col_ptr, int32_t *col_ent, int32_t *coord)
{
    int32_t *bid = block_id_map(L, R, S);
    int32_t e = 0;
    for (int c = 0; c < R; ++c) {
        row_ptr[c] = e;
        for (int k = 0; k < S; ++k)
            if (L[(size_t)c * S + k]) {
                row_ent[e] = k;
                coord[2 * e] = c;
                coord[2 * e + 1] = k;
                ++e;
            }
    }
    row_ptr[R] = e;
    e = 0;
    for (int k = 0; k < S; ++k) {
        col_ptr[k] = e;
        for (int c = 0; c < R; ++c)
            if (L[(size_t)c * S + k]) {
                col_ent[2 * e] = bid[(size_t)c * S + k];
                col_ent[2 * e + 1] = c;
                ++e;
            }
    }
    col_ptr[S] = e;
    free(bid);
}

/* Dense C x K weight from the layout and the (nnz, bs, bs) blocks. */
void oracle_densify(const uint8_t *L, int R, int S, int bs, const double *w, double *Wd)
{
    int64_t C = (int64_t)R * bs, K = (int64_t)S * bs;
    int32_t *bid = block_id_map(L, R, S);
    for (int64_t cc = 0; cc < C; ++cc)
        for (int64_t kk = 0; kk < K; ++kk) {
            int32_t b = bid[(cc / bs) * S + kk / bs];
            Wd[cc * K + kk] = b < 0 ? 0.0 : w[((int64_t)b * bs + cc % bs) * bs + kk % bs];
        }
    free(bid);
}

/* identity_init: w[b] = I if c_b == k_b else 0. */
void oracle_identity_init(const uint8_t *L, int R, int S, int bs, double *w)
{
    int64_t b = 0;
    for (int c = 0; c < R; ++c)
        for (int k = 0; k < S; ++k)
            if (L[(size_t)c * S + k]) {
                for (int i = 0; i < bs; ++i)
                    for (int j = 0; j < bs; ++j)
                        w[(b * bs + i) * bs + j] = (c == k && i == j) ? 1.0 : 0.0;
                ++b;
            }
}

/* Activation element (n, f) of an (N,F) [fa=1] or (F,N) [fa=0] array. */
static inline double act(const double *a, int64_t n, int64_t f, int64_t N, int64_t F, int fa)
{
    return fa ? a[n * F + f] : a[f * N + n];
}

static inline double *act_ptr(double *a, int64_t n, int64_t f, int64_t N, int64_t F, int fa)
{
    return fa ? &a[n * F + f] : &a[f * N + n];
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * fprop: y[n][kk] = sum_{cc=0}^{C-1} x[n][cc] * Wd[cc][kk]  (y = x . W).
 * Rows n in [n_lo, n_hi) only (the rest of y is left untouched).
 */
void oracle_fprop(const double *x, const double *Wd, double *y,
                  int N, int C, int K, int fa, int n_lo, int n_hi, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = n_lo; n < n_hi; ++n)
        for (int64_t kk = 0; kk < K; ++kk) {
            double s = 0.0;
            for (int64_t cc = 0; cc < C; ++cc)
                s += act(x, n, cc, N, C, fa) * Wd[cc * K + kk];
            *act_ptr(y, n, kk, N, K, fa) = s;
        }
}

/*
 * bprop: dx[n][cc] = sum_{kk=0}^{K-1} dy[n][kk] * Wd[cc][kk]  (dx = dy . W^T).
 */
void oracle_bprop(const double *dy, const double *Wd, double *dx,
                  int N, int C, int K, int fa, int n_lo, int n_hi, int nthreads)
{
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = n_lo; n < n_hi; ++n)
        for (int64_t cc = 0; cc < C; ++cc) {
            double s = 0.0;
            for (int64_t kk = 0; kk < K; ++kk)
                s += act(dy, n, kk, N, K, fa) * Wd[cc * K + kk];
            *act_ptr(dx, n, cc, N, C, fa) = s;
        }
}

/*
 * updat: dw[b][i][j] = sum_{n=0}^{N-1} x[n][c_b*bs+i] * dy[n][k_b*bs+j],
 * for blocks b in [b_lo, b_hi).  With accumulate != 0 the sum is added to the
 * value already in dw (one rounding-free float64 add).
 */
void oracle_updat(const uint8_t *L, int R, int S, int bs,
                  const double *x, const double *dy, double *dw,
                  int N, int fa, int accumulate, int64_t b_lo, int64_t b_hi, int nthreads)
{
    int64_t C = (int64_t)R * bs, K = (int64_t)S * bs;
    int64_t nnz = oracle_nnz(L, R, S);
    int32_t *cb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int32_t *kb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int64_t e = 0;
    for (int c = 0; c < R; ++c)
        for (int k = 0; k < S; ++k)
            if (L[(size_t)c * S + k]) {
                cb[e] = c;
                kb[e] = k;
                ++e;
            }
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = b_lo; b < b_hi; ++b)
        for (int i = 0; i < bs; ++i)
            for (int j = 0; j < bs; ++j) {
                double s = 0.0;
                for (int64_t n = 0; n < N; ++n)
                    s += act(x, n, (int64_t)cb[b] * bs + i, N, C, fa) *
                         act(dy, n, (int64_t)kb[b] * bs + j, N, K, fa);
                double *o = &dw[(b * bs + i) * bs + j];
                *o = accumulate ? *o + s : s;
            }
    free(cb);
    free(kb);
}

/*
 * Grouped updat (group_param_grads): dw[b] = (accumulate ? dw[b] : 0)
 *   + sum_{t<G} updat(x_t, dy_t)[b], each step's sum formed first and then
 * added in timestep order.  xs/dys point to G arrays of the activation shape.
 */
void oracle_updat_grouped(const uint8_t *L, int R, int S, int bs,
                          const double *const *xs, const double *const *dys, int G,
                          double *dw, int N, int fa, int accumulate, int nthreads)
{
    int64_t nnz = oracle_nnz(L, R, S);
    int64_t sz = nnz * bs * bs;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(sz ? sz : 1));
    if (!accumulate)
        memset(dw, 0, sizeof(double) * (size_t)sz);
    for (int t = 0; t < G; ++t) {
        oracle_updat(L, R, S, bs, xs[t], dys[t], tmp, N, fa, 0, 0, nnz, nthreads);
        for (int64_t q = 0; q < sz; ++q)
            dw[q] += tmp[q];
    }
    free(tmp);
}

/*
 * Single sampled outputs, computed straight from the definition without
 * densifying W (for checks at sizes where the full product is too slow).
 *   fprop_at: out[s] = y[n_s][f_s]   = sum_cc x[n][cc] * W(cc, f)
 *   bprop_at: out[s] = dx[n_s][f_s]  = sum_kk dy[n][kk] * W(f, kk)
 *   updat_at: out[s] = dw[b_s][i_s][j_s]
 * W(cc, kk) is looked up through the block-id map.
 */
void oracle_fprop_at(const uint8_t *L, int R, int S, int bs, const double *w, const double *x,
                     int N, int fa, const int64_t *n_s, const int64_t *f_s, int64_t count, double *out)
{
    int64_t C = (int64_t)R * bs, K = (int64_t)S * bs;
    int32_t *bid = block_id_map(L, R, S);
    for (int64_t s = 0; s < count; ++s) {
        int64_t n = n_s[s], kk = f_s[s];
        double acc = 0.0;
        for (int64_t cc = 0; cc < C; ++cc) {
            int32_t b = bid[(cc / bs) * S + kk / bs];
            double wv = b < 0 ? 0.0 : w[((int64_t)b * bs + cc % bs) * bs + kk % bs];
            acc += act(x, n, cc, N, C, fa) * wv;
        }
        out[s] = acc;
    }
    (void)K;
    free(bid);
}

void oracle_bprop_at(const uint8_t *L, int R, int S, int bs, const double *w, const double *dy,
                     int N, int fa, const int64_t *n_s, const int64_t *f_s, int64_t count, double *out)
{
    int64_t K = (int64_t)S * bs;
    int32_t *bid = block_id_map(L, R, S);
    for (int64_t s = 0; s < count; ++s) {
        int64_t n = n_s[s], cc = f_s[s];
        double acc = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) {
            int32_t b = bid[(cc / bs) * S + kk / bs];
            double wv = b < 0 ? 0.0 : w[((int64_t)b * bs + cc % bs) * bs + kk % bs];
            acc += act(dy, n, kk, N, K, fa) * wv;
        }
        out[s] = acc;
    }
    free(bid);
}

void oracle_updat_at(const uint8_t *L, int R, int S, int bs, const double *x, const double *dy,
                     int N, int fa, const int64_t *b_s, const int64_t *i_s, const int64_t *j_s,
                     int64_t count, double *out)
{
    int64_t C = (int64_t)R * bs, K = (int64_t)S * bs;
    int64_t nnz = oracle_nnz(L, R, S);
    int32_t *cb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int32_t *kb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int64_t e = 0;
    for (int c = 0; c < R; ++c)
        for (int k = 0; k < S; ++k)
            if (L[(size_t)c * S + k]) {
                cb[e] = c;
                kb[e] = k;
                ++e;
            }
    for (int64_t s = 0; s < count; ++s) {
        int64_t b = b_s[s];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n)
            acc += act(x, n, (int64_t)cb[b] * bs + i_s[s], N, C, fa) *
                   act(dy, n, (int64_t)kb[b] * bs + j_s[s], N, K, fa);
        out[s] = acc;
    }
    free(cb);
    free(kb);
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * layer_norm(x, g, b, axis, epsilon, relu)  [blocksparse README, section
 * "blocksparse.norms": a layernorm for both bsmm feature_axis activation layouts,
 * with an optional relu applied at the end].  The page gives the signature only;
 * the readings taken:
 *   - the statistics of sample n run over its C features: row n of an (N,C)
 *     array for axis = 1, column n of a (C,N) array for axis = 0 (the same
 *     meaning as feature_axis);
 *   - the variance is the biased one (divided by C), epsilon is added to it
 *     inside the square root, and g, b are per-feature scale and shift:
 *       y[n][f] = g[f] * (x[n][f] - mean_n) / sqrt(var_n + epsilon) + b[f];
 *   - relu replaces negative outputs by zero after the shift.
 * Mean first, then the variance of the deviations (two passes), all float64,
 * features in increasing order.
 */
void oracle_layer_norm(const double *x, const double *g, const double *b, double *y,
                       int N, int C, int axis, double epsilon, int relu)
{
    for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t f = 0; f < C; ++f)
            s += act(x, n, f, N, C, axis);
        const double mean = s / (double)C;
        double v = 0.0;
        for (int64_t f = 0; f < C; ++f) {
            const double d = act(x, n, f, N, C, axis) - mean;
            v += d * d;
        }
        const double sd = sqrt(v / (double)C + epsilon);
        for (int64_t f = 0; f < C; ++f) {
            double o = g[f] * (act(x, n, f, N, C, axis) - mean) / sd + b[f];
            if (relu && o < 0.0)
                o = 0.0;
            *act_ptr(y, n, f, N, C, axis) = o;
        }
    }
}

/*
 * Gradient of layer_norm with respect to x, g and b, for the gradient dy of its output
 * (training through the layernorm of the README's "blocksparse.norms" section; the page gives
 * the forward signature only).  Readings, besides those of the forward pass above:
 *   - with relu the gradient passes where the forward output y is positive and is zero where
 *     y <= 0 (the relu derivative at 0 taken as 0); y is the forward result the caller holds,
 *     so the mask is the one its forward pass produced (y is not read without relu);
 *   - the derivative is that of the forward formula, mean and variance included:
 *       xh = (x - mean_n) / sd_n,  dz = dy (masked),  a = g * dz
 *       db[f] = sum_n dz[n][f],  dg[f] = sum_n dz[n][f] * xh[n][f]
 *       dx[n][f] = (a[n][f] - mean_f' a[n][f'] - xh[n][f] * mean_f' a[n][f'] * xh[n][f']) / sd_n
 * Statistics as in the forward pass (mean, then the variance of the deviations), float64,
 * features and samples in increasing order.
 */
void oracle_layer_norm_grad(const double *x, const double *y, const double *g, const double *dy,
                            double *dx, double *dg, double *db, int N, int C, int axis, double epsilon,
                            int relu)
{
    for (int64_t f = 0; f < C; ++f) {
        dg[f] = 0.0;
        db[f] = 0.0;
    }
    for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t f = 0; f < C; ++f)
            s += act(x, n, f, N, C, axis);
        const double mean = s / (double)C;
        double v = 0.0;
        for (int64_t f = 0; f < C; ++f) {
            const double d = act(x, n, f, N, C, axis) - mean;
            v += d * d;
        }
        const double sd = sqrt(v / (double)C + epsilon);
        double sa = 0.0, sax = 0.0;
        for (int64_t f = 0; f < C; ++f) {
            const double xh = (act(x, n, f, N, C, axis) - mean) / sd;
            double dz = act(dy, n, f, N, C, axis);
            if (relu && !(act(y, n, f, N, C, axis) > 0.0))
                dz = 0.0;
            db[f] += dz;
            dg[f] += dz * xh;
            sa += g[f] * dz;
            sax += g[f] * dz * xh;
        }
        const double ma = sa / (double)C, max_ = sax / (double)C;
        for (int64_t f = 0; f < C; ++f) {
            const double xh = (act(x, n, f, N, C, axis) - mean) / sd;
            double dz = act(dy, n, f, N, C, axis);
            if (relu && !(act(y, n, f, N, C, axis) > 0.0))
                dz = 0.0;
            *act_ptr(dx, n, f, N, C, axis) = (g[f] * dz - ma - xh * max_) / sd;
        }
    }
}

/*
 * l2_normalize(W, gain=None, epsilon=1e-6, dtype)  [blocksparse README, section "API
 * Documentation: blocksparse.matmul": a BlocksparseMatMul method for weight normalisation].
 * The page gives the signature only; the readings taken:
 *   - the norm belongs to one output feature f = k*bs + j and runs over its whole incoming
 *     weight vector, column f of the dense C x K weight: w[b][i][j] for every block b of
 *     block column k and every i (weight normalisation of one output unit);
 *   - epsilon is a lower bound on the squared norm, as in TensorFlow's l2_normalize:
 *       s_f = sum of w^2 over the column,  y[b][i][j] = gain[f] * w[b][i][j] / sqrt(max(s_f, epsilon));
 *   - gain, when given, holds one value per output feature (K of them); without it the gain is 1;
 *   - dtype is the type the result is delivered in (rounding is the caller's).
 * Blocks of a column are visited in increasing c, rows i in increasing order.
 */
void oracle_l2_normalize(const uint8_t *L, int R, int S, int bs, const double *w, const double *gain,
                         double epsilon, double *y)
{
    int32_t *bid = block_id_map(L, R, S);
    const int64_t bb = (int64_t)bs * bs;
    for (int k = 0; k < S; ++k)
        for (int j = 0; j < bs; ++j) {
            double s = 0.0;
            for (int c = 0; c < R; ++c) {
                const int32_t b = bid[(size_t)c * S + k];
                if (b < 0)
                    continue;
                for (int i = 0; i < bs; ++i) {
                    const double v = w[b * bb + (int64_t)i * bs + j];
                    s += v * v;
                }
            }
            const double g = gain ? gain[(int64_t)k * bs + j] : 1.0;
            const double norm = sqrt(s > epsilon ? s : epsilon);
            for (int c = 0; c < R; ++c) {
                const int32_t b = bid[(size_t)c * S + k];
                if (b < 0)
                    continue;
                for (int i = 0; i < bs; ++i) {
                    const int64_t o = b * bb + (int64_t)i * bs + j;
                    y[o] = g * w[o] / norm;
                }
            }
        }
    free(bid);
}

/*
 * Gradient of l2_normalize, written out from the definition above by the chain rule.  With
 * rho = 1/sqrt(max(s_f, epsilon)) and D_f = sum over the column of dy * w:
 *   d y[m] / d w[i]  = gain * (rho * [m == i] - rho^3 * w[m] * w[i])  when s_f >= epsilon
 *                      (the squared norm is the larger argument of the max; ties go to it, as
 *                      TensorFlow's maximum does), and gain * rho * [m == i] otherwise;
 *   dw[i]     = gain * rho * (dy[i] - [s_f >= epsilon] * rho^2 * D_f * w[i]);
 *   dgain[f]  = rho * D_f  (the derivative with respect to gain, also when no gain was given).
 * dgain may be NULL.
 */
void oracle_l2_normalize_grad(const uint8_t *L, int R, int S, int bs, const double *w, const double *gain,
                              double epsilon, const double *dy, double *dw, double *dgain)
{
    int32_t *bid = block_id_map(L, R, S);
    const int64_t bb = (int64_t)bs * bs;
    for (int k = 0; k < S; ++k)
        for (int j = 0; j < bs; ++j) {
            double s = 0.0, d = 0.0;
            for (int c = 0; c < R; ++c) {
                const int32_t b = bid[(size_t)c * S + k];
                if (b < 0)
                    continue;
                for (int i = 0; i < bs; ++i) {
                    const int64_t o = b * bb + (int64_t)i * bs + j;
                    s += w[o] * w[o];
                    d += dy[o] * w[o];
                }
            }
            const int64_t f = (int64_t)k * bs + j;
            const double g = gain ? gain[f] : 1.0;
            const double rho = 1.0 / sqrt(s > epsilon ? s : epsilon);
            const double cw = s >= epsilon ? rho * rho * d : 0.0;
            for (int c = 0; c < R; ++c) {
                const int32_t b = bid[(size_t)c * S + k];
                if (b < 0)
                    continue;
                for (int i = 0; i < bs; ++i) {
                    const int64_t o = b * bb + (int64_t)i * bs + j;
                    dw[o] = g * rho * (dy[o] - cw * w[o]);
                }
            }
            if (dgain)
                dgain[f] = rho * d;
        }
    free(bid);
}

/*
 * SparseProj(nhidden, nproj, proj_stride, block_size, gather_lut) with gather, scatter,
 * scatter_add and scatter_mul  [blocksparse README, section "API Documentation:
 * blocksparse.matmul", class SparseProj: dense-to-sparse and sparse-to-dense projections like the
 * TensorFlow gather/scatter ops, over a unique one-to-one mapping].  The page gives the signatures
 * only; the readings taken:
 *   - gather_lut lists nproj distinct feature indices in [0, nhidden): sparse feature p is dense
 *     feature lut[p];
 *   - without gather_lut the map keeps runs of block_size consecutive features, one run starting
 *     every proj_stride features (proj_stride defaults to block_size):
 *       lut[r*block_size + i] = r*proj_stride + i;
 *   - activations are (N, F) row-major for axis = 1 and (F, N) for axis = 0 (the meaning of the
 *     matmul's feature_axis);
 *   - gather(x)          out[n][p] = x[n][lut[p]]                         (N, nproj)
 *     scatter(x)         out[n][lut[p]] = x[n][p], every other feature 0   (N, nhidden)
 *     scatter_add(x, y)  out = x, then out[n][lut[p]] = x[n][lut[p]] + y[n][p]
 *     scatter_mul(x, y)  out = x, then out[n][lut[p]] = x[n][lut[p]] * y[n][p]
 *     gather_mul(x, y)   out[n][p] = x[n][lut[p]] * y[n][lut[p]]  (x, y dense; the gradient of
 *                        scatter_mul with respect to its sparse operand is gather_mul(dout, x)).
 * Values are float64; the caller rounds.
 */
void oracle_proj_default_lut(int nproj, int proj_stride, int block_size, int32_t *lut)
{
    for (int p = 0; p < nproj; ++p)
        lut[p] = (p / block_size) * proj_stride + p % block_size;
}

static double *proj_at(double *a, int64_t n, int64_t f, int64_t N, int64_t F, int axis)
{
    return axis == 1 ? a + n * F + f : a + f * N + n;
}

/* op: 0 gather, 1 scatter, 2 scatter_add, 3 scatter_mul, 4 gather_mul. */
void oracle_sparse_proj(int op, const double *x, const double *y, double *out, const int32_t *lut,
                        int N, int nhidden, int nproj, int axis)
{
    double *xm = (double *)x, *ym = (double *)y;
    if (op == 1 || op == 2 || op == 3) {          /* dense output: start from 0 or from x */
        for (int64_t n = 0; n < N; ++n)
            for (int64_t f = 0; f < nhidden; ++f)
                *proj_at(out, n, f, N, nhidden, axis) = op == 1 ? 0.0 : *proj_at(xm, n, f, N, nhidden, axis);
    }
    for (int64_t n = 0; n < N; ++n)
        for (int64_t p = 0; p < nproj; ++p) {
            const int64_t f = lut[p];
            if (op == 0) {
                *proj_at(out, n, p, N, nproj, axis) = *proj_at(xm, n, f, N, nhidden, axis);
            } else if (op == 1) {
                *proj_at(out, n, f, N, nhidden, axis) = *proj_at(xm, n, p, N, nproj, axis);
            } else if (op == 2) {
                *proj_at(out, n, f, N, nhidden, axis) += *proj_at(ym, n, p, N, nproj, axis);
            } else if (op == 3) {
                *proj_at(out, n, f, N, nhidden, axis) *= *proj_at(ym, n, p, N, nproj, axis);
            } else {
                *proj_at(out, n, p, N, nproj, axis) =
                    *proj_at(xm, n, f, N, nhidden, axis) * *proj_at(ym, n, f, N, nhidden, axis);
            }
        }
}
