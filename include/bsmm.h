/*
 * bsmm.h -- C ABI of libbsmm, block-sparse matrix multiplication on GB300
 * (sm_103a).
 *
 * The operation is OpenAI blocksparse's BlocksparseMatMul, as documented in the
 * blocksparse README, section "API Documentation: blocksparse.matmul":
 *
 *   layout       R x S array of ones and zeros; R = C/bs input block rows (c),
 *                S = K/bs output block columns (k).
 *   block_size   bs in {32, 16, 8}.
 *   feature_axis 1: activations are (N, C) / (N, K) row-major;
 *                0: activations are (C, N) / (K, N) row-major.
 *   w            (nnz, bs, bs): one dense block per nonzero layout entry ("w_shape").
 *                Block ids follow the row-major scan of the layout (c outer, k
 *                inner); block b at layout (c, k) holds W[c*bs+i][k*bs+j] at
 *                w[b][i][j], W being the dense C x K block-sparse weight.
 *   fprop        y  = x  . W                         ("__call__(I, W)")
 *   bprop        dx = dy . W^T                       (gradient w.r.t. the input)
 *   updat        dw[b] = x[:, c_b block]^T . dy[:, k_b block]  (gradient w.r.t. W,
 *                float32 by default: "dw_dtype")
 *   updat_grouped  dw = sum over G <= 8 timesteps of updat(x_t, dy_t)
 *                ("group_param_grads(param_grad, group_size=8, cast32=True)")
 *
 * Conventions common to every call below:
 *   - Pointers named x, w, y, dx, dy, dw, xs[i], dys[i] are DEVICE pointers on
 *     the handle's device, owned by the caller, 16-byte aligned.  The library
 *     never frees or keeps them after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*, NULL = legacy default stream).  Inputs must stay valid until the
 *     work completes.
 *   - Host-side argument checks run first and return an error synchronously,
 *     without enqueuing anything.  Errors detected on the device (a bounded
 *     wait that gave up) are recorded in a sticky per-handle status word that
 *     bsmm_sync_status() reads and clears.  No call traps the device.
 *   - N (minibatch) may be 0 (no work).  With feature_axis = 0 the row pitch is
 *     N elements, so N * sizeof(element) must be a multiple of 16 bytes.
 *   - Outputs of empty block columns (fprop) or empty block rows (bprop) are
 *     written as zeros.
 *   - A handle may be used from several streams at once (its tables are read
 *     only after creation), but not while bsmm_destroy runs.
 *   - The passes launch with programmatic dependent launch: a kernel may start
 *     while the previous kernel on `stream` finishes and read the handle's own
 *     tables (fixed once bsmm_create returns), but it waits for that kernel to
 *     complete before it reads or writes any caller buffer, so stream order
 *     holds as for ordinary launches.
 */
#ifndef BSMM_H
#define BSMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bsmm_ctx *bsmm_t;

typedef enum {
    BSMM_OK = 0,
    BSMM_ERR_INVALID = 1,      /* bad argument (null pointer, bad shape, G out of range, ...) */
    BSMM_ERR_UNSUPPORTED = 2,  /* valid but not implemented (block size, dtype combination) */
    BSMM_ERR_ALIGN = 3,        /* pointer or row pitch not 16-byte aligned */
    BSMM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    BSMM_ERR_TIMEOUT = 5,      /* a device-side bounded wait gave up (sticky) */
    BSMM_ERR_OOM = 6,          /* device allocation failed */
    BSMM_ERR_BOUNDS = 7        /* a device-side index check failed (sticky): a kernel found a
                                  block id or source out of range in its schedule and skipped the
                                  access (the sparse-window fprop/bprop kernels check every one) */
} bsmm_status;

typedef enum { BSMM_F32 = 0, BSMM_F16 = 1, BSMM_BF16 = 2 } bsmm_dtype;

/* Kernel family used by the compute calls.  AUTO picks the tcgen05 tensor-core
 * kernels for 16-bit inputs and the IEEE fp32 SIMT kernels for fp32. */
typedef enum { BSMM_KERNEL_AUTO = 0, BSMM_KERNEL_SIMT = 1, BSMM_KERNEL_TC = 2 } bsmm_kernel;

/*
 * BlocksparseMatMul(layout, block_size, feature_axis)  [README: "class BlocksparseMatMul"]
 * layout_host: HOST pointer to R*S bytes, row-major, nonzero = block present
 * (copied; the caller keeps ownership).  Builds the per-output-column,
 * per-input-row and block-coordinate tables on the device with kernels on
 * `stream`, and waits for them.  On success *out owns device memory freed by
 * bsmm_destroy.  Errors: INVALID (null, R or S < 1, feature_axis not 0/1),
 * UNSUPPORTED (block_size not 8/16/32), OOM, CUDA.
 */
bsmm_status bsmm_create(bsmm_t *out, const uint8_t *layout_host, int R, int S,
                        int block_size, int feature_axis, void *stream);

/* Frees everything the handle owns.  Waits for the device first.  NULL is OK. */
bsmm_status bsmm_destroy(bsmm_t h);

/* w_shape [README: "self.w_shape"]: the weight is (nnz, bs, bs).  Also R, S, feature_axis. */
bsmm_status bsmm_w_shape(bsmm_t h, int64_t *nnz, int *block_size);
bsmm_status bsmm_layout_info(bsmm_t h, int *R, int *S, int *feature_axis);

/* block_coord(block) [README]: layout coordinates (c, k) of block id `block`
 * (host lookup).  INVALID if block is outside [0, nnz). */
bsmm_status bsmm_block_coord(bsmm_t h, int64_t block, int *c, int *k);

/*
 * Copies the device lookup tables to HOST buffers (any may be NULL):
 *   row_ptr[R+1], row_ent[nnz] = k of each block (row-major order, so the
 *   block id of entry e of row c is e itself), col_ptr[S+1],
 *   col_ent[2*nnz] = (block id, c) pairs per output column with c increasing,
 *   coord[2*nnz] = (c, k) per block id.  Synchronous.
 */
bsmm_status bsmm_get_luts(bsmm_t h, int32_t *row_ptr, int32_t *row_ent, int32_t *col_ptr,
                          int32_t *col_ent, int32_t *coord);

/*
 * identity_init(gpu=True) [README: "identity_init + layernorm is all you need",
 * "with gpu=True the init is performed by kernel on the device"]:
 * w[b] = I (bs x bs) when c_b == k_b, else 0.  w: (nnz, bs, bs) of type t.
 */
bsmm_status bsmm_identity_init(bsmm_t h, void *w, bsmm_dtype t, void *stream);

/*
 * fprop [README: "__call__(I, W)"]: y = x . W.
 * x: (N, C) if feature_axis = 1 else (C, N); y: (N, K) or (K, N); w: (nnz, bs, bs).
 * x, w, y share dtype t; accumulation is float32; y is rounded to nearest-even
 * once.  fp32 uses IEEE FMA (no TF32).  y must not overlap x or w.
 */
bsmm_status bsmm_fprop(bsmm_t h, const void *x, const void *w, void *y, int N, bsmm_dtype t,
                       void *stream);

/*
 * bprop (gradient of __call__ w.r.t. I): dx = dy . W^T.
 * dy: (N, K) or (K, N); dx: (N, C) or (C, N).  Same dtype and rounding rules as fprop.
 */
bsmm_status bsmm_bprop(bsmm_t h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t,
                       void *stream);

/*
 * updat (gradient of __call__ w.r.t. W, "dw_dtype"):
 * dw[b][i][j] (+)= sum_n x[n][c_b*bs+i] * dy[n][k_b*bs+j].
 * x, dy of dtype t; dw of dtype dw_t (BSMM_F32, the README's default, or t).
 * accumulate = 0: dw = result; 1: dw += result (float32 add, then one rounding
 * to dw_t).  dw must not overlap x or dy.
 */
bsmm_status bsmm_updat(bsmm_t h, const void *x, const void *dy, void *dw, int N, bsmm_dtype t,
                       bsmm_dtype dw_t, int accumulate, void *stream);

/*
 * Grouped updat [README: "group_param_grads(param_grad, group_size=8, cast32=True)"]:
 * dw (+)= sum_{t<G} sum_n x_t[n][c_b*bs+i] * dy_t[n][k_b*bs+j], all in float32.
 * xs, dys: HOST arrays of G DEVICE pointers (read during the call only), each
 * of the activation shape with minibatch N.  G in [1, 8].  dw: float32.
 */
bsmm_status bsmm_updat_grouped(bsmm_t h, const void *const *xs, const void *const *dys, int G,
                               int N, bsmm_dtype t, float *dw, int accumulate, void *stream);

/*
 * Allocation-free weight gradient.  The paper has no counterpart: this entry point exists
 * for callers that must not allocate device memory -- code running under a framework's
 * memory budget or caching allocator, where a raw cudaMalloc would bypass, fragment or
 * exhaust it, and latency-critical loops that cannot afford an allocation or its failure.
 * bsmm_updat allocates its work tables on first use; this call never allocates: it uses a
 * fixed 4 MB device array that the library holds on every GPU that loads it, until the
 * process exits.
 *
 * Computes the same as bsmm_updat with dw_t = BSMM_F32 for 16-bit x and dy (t = BSMM_F16
 * or BSMM_BF16), using the stacked-block tensor-core kernel.  x, dy, dw are DEVICE
 * pointers as in bsmm_updat; accumulate = 0 sets dw, 1 adds to it.
 * - The first call on a device looks up the array's device address; make that first call
 *   before any stream capture.
 * - The array is shared by every call and keeps the last call's contents.  Each call
 *   rewrites the part it uses (copied from the host, ordered on `stream` before the
 *   kernel), so calls on one stream are safe in sequence, but calls that overlap on the
 *   GPU (other streams, other threads) race on the array and must not be issued.
 * - Errors: INVALID (null handle or pointers, N < 0), ALIGN, UNSUPPORTED (fp32 inputs, a
 *   layout whose work tables need more than the 4 MB array: about 23,000 stacks of
 *   128/bs blocks, e.g. ~95,000 blocks at bs 32; or `stream` is capturing a graph, because
 *   the table is copied from a host buffer that the next call overwrites), CUDA.  Every
 *   error is returned before anything is enqueued.
 */
bsmm_status bsmm_updat_noalloc(bsmm_t h, const void *x, const void *dy, float *dw, int N, bsmm_dtype t,
                               int accumulate, void *stream);

/*
 * layer_norm(x, g, b, axis, epsilon, relu) [README, section "blocksparse.norms": a layernorm
 * for both bsmm feature_axis activation layouts, with an optional relu applied at the end].
 * For every sample n its C features are normalised with their mean and biased variance:
 *   y[n][f] = g[f] * (x[n][f] - mean_n) / sqrt(var_n + epsilon) + b[f],  then max(y, 0) if relu.
 * x, y: DEVICE pointers of dtype t, (N, C) row-major for axis = 1 or (C, N) for axis = 0 (the
 * meaning of feature_axis); g, b: DEVICE pointers to C float32 values.  Statistics and
 * arithmetic in float32, one rounding of y to t.  y may equal x (in place).  Needs no handle;
 * enqueued on `stream`.  N = 0 is a no-op (the pointers are then not used and may be NULL).
 * Errors: INVALID (null pointers, N < 0, C < 1, axis not 0/1, epsilon negative or NaN),
 * ALIGN (pointers not 16-byte aligned, the row pitch -- C for axis = 1, N for axis = 0 --
 * times the element size not a multiple of 16 bytes, or axis = 0 with N not a multiple of 8),
 * UNSUPPORTED (axis = 1 with C > 16384, axis = 0 with C > 163840), CUDA.
 */
bsmm_status bsmm_layer_norm(const void *x, const float *g, const float *b, void *y, int N, int C, int axis,
                            float epsilon, int relu, bsmm_dtype t, void *stream);

/*
 * Gradient of bsmm_layer_norm with respect to x, g and b (training through the layernorm of
 * README section "blocksparse.norms"), for the gradient dy of its output.  With mean_n, rstd_n
 * the statistics of sample n (recomputed from x as in the forward pass), xh = (x - mean_n) * rstd_n,
 * dz = dy, or with relu dy where the forward output y > 0 and 0 elsewhere, and a = g * dz:
 *   dx[n][f] = rstd_n * (a[n][f] - mean_f a[n][.] - xh[n][f] * mean_f (a * xh)[n][.])
 *   dg[f] = sum_n dz[n][f] * xh[n][f],   db[f] = sum_n dz[n][f]
 * x, y, dy, dx: DEVICE pointers of dtype t in the layout of bsmm_layer_norm (y, the forward
 * output, is read only with relu and may be NULL without); g: DEVICE C float32; dg, db: DEVICE
 * C float32 outputs.  Arithmetic in float32, dx rounded once to t; dg and db are sums of
 * per-CTA float32 partials added in a fixed order (deterministic).  workspace: DEVICE scratch
 * of at least bsmm_layer_norm_grad_workspace(N, C, axis) bytes, 16-byte aligned, owned by the
 * caller and free again when the stream reaches the end of the call.  The outputs must not
 * overlap the inputs (x, y and dy are read again after dx is written).  N = 0 sets dg = db = 0
 * and reads nothing else.  Two or three kernels are enqueued on `stream` (dx and per-chunk
 * partial sums, then their reduction).
 * Errors: INVALID (null pointers, dg == db, dx equal to x, y or dy, N < 0, C < 1, axis not 0/1,
 * epsilon negative or NaN, workspace too small), ALIGN (as bsmm_layer_norm, for x, y, dy, dx, g, dg, db, workspace),
 * UNSUPPORTED (axis = 1 with C > 16384, axis = 0 with C > 327680), CUDA.
 */
size_t bsmm_layer_norm_grad_workspace(int N, int C, int axis);
bsmm_status bsmm_layer_norm_grad(const void *x, const void *y, const float *g, const void *dy, void *dx,
                                 float *dg, float *db, int N, int C, int axis, float epsilon, int relu,
                                 bsmm_dtype t, void *workspace, size_t workspace_bytes, void *stream);

/*
 * l2_normalize(W, gain=None, epsilon=1e-6, dtype) [README, "API Documentation: blocksparse.matmul":
 * a BlocksparseMatMul method "to implement weight normalization"].  Every output feature
 * f = k*bs + j has one incoming weight vector, column f of the dense C x K weight: w[b][i][j]
 * for all blocks b of block column k and all rows i.  With s_f its sum of squares:
 *   y[b][i][j] = gain[f] * w[b][i][j] / sqrt(max(s_f, epsilon))      (gain = 1 when NULL)
 * w: DEVICE (nnz, bs, bs) float32; gain: DEVICE K = S*bs float32 values or NULL; y: DEVICE
 * (nnz, bs, bs) of dtype t (the README's dtype argument), rounded once to nearest-even.  Sums
 * in float32, added in a fixed order (deterministic).  y may equal w when t = BSMM_F32;
 * otherwise they must not overlap.  nnz = 0 is a no-op (w, y not used).
 * Errors: INVALID (null handle or pointers, t unknown, epsilon negative or NaN, y == w with a
 * 16-bit t), ALIGN (w or y not 16-byte aligned), CUDA.
 */
bsmm_status bsmm_l2_normalize(bsmm_t h, const float *w, const float *gain, void *y, float epsilon,
                              bsmm_dtype t, void *stream);

/*
 * Gradient of bsmm_l2_normalize with respect to w and gain, for the gradient dy of y.  With
 * rho_f = 1/sqrt(max(s_f, epsilon)) and D_f = sum of dy * w over feature f's vector:
 *   dw[b][i][j] = gain[f] * rho_f * (dy[b][i][j] - [s_f >= epsilon] * rho_f^2 * D_f * w[b][i][j])
 *   dgain[f]    = rho_f * D_f          (also when gain is NULL: the derivative at gain = 1)
 * w: DEVICE float32 (nnz, bs, bs); gain: DEVICE K float32 or NULL; dy: DEVICE (nnz, bs, bs) of
 * dtype t; dw: DEVICE float32 (nnz, bs, bs), must not overlap w or dy; dgain: DEVICE K float32
 * or NULL (not computed).  Features of empty block columns get dgain = 0.
 * Errors: INVALID (null handle, null w/dy/dw with nnz > 0, dw equal to w or dy, t unknown,
 * epsilon negative or NaN), ALIGN (w, dy or dw not 16-byte aligned), CUDA.
 */
bsmm_status bsmm_l2_normalize_grad(bsmm_t h, const float *w, const float *gain, const void *dy, float *dw,
                                   float *dgain, float epsilon, bsmm_dtype t, void *stream);

/*
 * SparseProj(nhidden, nproj=None, proj_stride=None, block_size=32, gather_lut=None) [README,
 * "API Documentation: blocksparse.matmul", class SparseProj: dense-to-sparse and sparse-to-dense
 * projections like the TensorFlow gather / scatter ops, over a unique one-to-one mapping so that
 * no backward op needs atomics].
 * The map: sparse feature p (p < nproj) is dense feature lut[p] (lut[p] < nhidden).
 * gather_lut: HOST array of nproj distinct indices in [0, nhidden) (copied), or NULL for runs of
 * block_size consecutive features, one run starting every proj_stride features:
 *   lut[r*block_size + i] = r*proj_stride + i,
 * where proj_stride <= 0 means block_size and nproj <= 0 means as many runs as fit in nhidden.
 * Copies the map and its inverse to the current device (synchronously).  On success *out owns
 * device memory freed by bsmm_proj_destroy.
 * Errors: INVALID (null out, nhidden < 1, entries out of range or repeated, nproj > nhidden, a
 * default map that does not fit, nproj not a multiple of block_size), OOM, CUDA.
 */
typedef struct bsmm_proj_ctx *bsmm_proj_t;
bsmm_status bsmm_proj_create(bsmm_proj_t *out, int nhidden, int nproj, int proj_stride, int block_size,
                             const int32_t *gather_lut);
bsmm_status bsmm_proj_destroy(bsmm_proj_t p);                      /* waits for the device; NULL is OK */
bsmm_status bsmm_proj_info(bsmm_proj_t p, int *nhidden, int *nproj);
bsmm_status bsmm_proj_get_lut(bsmm_proj_t p, int32_t *lut);        /* HOST array of nproj entries */

typedef enum {
    BSMM_PROJ_GATHER = 0,       /* out[n][p] = x[n][lut[p]]                         x dense, out sparse */
    BSMM_PROJ_SCATTER = 1,      /* out[n][lut[p]] = x[n][p], other features 0       x sparse, out dense */
    BSMM_PROJ_SCATTER_ADD = 2,  /* out = x; out[n][lut[p]] = x[n][lut[p]] + y[n][p]  x, out dense; y sparse */
    BSMM_PROJ_SCATTER_MUL = 3,  /* out = x; out[n][lut[p]] = x[n][lut[p]] * y[n][p]  x, out dense; y sparse */
    BSMM_PROJ_GATHER_MUL = 4    /* out[n][p] = x[n][lut[p]] * y[n][lut[p]]           x, y dense; out sparse
                                   (the gradient of scatter_mul with respect to y is gather_mul(dout, x)) */
} bsmm_proj_op;

/*
 * One SparseProj operation.  x, y, out: DEVICE pointers of dtype t, 16-byte aligned; dense
 * arrays have nhidden features, sparse ones nproj; (N, F) row-major for axis = 1, (F, N) for
 * axis = 0 (feature_axis), and for axis = 0 N * sizeof(element) must be a multiple of 16 bytes.
 * y is read only by SCATTER_ADD, SCATTER_MUL and GATHER_MUL.  Sums and products are formed in
 * float32 and rounded to t once (exact copies otherwise).  out may equal x for SCATTER_ADD and
 * SCATTER_MUL (then only the mapped features are read and written); otherwise out must not
 * overlap x or y.  N = 0 is a no-op.  Enqueued on `stream`.
 * Errors: INVALID (null handle or pointers, N < 0, op, axis or t unknown, out == x for another
 * op, out == y), ALIGN, CUDA.
 */
bsmm_status bsmm_proj(bsmm_proj_t p, bsmm_proj_op op, const void *x, const void *y, void *out, int N, int axis,
                      bsmm_dtype t, void *stream);

/* Kernel family for later calls on this handle (testing / comparison). */
bsmm_status bsmm_set_kernel(bsmm_t h, bsmm_kernel which);

/* Waits for `stream`, then returns and clears the handle's sticky device
 * status (OK, TIMEOUT or BOUNDS), or CUDA if the stream reports an error. */
bsmm_status bsmm_sync_status(bsmm_t h, void *stream);

/* Static description of a status code. */
const char *bsmm_status_string(bsmm_status s);

/* Number of kernels this library has launched since load (all handles). */
int64_t bsmm_launch_count(void);

/*
 * Failure-detection self-test (no counterpart in the README): enqueues a kernel whose
 * single thread waits on an mbarrier that nothing ever arrives on, using the same bounded
 * wait as the tensor-core kernels, with a limit of limit_ns nanoseconds (1 .. 1e10).  The
 * wait gives up, records BSMM_ERR_TIMEOUT in the handle's sticky status, and the kernel
 * returns normally: a following bsmm_sync_status() reports TIMEOUT and the CUDA context
 * stays usable.  Errors: INVALID (null handle, limit out of range), CUDA.
 */
bsmm_status bsmm_selftest_wait_timeout(bsmm_t h, uint64_t limit_ns, void *stream);

/*
 * Launch-cost self-test (no counterpart in the README; computes nothing): enqueues on `stream`
 * one empty kernel of `ctas` CTAs of 160 threads with the launch attributes of the library's
 * kernels (programmatic dependent launch).  With tensor_memory != 0 one warp of each CTA
 * allocates and frees 32 tensor-memory columns, as every tensor-core kernel does.  Timing it
 * gives the fixed cost that every pass carries when launched alone.
 * Errors: INVALID (null handle, ctas outside 1 .. 65535), CUDA.
 */
bsmm_status bsmm_selftest_empty_launch(bsmm_t h, int ctas, int tensor_memory, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BSMM_H */
