// C ABI of libbsmm: handle management, argument checks and kernel dispatch.
// The operations are those of BlocksparseMatMul in the blocksparse README
// ("API Documentation: blocksparse.matmul"); include/bsmm.h states each
// call's contract.
#include "bsmm_internal.cuh"

#include <cstdlib>
#include <new>

std::atomic<int64_t> g_bsmm_launches{0};

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool valid_dtype(bsmm_dtype t) { return t == BSMM_F32 || t == BSMM_F16 || t == BSMM_BF16; }

// Common checks of the compute calls.
bsmm_status check_call(bsmm_ctx *h, int N, bsmm_dtype t)
{
    if (!h) return BSMM_ERR_INVALID;
    if (N < 0) return BSMM_ERR_INVALID;
    if (!valid_dtype(t)) return BSMM_ERR_INVALID;
    if (h->fa == 0 && ((int64_t)N * dtype_size(t)) % 16 != 0) return BSMM_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSMM_ERR_CUDA;
    if (dev != h->device) cudaSetDevice(h->device);
    return BSMM_OK;
}

bool use_tc(bsmm_ctx *h, bsmm_dtype t)
{
    if (h->kernel == BSMM_KERNEL_SIMT) return false;
    if (t == BSMM_F32) return false;
    return tc_supported(h, t);
}

void free_ctx(bsmm_ctx *h)
{
    tc_release(h);
    sp_release(h);
    cudaFree(h->d_layout);
    cudaFree(h->d_row_ptr);
    cudaFree(h->d_row_ent);
    cudaFree(h->d_col_ptr);
    cudaFree(h->d_col_ent);
    cudaFree(h->d_coord);
    cudaFree(h->d_bid);
    cudaFree(h->d_status);
    delete h;
}

} // namespace

extern "C" {

bsmm_status bsmm_create(bsmm_t *out, const uint8_t *layout_host, int R, int S, int block_size,
                        int feature_axis, void *stream)
{
    if (!out || !layout_host || R < 1 || S < 1) return BSMM_ERR_INVALID;
    *out = nullptr;
    if (block_size != 8 && block_size != 16 && block_size != 32) return BSMM_ERR_UNSUPPORTED;
    if (feature_axis != 0 && feature_axis != 1) return BSMM_ERR_INVALID;
    if ((int64_t)R * block_size > (1 << 24) || (int64_t)S * block_size > (1 << 24)) return BSMM_ERR_INVALID;
    if ((int64_t)R * S > (int64_t)1 << 30) return BSMM_ERR_INVALID;

    bsmm_ctx *h = new (std::nothrow) bsmm_ctx();
    if (!h) return BSMM_ERR_OOM;
    h->R = R;
    h->S = S;
    h->bs = block_size;
    h->fa = feature_axis;
    if (const char *e = getenv("BSMM_TC_WLOG")) h->tc_wlog = atoi(e);
    if (const char *e = getenv("BSMM_TC_STAGE_KB")) h->tc_stage_kb = atoi(e);
    if (const char *e = getenv("BSMM_TC_ROWS")) h->tc_rows = atoi(e);
    if (const char *e = getenv("BSMM_TC_BINS")) h->tc_bins = atoi(e);
    if (const char *e = getenv("BSMM_TC_ESLOTS")) h->tc_eslots = atoi(e);
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        delete h;
        return BSMM_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMalloc(&h->d_status, sizeof(int32_t)) != cudaSuccess) {
        free_ctx(h);
        return BSMM_ERR_OOM;
    }
    if (cudaMemsetAsync(h->d_status, 0, sizeof(int32_t), s) != cudaSuccess) {
        free_ctx(h);
        return BSMM_ERR_CUDA;
    }
    bsmm_status st = lut_build(h, layout_host, s);
    if (st != BSMM_OK) {
        cudaStreamSynchronize(s);
        free_ctx(h);
        return st;
    }
    *out = h;
    return BSMM_OK;
}

bsmm_status bsmm_destroy(bsmm_t h)
{
    if (!h) return BSMM_OK;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    free_ctx(h);
    return BSMM_OK;
}

bsmm_status bsmm_w_shape(bsmm_t h, int64_t *nnz, int *block_size)
{
    if (!h) return BSMM_ERR_INVALID;
    if (nnz) *nnz = h->nnz;
    if (block_size) *block_size = h->bs;
    return BSMM_OK;
}

bsmm_status bsmm_layout_info(bsmm_t h, int *R, int *S, int *feature_axis)
{
    if (!h) return BSMM_ERR_INVALID;
    if (R) *R = h->R;
    if (S) *S = h->S;
    if (feature_axis) *feature_axis = h->fa;
    return BSMM_OK;
}

bsmm_status bsmm_block_coord(bsmm_t h, int64_t block, int *c, int *k)
{
    if (!h || block < 0 || block >= h->nnz) return BSMM_ERR_INVALID;
    if (c) *c = h->h_coord[2 * block];
    if (k) *k = h->h_coord[2 * block + 1];
    return BSMM_OK;
}

bsmm_status bsmm_get_luts(bsmm_t h, int32_t *row_ptr, int32_t *row_ent, int32_t *col_ptr, int32_t *col_ent,
                          int32_t *coord)
{
    if (!h) return BSMM_ERR_INVALID;
    cudaSetDevice(h->device);
    // Read the DEVICE tables (not the host mirrors) so callers can check what kernels use.
    if (row_ptr && cudaMemcpy(row_ptr, h->d_row_ptr, (h->R + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost))
        return BSMM_ERR_CUDA;
    if (col_ptr && cudaMemcpy(col_ptr, h->d_col_ptr, (h->S + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost))
        return BSMM_ERR_CUDA;
    if (h->nnz > 0) {
        if (row_ent && cudaMemcpy(row_ent, h->d_row_ent, h->nnz * sizeof(int32_t), cudaMemcpyDeviceToHost))
            return BSMM_ERR_CUDA;
        if (col_ent && cudaMemcpy(col_ent, h->d_col_ent, 2 * h->nnz * sizeof(int32_t), cudaMemcpyDeviceToHost))
            return BSMM_ERR_CUDA;
        if (coord && cudaMemcpy(coord, h->d_coord, 2 * h->nnz * sizeof(int32_t), cudaMemcpyDeviceToHost))
            return BSMM_ERR_CUDA;
    }
    return BSMM_OK;
}

bsmm_status bsmm_identity_init(bsmm_t h, void *w, bsmm_dtype t, void *stream)
{
    bsmm_status st = check_call(h, 0, t);
    if (st != BSMM_OK) return st;
    if (h->nnz > 0 && !w) return BSMM_ERR_INVALID;
    if (h->nnz > 0 && !aligned16(w)) return BSMM_ERR_ALIGN;
    return launch_identity_init(h, w, t, (cudaStream_t)stream);
}

bsmm_status bsmm_fprop(bsmm_t h, const void *x, const void *w, void *y, int N, bsmm_dtype t, void *stream)
{
    bsmm_status st = check_call(h, N, t);
    if (st != BSMM_OK) return st;
    if (N == 0) return BSMM_OK;
    if (!x || !y || (h->nnz > 0 && !w)) return BSMM_ERR_INVALID;
    if (!aligned16(x) || !aligned16(y) || (h->nnz > 0 && !aligned16(w))) return BSMM_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    if (use_tc(h, t)) {
        st = tc_fprop(h, x, w, y, N, t, s);
        if (st != BSMM_ERR_UNSUPPORTED) return st;
    }
    return simt_fprop(h, x, w, y, N, t, s);
}

bsmm_status bsmm_bprop(bsmm_t h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t, void *stream)
{
    bsmm_status st = check_call(h, N, t);
    if (st != BSMM_OK) return st;
    if (N == 0) return BSMM_OK;
    if (!dy || !dx || (h->nnz > 0 && !w)) return BSMM_ERR_INVALID;
    if (!aligned16(dy) || !aligned16(dx) || (h->nnz > 0 && !aligned16(w))) return BSMM_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    if (use_tc(h, t)) {
        st = tc_bprop(h, dy, w, dx, N, t, s);
        if (st != BSMM_ERR_UNSUPPORTED) return st;
    }
    return simt_bprop(h, dy, w, dx, N, t, s);
}

static bsmm_status updat_common(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, bsmm_dtype t, bsmm_dtype dw_t,
                                int accumulate, cudaStream_t s)
{
    if (h->nnz == 0) return BSMM_OK;
    if (!dw) return BSMM_ERR_INVALID;
    if (!aligned16(dw)) return BSMM_ERR_ALIGN;
    if (N == 0) {
        // An empty minibatch contributes nothing: dw = 0 (or unchanged when accumulating).
        if (accumulate) return BSMM_OK;
        size_t bytes = (size_t)h->nnz * h->bs * h->bs * dtype_size(dw_t);
        return cudaMemsetAsync(dw, 0, bytes, s) == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
    }
    for (int i = 0; i < g.G; ++i) {
        if (!g.x[i] || !g.dy[i]) return BSMM_ERR_INVALID;
        if (!aligned16(g.x[i]) || !aligned16(g.dy[i])) return BSMM_ERR_ALIGN;
    }
    if (use_tc(h, t)) return tc_updat(h, g, dw, N, t, dw_t, accumulate, s);
    return simt_updat(h, g, dw, N, t, dw_t, accumulate, s);
}

bsmm_status bsmm_updat(bsmm_t h, const void *x, const void *dy, void *dw, int N, bsmm_dtype t, bsmm_dtype dw_t,
                       int accumulate, void *stream)
{
    bsmm_status st = check_call(h, N, t);
    if (st != BSMM_OK) return st;
    if (!valid_dtype(dw_t)) return BSMM_ERR_INVALID;
    if (dw_t != BSMM_F32 && dw_t != t) return BSMM_ERR_UNSUPPORTED;
    GroupPtrs g{};
    g.x[0] = x;
    g.dy[0] = dy;
    g.G = 1;
    return updat_common(h, g, dw, N, t, dw_t, accumulate ? 1 : 0, (cudaStream_t)stream);
}

bsmm_status bsmm_updat_grouped(bsmm_t h, const void *const *xs, const void *const *dys, int G, int N, bsmm_dtype t,
                               float *dw, int accumulate, void *stream)
{
    bsmm_status st = check_call(h, N, t);
    if (st != BSMM_OK) return st;
    if (G < 1 || G > 8 || !xs || !dys) return BSMM_ERR_INVALID;
    GroupPtrs g{};
    for (int i = 0; i < G; ++i) {
        g.x[i] = xs[i];
        g.dy[i] = dys[i];
    }
    g.G = G;
    return updat_common(h, g, dw, N, t, BSMM_F32, accumulate ? 1 : 0, (cudaStream_t)stream);
}

bsmm_status bsmm_set_kernel(bsmm_t h, bsmm_kernel which)
{
    if (!h) return BSMM_ERR_INVALID;
    if (which != BSMM_KERNEL_AUTO && which != BSMM_KERNEL_SIMT && which != BSMM_KERNEL_TC) return BSMM_ERR_INVALID;
    h->kernel = which;
    return BSMM_OK;
}

bsmm_status bsmm_sync_status(bsmm_t h, void *stream)
{
    if (!h) return BSMM_ERR_INVALID;
    cudaSetDevice(h->device);
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BSMM_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, h->d_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return BSMM_ERR_CUDA;
    if (v != 0 && cudaMemset(h->d_status, 0, sizeof(int32_t)) != cudaSuccess) return BSMM_ERR_CUDA;
    if (v == BSMM_ERR_TIMEOUT || v == BSMM_ERR_BOUNDS) return (bsmm_status)v;
    return v == 0 ? BSMM_OK : BSMM_ERR_CUDA;
}

const char *bsmm_status_string(bsmm_status s)
{
    switch (s) {
    case BSMM_OK: return "ok";
    case BSMM_ERR_INVALID: return "invalid argument";
    case BSMM_ERR_UNSUPPORTED: return "unsupported block size or dtype combination";
    case BSMM_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case BSMM_ERR_CUDA: return "CUDA error";
    case BSMM_ERR_TIMEOUT: return "device-side wait timed out";
    case BSMM_ERR_OOM: return "device out of memory";
    case BSMM_ERR_BOUNDS: return "device-side index check failed";
    }
    return "unknown status";
}

int64_t bsmm_launch_count(void) { return g_bsmm_launches.load(); }

bsmm_status bsmm_selftest_wait_timeout(bsmm_t h, uint64_t limit_ns, void *stream)
{
    if (!h || limit_ns == 0 || limit_ns > 10000000000ull) return BSMM_ERR_INVALID;
    cudaSetDevice(h->device);
    return launch_wait_selftest(h, limit_ns, (cudaStream_t)stream);
}

bsmm_status bsmm_selftest_empty_launch(bsmm_t h, int ctas, int tensor_memory, void *stream)
{
    if (!h || ctas < 1 || ctas > 65535) return BSMM_ERR_INVALID;
    cudaSetDevice(h->device);
    return launch_empty_selftest(h, ctas, tensor_memory != 0, (cudaStream_t)stream);
}

} // extern "C"
