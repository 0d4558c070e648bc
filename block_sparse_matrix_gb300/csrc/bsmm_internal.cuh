// Internal declarations shared by the libbsmm translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <vector>

#include "bsmm.h"

// Per-handle state.  Device tables are built once by bsmm_create and then only read.
struct bsmm_ctx {
    int R = 0, S = 0, bs = 0, fa = 1;
    int64_t nnz = 0;
    int device = 0;
    int sm_count = 0;
    bsmm_kernel kernel = BSMM_KERNEL_AUTO;

    uint8_t *d_layout = nullptr;   // R*S
    int32_t *d_row_ptr = nullptr;  // R+1
    int32_t *d_row_ent = nullptr;  // nnz: k of each block (row-major order)
    int32_t *d_col_ptr = nullptr;  // S+1
    int32_t *d_col_ent = nullptr;  // 2*nnz: (block id, c) per column, c increasing
    int32_t *d_coord = nullptr;    // 2*nnz: (c, k) per block id
    int32_t *d_bid = nullptr;      // R*S: block id or -1
    int32_t *d_status = nullptr;   // sticky device error word

    // Host mirrors of the tables (block_coord lookups, tensor-core schedules).
    std::vector<int32_t> h_row_ptr, h_row_ent, h_col_ptr, h_col_ent, h_coord;

    // Tensor-core schedules (built lazily by the tcgen05 path).
    void *tc = nullptr;
    void *sp = nullptr;        // sparse-window kernel plans and (F, N) panel scratch (bsmm_sp.cu)
    int tc_wlog = -1;   // fprop/bprop window size override (log2), from BSMM_TC_WLOG; -1 = automatic
    int tc_stage_kb = -1;  // fprop/bprop per-CTA stage budget override (KB), from BSMM_TC_STAGE_KB
    int tc_rows = -1;      // window-kernel minibatch tile height override (64 or 128), from BSMM_TC_ROWS
    int tc_bins = -1;      // window kernel: 1 forces binned windows, 0 forbids them, from BSMM_TC_BINS
    int tc_eslots = -1;    // window kernel: activation panels per chunk override (1..8), from BSMM_TC_ESLOTS
};

extern std::atomic<int64_t> g_bsmm_launches;

static inline int dtype_size(bsmm_dtype t) { return t == BSMM_F32 ? 4 : 2; }

#define BSMM_CUDA_TRY(expr)                              \
    do {                                                 \
        cudaError_t e_ = (expr);                         \
        if (e_ != cudaSuccess) return BSMM_ERR_CUDA;     \
    } while (0)

// Grouped-gradient pointer pack, passed by value to kernels.
struct GroupPtrs {
    const void *x[8];
    const void *dy[8];
    int G;
};

// LUT / init kernels (bsmm_lut.cu)
bsmm_status lut_build(bsmm_ctx *h, const uint8_t *layout_host, cudaStream_t s);
bsmm_status launch_identity_init(bsmm_ctx *h, void *w, bsmm_dtype t, cudaStream_t s);
bsmm_status launch_zero(void *p, size_t bytes, cudaStream_t s);

// IEEE SIMT kernels, any dtype (bsmm_simt.cu)
bsmm_status simt_fprop(bsmm_ctx *h, const void *x, const void *w, void *y, int N, bsmm_dtype t,
                       cudaStream_t s);
bsmm_status simt_bprop(bsmm_ctx *h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t,
                       cudaStream_t s);
bsmm_status simt_updat(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, bsmm_dtype t,
                       bsmm_dtype dw_t, int accumulate, cudaStream_t s);

// tcgen05 tensor-core kernels, 16-bit inputs (bsmm_tc.cu)
bool tc_supported(bsmm_ctx *h, bsmm_dtype t);
bsmm_status tc_fprop(bsmm_ctx *h, const void *x, const void *w, void *y, int N, bsmm_dtype t,
                     cudaStream_t s);
bsmm_status tc_bprop(bsmm_ctx *h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t,
                     cudaStream_t s);
bsmm_status tc_updat(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, bsmm_dtype t, bsmm_dtype dw_t,
                     int accumulate, cudaStream_t s);
void tc_release(bsmm_ctx *h);

// Sparse-window fprop/bprop with the activation operand in tensor memory (bsmm_sp.cu).
bool sp_supported(const bsmm_ctx *h, bsmm_dtype t);
bsmm_status sp_fb(bsmm_ctx *h, bool bwd, const void *act, const void *w, void *out, int N, bsmm_dtype t,
                  cudaStream_t s);
void sp_release(bsmm_ctx *h);
bsmm_status launch_wait_selftest(bsmm_ctx *h, uint64_t limit_ns, cudaStream_t s);
bsmm_status launch_empty_selftest(bsmm_ctx *h, int ctas, bool tensor_memory, cudaStream_t s);
