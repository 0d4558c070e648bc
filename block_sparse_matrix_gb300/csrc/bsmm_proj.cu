// SparseProj: dense <-> sparse feature projections over a one-to-one map (README, "API
// Documentation: blocksparse.matmul", class SparseProj(nhidden, nproj, proj_stride, block_size,
// gather_lut) with gather, scatter, scatter_add and scatter_mul: the TensorFlow gather / scatter
// operations over a unique mapping, so that no output is written twice and no atomics are needed).
//
// The map lut[p] (p < nproj) names the dense feature of sparse feature p; inv[f] is p, or -1 for
// dense features outside the map.  Both live on the device.  Without gather_lut the map keeps runs
// of block_size consecutive features, one run starting every proj_stride features.
//
// Every dense or sparse output element is written by exactly one thread:
//   (F, N) layout (axis 0): a work item is one 16-byte vector of an output row (rows are features);
//   (N, F) layout (axis 1): a work item is 16 bytes of consecutive walked features when both row
//   pitches are multiples of 16 bytes (k_proj_vec), else one element (k_proj_elems).
// Ops whose output is dense (scatter, and scatter_add / scatter_mul out of place) walk the dense
// features and look their source up in inv; gather, gather_mul and the in-place updates walk the
// sparse features through lut.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "bsmm.h"
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

struct bsmm_proj_ctx {
    int nhidden = 0, nproj = 0, device = 0, sm_count = 0;
    int32_t *d_lut = nullptr;     // nproj: dense feature of each sparse feature
    int32_t *d_inv = nullptr;     // nhidden: sparse feature of each dense feature, or -1
    std::vector<int32_t> h_lut;
};

namespace {

constexpr int kPjThreads = 256;

template <typename T> __device__ __forceinline__ float pf(T v);
template <> __device__ __forceinline__ float pf<float>(float v) { return v; }
template <> __device__ __forceinline__ float pf<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float pf<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T pt(float v);
template <> __device__ __forceinline__ float pt<float>(float v) { return v; }
template <> __device__ __forceinline__ __half pt<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 pt<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// The arithmetic of the combining ops, one rounding to T.
template <int OP, typename T> __device__ __forceinline__ T combine(T a, T b)
{
    if (OP == BSMM_PROJ_SCATTER_ADD) return pt<T>(pf<T>(a) + pf<T>(b));
    return pt<T>(pf<T>(a) * pf<T>(b));              // SCATTER_MUL, GATHER_MUL
}

template <int OP, typename T> __device__ __forceinline__ uint4 combine4(uint4 a, uint4 b)
{
    constexpr int E = 16 / sizeof(T);
    const T *ea = reinterpret_cast<const T *>(&a);
    const T *eb = reinterpret_cast<const T *>(&b);
    uint4 r;
    T *er = reinterpret_cast<T *>(&r);
#pragma unroll
    for (int i = 0; i < E; ++i) er[i] = combine<OP, T>(ea[i], eb[i]);
    return r;
}

// Output rows walked by a launch: sparse (through lut) or dense (through inv).
__host__ __device__ __forceinline__ bool walks_sparse(int op, bool in_place)
{
    return op == BSMM_PROJ_GATHER || op == BSMM_PROJ_GATHER_MUL || in_place;
}

// (F, N): rows of N elements, vpr 16-byte vectors each.  items = rows * vpr.
template <int OP, typename T>
__global__ void __launch_bounds__(kPjThreads)
k_proj_rows(const T *x, const T *y, T *out, const int32_t *__restrict__ lut, const int32_t *__restrict__ inv,
            int64_t items, int64_t vpr, int64_t N, int in_place)
{
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    constexpr int E = 16 / sizeof(T);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = blockIdx.x * (int64_t)kPjThreads + threadIdx.x; i < items; i += (int64_t)gridDim.x * kPjThreads) {
        const int64_t r = i / vpr, col = (i - r * vpr) * E;
        auto at = [&](const T *a, int64_t row) { return *reinterpret_cast<const uint4 *>(a + row * N + col); };
        uint4 v;
        int64_t orow = r;
        if (OP == BSMM_PROJ_GATHER) {
            v = at(x, lut[r]);
        } else if (OP == BSMM_PROJ_GATHER_MUL) {
            const int64_t f = lut[r];
            v = combine4<OP, T>(at(x, f), at(y, f));
        } else if (OP == BSMM_PROJ_SCATTER) {
            const int s = inv[r];
            v = s >= 0 ? at(x, s) : zero;
        } else if (in_place) {                      // scatter_add / scatter_mul into x itself
            orow = lut[r];
            v = combine4<OP, T>(at(x, orow), at(y, r));
        } else {
            const int s = inv[r];
            v = s >= 0 ? combine4<OP, T>(at(x, r), at(y, s)) : at(x, r);
        }
        *reinterpret_cast<uint4 *>(out + orow * N + col) = v;
    }
}

// (N, F): one element per item; items = N * cols, cols = the walked features.
template <int OP, typename T>
__global__ void __launch_bounds__(kPjThreads)
k_proj_elems(const T *x, const T *y, T *out, const int32_t *__restrict__ lut, const int32_t *__restrict__ inv,
             int64_t items, int64_t cols, int64_t nhidden, int64_t nproj, int in_place)
{
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)kPjThreads + threadIdx.x; i < items; i += (int64_t)gridDim.x * kPjThreads) {
        const int64_t n = i / cols, c = i - n * cols;
        const int64_t dn = n * nhidden, sn = n * nproj;   // starts of sample n's dense / sparse row
        if (OP == BSMM_PROJ_GATHER) {
            out[sn + c] = x[dn + lut[c]];
        } else if (OP == BSMM_PROJ_GATHER_MUL) {
            const int64_t f = lut[c];
            out[sn + c] = combine<OP, T>(x[dn + f], y[dn + f]);
        } else if (OP == BSMM_PROJ_SCATTER) {
            const int s = inv[c];
            out[dn + c] = s >= 0 ? x[sn + s] : pt<T>(0.f);
        } else if (in_place) {
            const int64_t f = lut[c];
            out[dn + f] = combine<OP, T>(x[dn + f], y[sn + c]);
        } else {
            const int s = inv[c];
            out[dn + c] = s >= 0 ? combine<OP, T>(x[dn + c], y[sn + s]) : x[dn + c];
        }
    }
}


// (N, F) with both row pitches a multiple of 16 bytes: an item is E = 16 / sizeof(T) consecutive
// walked features of one sample.  Their E map entries are read as one vector; when they name E
// consecutive features starting on a 16-byte boundary (runs of the default map, identity-like
// stretches of a given one) the source moves as one 16-byte vector, otherwise element by element.
// The output always moves as one vector except for the scattered in-place update of a broken run.
template <int OP, typename T>
__global__ void __launch_bounds__(kPjThreads)
k_proj_vec(const T *x, const T *y, T *out, const int32_t *__restrict__ lut, const int32_t *__restrict__ inv,
           int64_t items, int64_t vpr, int64_t nhidden, int64_t nproj, int in_place)
{
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    constexpr int E = 16 / sizeof(T);
    const bool sparse_walk = OP == BSMM_PROJ_GATHER || OP == BSMM_PROJ_GATHER_MUL || in_place;
    const int32_t *map = sparse_walk ? lut : inv;
    for (int64_t i = blockIdx.x * (int64_t)kPjThreads + threadIdx.x; i < items; i += (int64_t)gridDim.x * kPjThreads) {
        const int64_t n = i / vpr, c0 = (i - n * vpr) * E;
        const int64_t dn = n * nhidden, sn = n * nproj;
        int idx[E];
#pragma unroll
        for (int q = 0; q < E; q += 4) *reinterpret_cast<int4 *>(idx + q) = *reinterpret_cast<const int4 *>(map + c0 + q);
        bool run = (idx[0] % E) == 0, none = true;
#pragma unroll
        for (int q = 0; q < E; ++q) {
            run = run && idx[q] == idx[0] + q;
            none = none && idx[q] < 0;
        }
        run = run && idx[0] >= 0;
        auto vec = [](const T *a) { return *reinterpret_cast<const uint4 *>(a); };
        uint4 v;
        T *ev = reinterpret_cast<T *>(&v);
        if (OP == BSMM_PROJ_GATHER || OP == BSMM_PROJ_GATHER_MUL) {
            if (run) {
                v = vec(x + dn + idx[0]);
                if (OP == BSMM_PROJ_GATHER_MUL) v = combine4<OP, T>(v, vec(y + dn + idx[0]));
            } else {
#pragma unroll
                for (int q = 0; q < E; ++q)
                    ev[q] = OP == BSMM_PROJ_GATHER ? x[dn + idx[q]] : combine<OP, T>(x[dn + idx[q]], y[dn + idx[q]]);
            }
            *reinterpret_cast<uint4 *>(out + sn + c0) = v;
        } else if (OP == BSMM_PROJ_SCATTER) {
            if (none) {
                v = make_uint4(0u, 0u, 0u, 0u);
            } else if (run) {
                v = vec(x + sn + idx[0]);
            } else {
#pragma unroll
                for (int q = 0; q < E; ++q) ev[q] = idx[q] >= 0 ? x[sn + idx[q]] : pt<T>(0.f);
            }
            *reinterpret_cast<uint4 *>(out + dn + c0) = v;
        } else if (in_place) {                      // scatter_add / scatter_mul into x itself
            const uint4 b = vec(y + sn + c0);
            if (run) {
                *reinterpret_cast<uint4 *>(out + dn + idx[0]) = combine4<OP, T>(vec(x + dn + idx[0]), b);
            } else {
                const T *eb = reinterpret_cast<const T *>(&b);
#pragma unroll
                for (int q = 0; q < E; ++q) out[dn + idx[q]] = combine<OP, T>(x[dn + idx[q]], eb[q]);
            }
        } else {
            v = vec(x + dn + c0);
            if (run) {
                v = combine4<OP, T>(v, vec(y + sn + idx[0]));
            } else if (!none) {
#pragma unroll
                for (int q = 0; q < E; ++q)
                    if (idx[q] >= 0) ev[q] = combine<OP, T>(ev[q], y[sn + idx[q]]);
            }
            *reinterpret_cast<uint4 *>(out + dn + c0) = v;
        }
    }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_pj(void (*kern)(KArgs...), int grid, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPjThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int OP, typename T>
cudaError_t launch_op(bsmm_proj_ctx *p, const void *x, const void *y, void *out, int N, int axis, bool in_place,
                      cudaStream_t s)
{
    const int64_t cols = walks_sparse(OP, in_place) ? p->nproj : p->nhidden;
    const T *xt = static_cast<const T *>(x), *yt = static_cast<const T *>(y);
    T *ot = static_cast<T *>(out);
    int64_t items;
    if (axis == 0) {
        const int64_t vpr = (int64_t)N / (16 / (int)sizeof(T));
        items = cols * vpr;
        const int grid = (int)std::min<int64_t>((items + kPjThreads - 1) / kPjThreads, (int64_t)p->sm_count * 16);
        return launch_pdl_pj(k_proj_rows<OP, T>, std::max(grid, 1), s, xt, yt, ot, (const int32_t *)p->d_lut,
                             (const int32_t *)p->d_inv, items, vpr, (int64_t)N, (int)in_place);
    }
    constexpr int E = 16 / (int)sizeof(T);
    if ((p->nhidden % E) == 0 && (p->nproj % E) == 0) {       // both row pitches 16-byte multiples
        const int64_t vpr = cols / E;
        items = (int64_t)N * vpr;
        const int grid = (int)std::min<int64_t>((items + kPjThreads - 1) / kPjThreads, (int64_t)p->sm_count * 16);
        return launch_pdl_pj(k_proj_vec<OP, T>, std::max(grid, 1), s, xt, yt, ot, (const int32_t *)p->d_lut,
                             (const int32_t *)p->d_inv, items, vpr, (int64_t)p->nhidden, (int64_t)p->nproj,
                             (int)in_place);
    }
    items = cols * (int64_t)N;
    const int grid = (int)std::min<int64_t>((items + kPjThreads - 1) / kPjThreads, (int64_t)p->sm_count * 16);
    return launch_pdl_pj(k_proj_elems<OP, T>, std::max(grid, 1), s, xt, yt, ot, (const int32_t *)p->d_lut,
                         (const int32_t *)p->d_inv, items, cols, (int64_t)p->nhidden, (int64_t)p->nproj,
                         (int)in_place);
}

template <typename T>
cudaError_t launch_t(bsmm_proj_ctx *p, int op, const void *x, const void *y, void *out, int N, int axis,
                     bool in_place, cudaStream_t s)
{
    switch (op) {
    case BSMM_PROJ_GATHER: return launch_op<BSMM_PROJ_GATHER, T>(p, x, y, out, N, axis, in_place, s);
    case BSMM_PROJ_SCATTER: return launch_op<BSMM_PROJ_SCATTER, T>(p, x, y, out, N, axis, in_place, s);
    case BSMM_PROJ_SCATTER_ADD: return launch_op<BSMM_PROJ_SCATTER_ADD, T>(p, x, y, out, N, axis, in_place, s);
    case BSMM_PROJ_SCATTER_MUL: return launch_op<BSMM_PROJ_SCATTER_MUL, T>(p, x, y, out, N, axis, in_place, s);
    default: return launch_op<BSMM_PROJ_GATHER_MUL, T>(p, x, y, out, N, axis, in_place, s);
    }
}

} // namespace

extern "C" bsmm_status bsmm_proj_create(bsmm_proj_t *out, int nhidden, int nproj, int proj_stride, int block_size,
                                        const int32_t *gather_lut)
{
    if (!out || nhidden < 1) return BSMM_ERR_INVALID;
    *out = nullptr;
    std::vector<int32_t> lut;
    if (gather_lut) {
        if (nproj < 1 || nproj > nhidden) return BSMM_ERR_INVALID;
        lut.assign(gather_lut, gather_lut + nproj);
    } else {
        if (block_size < 1) return BSMM_ERR_INVALID;
        const int stride = proj_stride > 0 ? proj_stride : block_size;
        if (stride < block_size || nhidden < block_size) return BSMM_ERR_INVALID;
        const int64_t runs = nproj > 0 ? nproj / block_size : (int64_t)(nhidden - block_size) / stride + 1;
        if (nproj > 0 && nproj % block_size) return BSMM_ERR_INVALID;
        if (runs < 1 || (runs - 1) * stride + block_size > nhidden) return BSMM_ERR_INVALID;
        nproj = (int)(runs * block_size);
        lut.resize(nproj);
        for (int q = 0; q < nproj; ++q) lut[q] = (q / block_size) * stride + q % block_size;
    }
    std::vector<int32_t> inv(nhidden, -1);
    for (int q = 0; q < nproj; ++q) {               // one to one: in range and distinct
        if (lut[q] < 0 || lut[q] >= nhidden || inv[lut[q]] >= 0) return BSMM_ERR_INVALID;
        inv[lut[q]] = q;
    }
    bsmm_proj_ctx *p = new bsmm_proj_ctx;
    p->nhidden = nhidden;
    p->nproj = nproj;
    p->h_lut = lut;
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        delete p;
        return BSMM_ERR_CUDA;
    }
    if (cudaMalloc(&p->d_lut, sizeof(int32_t) * nproj) != cudaSuccess ||
        cudaMalloc(&p->d_inv, sizeof(int32_t) * nhidden) != cudaSuccess) {
        cudaFree(p->d_lut);
        cudaFree(p->d_inv);
        delete p;
        return BSMM_ERR_OOM;
    }
    if (cudaMemcpy(p->d_lut, lut.data(), sizeof(int32_t) * nproj, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(p->d_inv, inv.data(), sizeof(int32_t) * nhidden, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(p->d_lut);
        cudaFree(p->d_inv);
        delete p;
        return BSMM_ERR_CUDA;
    }
    *out = p;
    return BSMM_OK;
}

extern "C" bsmm_status bsmm_proj_destroy(bsmm_proj_t p)
{
    if (!p) return BSMM_OK;
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    cudaFree(p->d_lut);
    cudaFree(p->d_inv);
    delete p;
    return BSMM_OK;
}

extern "C" bsmm_status bsmm_proj_info(bsmm_proj_t p, int *nhidden, int *nproj)
{
    if (!p) return BSMM_ERR_INVALID;
    if (nhidden) *nhidden = p->nhidden;
    if (nproj) *nproj = p->nproj;
    return BSMM_OK;
}

extern "C" bsmm_status bsmm_proj_get_lut(bsmm_proj_t p, int32_t *lut)
{
    if (!p || !lut) return BSMM_ERR_INVALID;
    std::copy(p->h_lut.begin(), p->h_lut.end(), lut);
    return BSMM_OK;
}

extern "C" bsmm_status bsmm_proj(bsmm_proj_t p, bsmm_proj_op op, const void *x, const void *y, void *out, int N,
                                 int axis, bsmm_dtype t, void *stream)
{
    if (!p || N < 0 || (axis != 0 && axis != 1)) return BSMM_ERR_INVALID;
    if (op < BSMM_PROJ_GATHER || op > BSMM_PROJ_GATHER_MUL) return BSMM_ERR_INVALID;
    if (t != BSMM_F32 && t != BSMM_F16 && t != BSMM_BF16) return BSMM_ERR_INVALID;
    if (N == 0) return BSMM_OK;                       // no samples: nothing is read or written
    const bool needs_y = op == BSMM_PROJ_SCATTER_ADD || op == BSMM_PROJ_SCATTER_MUL || op == BSMM_PROJ_GATHER_MUL;
    if (!x || !out || (needs_y && !y)) return BSMM_ERR_INVALID;
    const bool in_place = out == x;
    if (in_place && op != BSMM_PROJ_SCATTER_ADD && op != BSMM_PROJ_SCATTER_MUL) return BSMM_ERR_INVALID;
    if (needs_y && out == y) return BSMM_ERR_INVALID;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) |
                          reinterpret_cast<uintptr_t>(needs_y ? y : x);
    if (mis & 15u) return BSMM_ERR_ALIGN;
    const int e = t == BSMM_F32 ? 4 : 2;
    if (axis == 0 && ((int64_t)N * e) % 16) return BSMM_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSMM_ERR_CUDA;
    if (dev != p->device && cudaSetDevice(p->device) != cudaSuccess) return BSMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (t == BSMM_F32) err = launch_t<float>(p, op, x, y, out, N, axis, in_place, s);
    else if (t == BSMM_F16) err = launch_t<__half>(p, op, x, y, out, N, axis, in_place, s);
    else err = launch_t<__nv_bfloat16>(p, op, x, y, out, N, axis, in_place, s);
    g_bsmm_launches += 1;
    return err == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}
