// layer_norm for both activation layouts of the block-sparse matmul (README, section
// "blocksparse.norms": a layernorm supporting both bsmm feature_axis layouts, with an
// optional relu applied at the end).  For every sample n the C features are normalised with
// their mean and biased variance, scaled by g and shifted by b:
//     y[n][f] = g[f] * (x[n][f] - mean_n) / sqrt(var_n + epsilon) + b[f]   (then max(y, 0)).
// Statistics in float32 (mean first, then the mean of the squared deviations), one rounding
// of y to the input type.
//
//   axis = 1, (N, C) rows:  k_ln_rows, one CTA per sample; the row stays in registers between
//                           the two reductions and the output pass, so x is read once.
//   axis = 0, (C, N):       k_ln_cols, a cluster of kLnSplit CTAs per tile of 64 samples
//                           (columns); CTA r reduces its share of the C rows, the partial sums
//                           are exchanged in distributed shared memory and every CTA adds them
//                           in the same (rank) order, so all CTAs of a cluster use identical
//                           statistics.  x is re-read for the second and third pass (from L2).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "bsmm.h"
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kLnThreads = 256;
constexpr int kLnMaxC = 16384;          // axis = 1: at most 16 vectors of 16 bytes per thread
constexpr int kLnSplit = 8;             // axis = 0: CTAs per cluster along the features
constexpr int kLnCols = 64;             // axis = 0: samples (columns) per cluster
constexpr int kLnCacheMax = 160 * 1024; // axis = 0: dynamic shared memory of a CTA (slice + g, b)

template <typename T> __device__ __forceinline__ float ld1(const T *p);
template <> __device__ __forceinline__ float ld1<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld1<__half>(const __half *p) { return __half2float(*p); }
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ T st1(float v);
template <> __device__ __forceinline__ float st1<float>(float v) { return v; }
template <> __device__ __forceinline__ __half st1<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 st1<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Sum over the CTA (kLnThreads threads); every thread gets the total.  `red` has one slot per warp.
__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    __syncthreads();                                   // red may still be read by a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kLnThreads / 32; ++w) s += red[w];
    return s;
}

// axis = 1: one CTA per row of C features.  Thread t holds the 16-byte vectors t, t + 256, ...,
// IT of them (IT * 256 * VEC >= C, chosen per call so short rows need few registers).
template <typename T, int IT>
__global__ void __launch_bounds__(kLnThreads) k_ln_rows(const T *__restrict__ x, const float *__restrict__ g,
                                                        const float *__restrict__ b, T *y, int C, float eps,
                                                        int relu)
{
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float red[kLnThreads / 32];
    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    tc::pdl_wait();                                    // the previous kernel's writes are visible
    const T *xr = x + (size_t)blockIdx.x * C;
    T *yr = y + (size_t)blockIdx.x * C;
    float v[IT][VEC];
    float s = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(xr + f0);
            const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                v[it][j] = ld1<T>(e + j);
                s += v[it][j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) v[it][j] = 0.f;
        }
    }
    const float mean = block_sum(s, red) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const float d = v[it][j] - mean;
                q += d * d;
            }
        }
    }
    const float rstd = rsqrtf(block_sum(q, red) / (float)C + eps);
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
            float gv[VEC], bv[VEC];
#pragma unroll
            for (int j = 0; j < VEC; j += 4) {          // g, b are 16-byte aligned and f0 % VEC == 0
                *reinterpret_cast<float4 *>(gv + j) = *reinterpret_cast<const float4 *>(g + f0 + j);
                *reinterpret_cast<float4 *>(bv + j) = *reinterpret_cast<const float4 *>(b + f0 + j);
            }
            uint4 raw;
            T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                float o = gv[j] * ((v[it][j] - mean) * rstd) + bv[j];
                if (relu) o = fmaxf(o, 0.f);
                e[j] = st1<T>(o);
            }
            *reinterpret_cast<uint4 *>(yr + f0) = raw;
        }
    }
}

// Sum of element idx of the kLnSplit = 8 CTAs' partial buffers at `part` (shared memory of
// each CTA of the cluster), in rank order.  The eight remote loads are issued together.
__device__ __forceinline__ float cluster_sum(const float *part, int idx)
{
    static_assert(kLnSplit == 8, "one load per CTA of the cluster");
    uint32_t a[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) a[r] = tc::map_to_rank(tc::smem_u32(part + idx), (uint32_t)r);
    float t[8];
    asm volatile("ld.shared::cluster.f32 %0, [%8];\n\tld.shared::cluster.f32 %1, [%9];\n\t"
                 "ld.shared::cluster.f32 %2, [%10];\n\tld.shared::cluster.f32 %3, [%11];\n\t"
                 "ld.shared::cluster.f32 %4, [%12];\n\tld.shared::cluster.f32 %5, [%13];\n\t"
                 "ld.shared::cluster.f32 %6, [%14];\n\tld.shared::cluster.f32 %7, [%15];"
                 : "=f"(t[0]), "=f"(t[1]), "=f"(t[2]), "=f"(t[3]), "=f"(t[4]), "=f"(t[5]), "=f"(t[6]), "=f"(t[7])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7])
                 : "memory");
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) s += t[r];
    return s;
}

// 16 bytes of 8 consecutive elements (two float4 for float).
template <typename T> struct Vec8 {
    uint4 u[sizeof(T) / 2];
};

// 16-byte asynchronous global -> shared copy (completion: cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <typename T> __device__ __forceinline__ void unpack8(const Vec8<T> &v, float (&f)[8])
{
    const T *e = reinterpret_cast<const T *>(&v);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = ld1<T>(e + j);
}

// axis = 0: (C, N).  A cluster of kLnSplit CTAs owns kLnCols = 64 consecutive samples
// (columns); CTA r takes rows [r * rows, (r + 1) * rows).  Thread t reads 8 consecutive columns
// (cc = t % 8) of rows rg, rg + 32, ... (rg = t / 8), so a warp reads 4 rows of 128 bytes per
// instruction.  The CTA's slice is kept in shared memory (CACHE), so x is read from memory
// once; the second and third pass (squared deviations, output) read the slice.
template <typename T, bool CACHE>
__global__ void __cluster_dims__(kLnSplit, 1, 1) __launch_bounds__(kLnThreads)
k_ln_cols(const T *__restrict__ x, const float *__restrict__ g, const float *__restrict__ b, T *y, int C, int N,
          float eps, int relu)
{
    extern __shared__ __align__(16) uint8_t ln_smem[];
    Vec8<T> *slice = reinterpret_cast<Vec8<T> *>(ln_smem);          // [rows][8] vectors (CACHE)
    __shared__ float acc[kLnThreads / 8][kLnCols];                    // per row group, per column
    __shared__ float part1[kLnCols], part2[kLnCols];                  // this CTA's partial sums
    __shared__ float stat[2][kLnCols];                                // cluster-wide mean, 1 / std
    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    tc::pdl_wait();                                    // the previous kernel's writes are visible
    const uint32_t rank = tc::cluster_ctarank();
    const int tile = blockIdx.x / kLnSplit;
    const int rg = threadIdx.x / 8, cc = threadIdx.x & 7;
    const int n0 = tile * kLnCols + cc * 8;                            // first of this thread's 8 columns
    const bool has = n0 < N;                                           // N % 8 == 0: all 8 or none
    const int rows = (C + kLnSplit - 1) / kLnSplit;
    const int r0 = (int)rank * rows, r1 = min(C, r0 + rows);
    const int nr = max(0, r1 - r0);
    constexpr int RG = kLnThreads / 8;                                 // 32 row groups
    // g, b of this CTA's rows, staged once so the output pass does not wait on them per row
    float *sg = reinterpret_cast<float *>(ln_smem + (CACHE ? (size_t)rows * sizeof(Vec8<T>) * 8 : 0));
    float *sb = sg + rows;
    for (int i = threadIdx.x; i < nr; i += kLnThreads) {
        sg[i] = g[r0 + i];
        sb[i] = b[r0 + i];
    }
    auto gload = [&](int f) { return *reinterpret_cast<const Vec8<T> *>(x + (size_t)f * N + n0); };

    // pass 1: sums.  With CACHE the whole slice is first copied to shared memory with
    // asynchronous copies, all in flight at once.
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (CACHE) {
        if (has)
            for (int i = rg; i < nr; i += RG) {
                const T *src = x + (size_t)(r0 + i) * N + n0;
#pragma unroll
                for (int h = 0; h < (int)(sizeof(Vec8<T>) / 16); ++h)
                    cp_async16(reinterpret_cast<uint8_t *>(&slice[i * 8 + cc]) + 16 * h,
                               reinterpret_cast<const uint8_t *>(src) + 16 * h);
            }
        cp_async_wait_all();                           // this thread's copies have landed
        if (has)
            for (int i = rg; i < nr; i += RG) {        // each thread reads back only its own copies
                float f[8];
                unpack8<T>(slice[i * 8 + cc], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] += f[j];
            }
    } else if (has) {
        int i = rg;
        for (; i + 3 * RG < nr; i += 4 * RG) {                        // four independent loads in flight
            Vec8<T> v4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v4[u] = gload(r0 + i + u * RG);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float f[8];
                unpack8<T>(v4[u], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] += f[j];
            }
        }
        for (; i < nr; i += RG) {
            const Vec8<T> v = gload(r0 + i);
            float f[8];
            unpack8<T>(v, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] += f[j];
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[rg][cc * 8 + j] = s[j];
    __syncthreads();
    if (threadIdx.x < kLnCols) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part1[threadIdx.x] = t;
    }
    tc::cluster_sync();                                // every CTA's part1 is written
    if (threadIdx.x < kLnCols) stat[0][threadIdx.x] = cluster_sum(part1, threadIdx.x) / (float)C;
    __syncthreads();
    float mean[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mean[j] = stat[0][cc * 8 + j];

    // pass 2: squared deviations
    float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (has)
        for (int i = rg; i < nr; i += RG) {
            float f[8];
            unpack8<T>(CACHE ? slice[i * 8 + cc] : gload(r0 + i), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float d = f[j] - mean[j];
                q[j] += d * d;
            }
        }
    __syncthreads();                                   // acc of pass 1 has been read
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[rg][cc * 8 + j] = q[j];
    __syncthreads();
    if (threadIdx.x < kLnCols) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part2[threadIdx.x] = t;
    }
    tc::cluster_sync();                                // every CTA's part2 is written
    if (threadIdx.x < kLnCols) stat[1][threadIdx.x] = rsqrtf(cluster_sum(part2, threadIdx.x) / (float)C + eps);
    __syncthreads();
    float rstd[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rstd[j] = stat[1][cc * 8 + j];

    // pass 3: normalise this CTA's rows
    if (has)
        for (int i = rg; i < nr; i += RG) {
            const int f = r0 + i;
            float v[8];
            unpack8<T>(CACHE ? slice[i * 8 + cc] : gload(f), v);
            const float gf = sg[i], bf = sb[i];
            Vec8<T> o;
            T *e = reinterpret_cast<T *>(&o);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float t = gf * ((v[j] - mean[j]) * rstd[j]) + bf;
                if (relu) t = fmaxf(t, 0.f);
                e[j] = st1<T>(t);
            }
            *reinterpret_cast<Vec8<T> *>(y + (size_t)f * N + n0) = o;
        }
    tc::cluster_sync();                                // no CTA leaves while a peer reads its partials
}


// Launch with programmatic stream serialisation: the kernel's launch overlaps the previous
// kernel's tail; it waits in griddepcontrol.wait before reading anything.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_ln(void (*kern)(KArgs...), int grid, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kLnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T, int IT>
cudaError_t launch_rows(const void *x, const float *g, const float *b, void *y, int N, int C, float eps, int relu,
                        cudaStream_t s)
{
    return launch_pdl_ln(k_ln_rows<T, IT>, N, 0, s, static_cast<const T *>(x), g, b, static_cast<T *>(y), C, eps,
                         relu);
}

template <typename T>
cudaError_t launch_ln(const void *x, const float *g, const float *b, void *y, int N, int C, int axis, float eps,
                      int relu, cudaStream_t s)
{
    cudaError_t le;
    if (axis == 1) {
        const int need = (C + kLnThreads * (16 / (int)sizeof(T)) - 1) / (kLnThreads * (16 / (int)sizeof(T)));
        if (need <= 1) le = launch_rows<T, 1>(x, g, b, y, N, C, eps, relu, s);
        else if (need <= 2) le = launch_rows<T, 2>(x, g, b, y, N, C, eps, relu, s);
        else if (need <= 4) le = launch_rows<T, 4>(x, g, b, y, N, C, eps, relu, s);
        else if (need <= 8) le = launch_rows<T, 8>(x, g, b, y, N, C, eps, relu, s);
        else le = launch_rows<T, 16>(x, g, b, y, N, C, eps, relu, s);
    } else {
        const int tiles = (N + kLnCols - 1) / kLnCols;
        const int rows = (C + kLnSplit - 1) / kLnSplit;
        const size_t slice = (size_t)rows * kLnCols * sizeof(T);
        const size_t gb = (size_t)rows * 2 * sizeof(float);             // staged g, b
        if (slice + gb <= (size_t)kLnCacheMax) {
            auto kern = k_ln_cols<T, true>;
            static std::atomic<int> attr_set{-1};      // device whose limit has been raised
            int dev = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return e;
            if (attr_set.load() != dev) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLnCacheMax);
                if (e != cudaSuccess) return e;
                attr_set.store(dev);
            }
            le = launch_pdl_ln(kern, tiles * kLnSplit, slice + gb, s, static_cast<const T *>(x), g, b,
                               static_cast<T *>(y), C, N, eps, relu);
        } else {
            auto kern = k_ln_cols<T, false>;
            static std::atomic<int> attr_set{-1};
            int dev = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return e;
            if (attr_set.load() != dev) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLnCacheMax);
                if (e != cudaSuccess) return e;
                attr_set.store(dev);
            }
            if (gb > (size_t)kLnCacheMax) return cudaErrorInvalidValue;   // C beyond 8 x 20480 rows
            le = launch_pdl_ln(kern, tiles * kLnSplit, gb, s, static_cast<const T *>(x), g, b, static_cast<T *>(y), C,
                               N, eps, relu);
        }
    }
    g_bsmm_launches += 1;
    return le;
}

} // namespace

extern "C" bsmm_status bsmm_layer_norm(const void *x, const float *g, const float *b, void *y, int N, int C,
                                       int axis, float epsilon, int relu, bsmm_dtype t, void *stream)
{
    if (N < 0 || C < 1 || (axis != 0 && axis != 1) || !(epsilon >= 0.f)) return BSMM_ERR_INVALID;
    if (t != BSMM_F32 && t != BSMM_F16 && t != BSMM_BF16) return BSMM_ERR_INVALID;
    if (N == 0) return BSMM_OK;                        // no samples: nothing is read or written
    if (!x || !g || !b || !y) return BSMM_ERR_INVALID;
    const size_t e = t == BSMM_F32 ? 4 : 2;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                          reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(b);
    if (mis & 15u) return BSMM_ERR_ALIGN;
    if (((size_t)(axis == 1 ? C : N) * e) % 16u) return BSMM_ERR_ALIGN;
    if (axis == 0 && N % 8) return BSMM_ERR_ALIGN;     // (C, N): 8 samples per thread
    if (axis == 1 && C > kLnMaxC) return BSMM_ERR_UNSUPPORTED;
    if (axis == 0 && (size_t)((C + kLnSplit - 1) / kLnSplit) * 2 * sizeof(float) > (size_t)kLnCacheMax)
        return BSMM_ERR_UNSUPPORTED;                   // the staged g, b of a CTA's rows must fit
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (t == BSMM_F32) err = launch_ln<float>(x, g, b, y, N, C, axis, epsilon, relu, s);
    else if (t == BSMM_F16) err = launch_ln<__half>(x, g, b, y, N, C, axis, epsilon, relu, s);
    else err = launch_ln<__nv_bfloat16>(x, g, b, y, N, C, axis, epsilon, relu, s);
    return err == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}
