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
//
// Gradient (bsmm_layer_norm_grad): with xh = (x - mean_n) * rstd_n, dz = dy (zero where the
// forward output y <= 0 when relu), a = g * dz,
//     dx = rstd_n * (a - mean_f(a) - xh * mean_f(a * xh)),  dg[f] = sum_n dz * xh,  db[f] = sum_n dz.
//   axis = 1: k_lng_rows, one CTA per sample, computes dx and stores the sample's mean and rstd;
//             k_lng_colsum then sums dz * xh and dz per feature over chunks of samples (the
//             inputs are still in L2) into one partial set per chunk.
//   axis = 0: k_lng_cols, the cluster layout of k_ln_cols with two more cluster sums (of a and
//             a * xh), the x, dy, y slices in shared memory; each cluster writes per-feature
//             partials of its 64 samples.
//   k_lng_reduce adds the partial sets in a fixed order (deterministic dg, db).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>

#include "bsmm.h"
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kLnThreads = 256;
constexpr int kLnMaxC = 16384;          // axis = 1: at most 16 vectors of 16 bytes per thread
constexpr int kLnSplit = 8;             // axis = 0: CTAs per cluster along the features
constexpr int kLnCols = 64;             // axis = 0: samples (columns) per cluster (32 measured slower)
constexpr int kLnCacheMax = 160 * 1024; // axis = 0: dynamic shared memory of a CTA (slice + g, b)
constexpr int kLngCacheMax = 66 * 1024;  // axis = 0 gradient: cached slices + g (three CTAs per SM)
constexpr int kLngCols = 32;            // axis = 0 gradient: samples (columns) per cluster

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

// RPC sums over the CTA at once (kLnThreads threads); every thread gets the totals.  `red` has
// RPC slots per warp.  Two barriers for all RPC sums.
template <int RPC>
__device__ __forceinline__ void block_sums(float (&v)[RPC], float *red)
{
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < RPC; ++r)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
    __syncthreads();                                   // red may still be read by a previous call
    if (lane == 0)
#pragma unroll
        for (int r = 0; r < RPC; ++r) red[warp * RPC + r] = v[r];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPC; ++r) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kLnThreads / 32; ++w) s += red[w * RPC + r];
        v[r] = s;
    }
}

// axis = 1: a CTA normalises RPC consecutive rows of C features.  Thread t holds the 16-byte
// vectors t, t + 256, ..., IT of them per row (IT * 256 * VEC >= C, chosen per call so short rows
// need few registers); all RPC rows' loads are issued before the first sum, and the RPC rows'
// sums share each pair of barriers.
template <typename T, int IT, int RPC>
__global__ void __launch_bounds__(kLnThreads) k_ln_rows(const T *__restrict__ x, const float *__restrict__ g,
                                                        const float *__restrict__ b, T *y, int N, int C, float eps,
                                                        int relu)
{
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float red[RPC * kLnThreads / 32];
    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    tc::pdl_wait();                                    // the previous kernel's writes are visible
    const int n0 = blockIdx.x * RPC;
    float v[RPC][IT][VEC];
    float s[RPC];
#pragma unroll
    for (int r = 0; r < RPC; ++r) {
        s[r] = 0.f;
        const bool live = n0 + r < N;
        const T *xr = x + (size_t)(n0 + r) * C;
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            if (live && f0 < C) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(xr + f0);
                const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
                for (int j = 0; j < VEC; ++j) v[r][it][j] = ld1<T>(e + j);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j) v[r][it][j] = 0.f;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPC; ++r)
#pragma unroll
        for (int it = 0; it < IT; ++it)
#pragma unroll
            for (int j = 0; j < VEC; ++j) s[r] += v[r][it][j];
    block_sums<RPC>(s, red);
    float mean[RPC], q[RPC];
#pragma unroll
    for (int r = 0; r < RPC; ++r) {
        mean[r] = s[r] / (float)C;
        q[r] = 0.f;
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            if (f0 < C) {
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float d = v[r][it][j] - mean[r];
                    q[r] += d * d;
                }
            }
        }
    }
    block_sums<RPC>(q, red);
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
#pragma unroll
            for (int r = 0; r < RPC; ++r) {
                if (n0 + r >= N) continue;
                const float rstd = rsqrtf(q[r] / (float)C + eps);
                uint4 raw;
                T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    float o = gv[j] * ((v[r][it][j] - mean[r]) * rstd) + bv[j];
                    if (relu) o = fmaxf(o, 0.f);
                    e[j] = st1<T>(o);
                }
                *reinterpret_cast<uint4 *>(y + (size_t)(n0 + r) * C + f0) = raw;
            }
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

// axis = 0: (C, N).  A cluster of kLnSplit CTAs owns COLS consecutive samples (columns); CTA r
// takes rows [r * rows, (r + 1) * rows).  Thread t reads 8 consecutive columns (cc = t % TPR,
// TPR = COLS / 8) of rows rg, rg + RG, ... (rg = t / TPR), so a warp reads 32 / TPR rows of
// 16 * TPR bytes per instruction.  (32-sample tiles, twice the clusters, measured slower than 64:
// 12.1 against 11.0 us at N = 1024, C = 4096.)  The CTA's slice is kept in shared memory (CACHE), so x is read from memory
// once; the second and third pass (squared deviations, output) read the slice.
template <typename T, bool CACHE, int COLS>
__global__ void __cluster_dims__(kLnSplit, 1, 1) __launch_bounds__(kLnThreads)
k_ln_cols(const T *__restrict__ x, const float *__restrict__ g, const float *__restrict__ b, T *y, int C, int N,
          float eps, int relu)
{
    extern __shared__ __align__(16) uint8_t ln_smem[];
    Vec8<T> *slice = reinterpret_cast<Vec8<T> *>(ln_smem);          // [rows][8] vectors (CACHE)
    constexpr int TPR = COLS / 8, RG = kLnThreads / TPR;              // threads per row, row groups
    __shared__ float acc[RG][COLS];                                    // per row group, per column
    __shared__ float part1[COLS], part2[COLS];                  // this CTA's partial sums
    __shared__ float stat[2][COLS];                                // cluster-wide mean, 1 / std
    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    tc::pdl_wait();                                    // the previous kernel's writes are visible
    const uint32_t rank = tc::cluster_ctarank();
    const int tile = blockIdx.x / kLnSplit;
    const int rg = threadIdx.x / TPR, cc = threadIdx.x % TPR;
    const int n0 = tile * COLS + cc * 8;                            // first of this thread's 8 columns
    const bool has = n0 < N;                                           // N % 8 == 0: all 8 or none
    const int rows = (C + kLnSplit - 1) / kLnSplit;
    const int r0 = (int)rank * rows, r1 = min(C, r0 + rows);
    const int nr = max(0, r1 - r0);
    // g, b of this CTA's rows, staged once so the output pass does not wait on them per row
    float *sg = reinterpret_cast<float *>(ln_smem + (CACHE ? (size_t)rows * sizeof(Vec8<T>) * TPR : 0));
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
                    cp_async16(reinterpret_cast<uint8_t *>(&slice[i * TPR + cc]) + 16 * h,
                               reinterpret_cast<const uint8_t *>(src) + 16 * h);
            }
        cp_async_wait_all();                           // this thread's copies have landed
        if (has)
            for (int i = rg; i < nr; i += RG) {        // each thread reads back only its own copies
                float f[8];
                unpack8<T>(slice[i * TPR + cc], f);
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
    if (threadIdx.x < COLS) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part1[threadIdx.x] = t;
    }
    tc::cluster_sync();                                // every CTA's part1 is written
    if (threadIdx.x < COLS) stat[0][threadIdx.x] = cluster_sum(part1, threadIdx.x) / (float)C;
    __syncthreads();
    float mean[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mean[j] = stat[0][cc * 8 + j];

    // pass 2: squared deviations
    float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (has)
        for (int i = rg; i < nr; i += RG) {
            float f[8];
            unpack8<T>(CACHE ? slice[i * TPR + cc] : gload(r0 + i), f);
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
    if (threadIdx.x < COLS) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part2[threadIdx.x] = t;
    }
    tc::cluster_sync();                                // every CTA's part2 is written
    if (threadIdx.x < COLS) stat[1][threadIdx.x] = rsqrtf(cluster_sum(part2, threadIdx.x) / (float)C + eps);
    __syncthreads();
    float rstd[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rstd[j] = stat[1][cc * 8 + j];

    // pass 3: normalise this CTA's rows
    if (has)
        for (int i = rg; i < nr; i += RG) {
            const int f = r0 + i;
            float v[8];
            unpack8<T>(CACHE ? slice[i * TPR + cc] : gload(f), v);
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


constexpr int kLngChunks = 1024;        // axis = 1: at most this many partial sets (row chunks)
constexpr int kLngChunkRows = 4;        // axis = 1: at least this many samples per chunk

// Two sums over the CTA at once; every thread gets both totals.  `red` has two slots per warp.
__device__ __forceinline__ float2 block_sum2(float u, float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        u += __shfl_xor_sync(0xffffffffu, u, o);
        v += __shfl_xor_sync(0xffffffffu, v, o);
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) {
        red[2 * warp] = u;
        red[2 * warp + 1] = v;
    }
    __syncthreads();
    float su = 0.f, sv = 0.f;
#pragma unroll
    for (int w = 0; w < kLnThreads / 32; ++w) {
        su += red[2 * w];
        sv += red[2 * w + 1];
    }
    return make_float2(su, sv);
}

// axis = 1 gradient, first kernel: one CTA per sample; thread t owns the 16-byte vectors
// t, t + 256, ... of the row (as k_ln_rows).  Computes dx and stores the sample's mean and
// rstd at stats[2 n], stats[2 n + 1] for the column sums of dg, db.
template <typename T, int IT>
__global__ void __launch_bounds__(kLnThreads)
k_lng_rows(const T *__restrict__ x, const T *__restrict__ y, const float *__restrict__ g, const T *dy, T *dx,
           float *__restrict__ stats, int C, float eps, int relu)
{
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float red[2 * kLnThreads / 32];
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    const size_t row = (size_t)blockIdx.x * C;
    float xh[IT][VEC], a[IT][VEC];
    float s = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
            const uint4 rx = *reinterpret_cast<const uint4 *>(x + row + f0);
            const uint4 rd = *reinterpret_cast<const uint4 *>(dy + row + f0);
            uint4 ry = make_uint4(0u, 0u, 0u, 0u);
            if (relu) ry = *reinterpret_cast<const uint4 *>(y + row + f0);
            const T *ex = reinterpret_cast<const T *>(&rx);
            const T *ed = reinterpret_cast<const T *>(&rd);
            const T *ey = reinterpret_cast<const T *>(&ry);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                xh[it][j] = ld1<T>(ex + j);
                s += xh[it][j];
                const float d = ld1<T>(ed + j);
                a[it][j] = (relu && !(ld1<T>(ey + j) > 0.f)) ? 0.f : d;         // dz, for now
            }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) xh[it][j] = a[it][j] = 0.f;
        }
    }
    const float mean = block_sum(s, red) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C)
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const float d = xh[it][j] - mean;
                q += d * d;
            }
    }
    const float rstd = rsqrtf(block_sum(q, red) / (float)C + eps);
    float sa = 0.f, sax = 0.f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
            float gv[VEC];
#pragma unroll
            for (int j = 0; j < VEC; j += 4)
                *reinterpret_cast<float4 *>(gv + j) = *reinterpret_cast<const float4 *>(g + f0 + j);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const float h = (xh[it][j] - mean) * rstd;
                xh[it][j] = h;
                a[it][j] *= gv[j];
                sa += a[it][j];
                sax += a[it][j] * h;
            }
        }
    }
    const float2 t = block_sum2(sa, sax, red);
    const float ma = t.x / (float)C, mx = t.y / (float)C;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C) {
            uint4 raw;
            T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
            for (int j = 0; j < VEC; ++j) e[j] = st1<T>(rstd * (a[it][j] - ma - xh[it][j] * mx));
            *reinterpret_cast<uint4 *>(dx + row + f0) = raw;
        }
    }
    if (threadIdx.x == 0) {
        stats[2 * blockIdx.x] = mean;
        stats[2 * blockIdx.x + 1] = rstd;
    }
}

// axis = 1 gradient in one pass for rows of at most 4 vectors per thread: CTA p takes the R
// consecutive samples of chunk p in turn, loading the next sample's x, dy (and y) while it
// finishes the current one, and keeps the per-feature partial dg, db of its chunk in registers
// (each thread owns the same features in every row); it writes them to ws[p][f], ws[p][C + f]
// for k_lng_reduce.  Three two-barrier block sums per sample: mean, variance, (sum a, sum a xh).
template <typename T, int IT>
__global__ void __launch_bounds__(kLnThreads)
k_lng_rows_fused(const T *__restrict__ x, const T *__restrict__ y, const float *__restrict__ g, const T *dy, T *dx,
                 float *__restrict__ ws, int N, int C, int R, float eps, int relu)
{
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float red[2 * kLnThreads / 32];
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    const int n0 = blockIdx.x * R, n1 = min(N, n0 + R);
    float pg[IT][VEC], pb[IT][VEC], gv[IT][VEC];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
#pragma unroll
        for (int j = 0; j < VEC; ++j) pg[it][j] = pb[it][j] = gv[it][j] = 0.f;
        if (f0 < C)
#pragma unroll
            for (int j = 0; j < VEC; j += 4)
                *reinterpret_cast<float4 *>(&gv[it][j]) = *reinterpret_cast<const float4 *>(g + f0 + j);
    }
    uint4 cx[IT], cd[IT], cy[IT];                      // the current sample's raw vectors
    auto load = [&](int n, uint4 (&lx)[IT], uint4 (&ld)[IT], uint4 (&ly)[IT]) {
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            lx[it] = ld[it] = ly[it] = make_uint4(0u, 0u, 0u, 0u);
            if (n < n1 && f0 < C) {
                const size_t o = (size_t)n * C + f0;
                lx[it] = *reinterpret_cast<const uint4 *>(x + o);
                ld[it] = *reinterpret_cast<const uint4 *>(dy + o);
                if (relu) ly[it] = *reinterpret_cast<const uint4 *>(y + o);
            }
        }
    };
    load(n0, cx, cd, cy);
    for (int n = n0; n < n1; ++n) {
        uint4 nx[IT], nd[IT], ny[IT];
        load(n + 1, nx, nd, ny);                       // in flight while this sample is finished
        float xh[IT][VEC], a[IT][VEC];
        float s1[1] = {0.f};
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const T *ex = reinterpret_cast<const T *>(&cx[it]);
            const T *ed = reinterpret_cast<const T *>(&cd[it]);
            const T *ey = reinterpret_cast<const T *>(&cy[it]);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                xh[it][j] = ld1<T>(ex + j);
                s1[0] += xh[it][j];
                a[it][j] = (relu && !(ld1<T>(ey + j) > 0.f)) ? 0.f : ld1<T>(ed + j);   // dz, for now
            }
        }
        block_sums<1>(s1, red);
        const float mean = s1[0] / (float)C;
        float q1[1] = {0.f};
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            if (f0 < C)
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float d = xh[it][j] - mean;
                    q1[0] += d * d;
                }
        }
        block_sums<1>(q1, red);
        const float rstd = rsqrtf(q1[0] / (float)C + eps);
        float t2[2] = {0.f, 0.f};
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            if (f0 < C)
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float h = (xh[it][j] - mean) * rstd;
                    const float dz = a[it][j];
                    xh[it][j] = h;
                    pg[it][j] += dz * h;
                    pb[it][j] += dz;
                    a[it][j] = gv[it][j] * dz;
                    t2[0] += a[it][j];
                    t2[1] += a[it][j] * h;
                }
        }
        block_sums<2>(t2, red);
        const float ma = t2[0] / (float)C, mx = t2[1] / (float)C;
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
            if (f0 < C) {
                uint4 raw;
                T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
                for (int j = 0; j < VEC; ++j) e[j] = st1<T>(rstd * (a[it][j] - ma - xh[it][j] * mx));
                *reinterpret_cast<uint4 *>(dx + (size_t)n * C + f0) = raw;
            }
        }
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            cx[it] = nx[it];
            cd[it] = nd[it];
            cy[it] = ny[it];
        }
    }
    float *w0 = ws + (size_t)blockIdx.x * 2 * C;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const int f0 = (it * kLnThreads + (int)threadIdx.x) * VEC;
        if (f0 < C)
#pragma unroll
            for (int j = 0; j < VEC; j += 4) {
                *reinterpret_cast<float4 *>(w0 + f0 + j) = make_float4(pg[it][j], pg[it][j + 1], pg[it][j + 2], pg[it][j + 3]);
                *reinterpret_cast<float4 *>(w0 + C + f0 + j) =
                    make_float4(pb[it][j], pb[it][j + 1], pb[it][j + 2], pb[it][j + 3]);
            }
    }
}

// axis = 1 gradient, second kernel: per-feature sums over a chunk of R samples.  CTA
// (blockIdx.x, blockIdx.y) covers features [blockIdx.x * 256 * VEC, + 256 * VEC) (thread t the
// VEC features from (blockIdx.x * 256 + t) * VEC) and samples [blockIdx.y * R, + R); it writes
// sum dz * xh to ws[blockIdx.y][f] and sum dz to ws[blockIdx.y][C + f].  x, dy, y were just read
// by the first kernel and come from L2; four samples' loads are in flight per thread.
template <typename T>
__global__ void __launch_bounds__(kLnThreads)
k_lng_colsum(const T *__restrict__ x, const T *__restrict__ y, const T *__restrict__ dy,
             const float *__restrict__ stats, float *__restrict__ ws, int N, int C, int R, int relu)
{
    constexpr int VEC = 16 / sizeof(T);
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    const int f0 = (blockIdx.x * kLnThreads + (int)threadIdx.x) * VEC;
    if (f0 >= C) return;
    const int n0 = blockIdx.y * R, n1 = min(N, n0 + R);
    float pg[VEC], pb[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) pg[j] = pb[j] = 0.f;
    auto add = [&](int n, const uint4 &rx, const uint4 &rd, const uint4 &ry) {
        const float mean = stats[2 * n], rstd = stats[2 * n + 1];
        const T *ex = reinterpret_cast<const T *>(&rx);
        const T *ed = reinterpret_cast<const T *>(&rd);
        const T *ey = reinterpret_cast<const T *>(&ry);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float dz = (relu && !(ld1<T>(ey + j) > 0.f)) ? 0.f : ld1<T>(ed + j);
            pg[j] += dz * ((ld1<T>(ex + j) - mean) * rstd);
            pb[j] += dz;
        }
    };
    int n = n0;
    for (; n + 3 < n1; n += 4) {
        uint4 rx[4], rd[4], ry[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t o = (size_t)(n + u) * C + f0;
            rx[u] = *reinterpret_cast<const uint4 *>(x + o);
            rd[u] = *reinterpret_cast<const uint4 *>(dy + o);
            ry[u] = relu ? *reinterpret_cast<const uint4 *>(y + o) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) add(n + u, rx[u], rd[u], ry[u]);
    }
    for (; n < n1; ++n) {
        const size_t o = (size_t)n * C + f0;
        add(n, *reinterpret_cast<const uint4 *>(x + o), *reinterpret_cast<const uint4 *>(dy + o),
            relu ? *reinterpret_cast<const uint4 *>(y + o) : make_uint4(0u, 0u, 0u, 0u));
    }
    float *w0 = ws + (size_t)blockIdx.y * 2 * C;
#pragma unroll
    for (int j = 0; j < VEC; j += 4) {
        *reinterpret_cast<float4 *>(w0 + f0 + j) = make_float4(pg[j], pg[j + 1], pg[j + 2], pg[j + 3]);
        *reinterpret_cast<float4 *>(w0 + C + f0 + j) = make_float4(pb[j], pb[j + 1], pb[j + 2], pb[j + 3]);
    }
}

// Cluster-wide per-column sums of two per-thread partial vectors (8 columns each, COLS / 8
// threads per row): the row groups' partials are added in the CTA (fixed order), exchanged over
// the cluster and added in rank order, into out0[COLS], out1[COLS] of every CTA.
template <int COLS>
__device__ __forceinline__ void cluster_col_sums2(const float (&u)[8], const float (&v)[8], float (*acc)[COLS],
                                                  float *part_u, float *part_v, float *out0, float *out1)
{
    constexpr int TPR = COLS / 8, RG = kLnThreads / TPR;
    const int rg = threadIdx.x / TPR, cc = threadIdx.x % TPR;
    __syncthreads();                                   // acc may still be read
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[rg][cc * 8 + j] = u[j];
    __syncthreads();
    if (threadIdx.x < COLS) {
        float t = 0.f;
#pragma unroll 8
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part_u[threadIdx.x] = t;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[rg][cc * 8 + j] = v[j];
    __syncthreads();
    if (threadIdx.x < COLS) {
        float t = 0.f;
#pragma unroll 8
        for (int w = 0; w < RG; ++w) t += acc[w][threadIdx.x];
        part_v[threadIdx.x] = t;
    }
    tc::cluster_sync();                                // every CTA's partials are written
    if (threadIdx.x < COLS) {
        out0[threadIdx.x] = cluster_sum(part_u, threadIdx.x);
        out1[threadIdx.x] = cluster_sum(part_v, threadIdx.x);
    }
    __syncthreads();
}

// axis = 0 gradient: the cluster layout of k_ln_cols with kLngCols = 32 samples per cluster
// (kLnSplit CTAs, CTA r owns a share of the C feature rows, thread t 8 consecutive samples of
// rows rg, rg + 64, ...), so that the cached slices of two CTAs fit one SM.
// Passes: mean, variance (as the forward), then the cluster sums of a and a * xh, then dx and
// the per-row (feature) partial dg, db over this tile's samples, written to ws[tile][0|1][f].
// With CACHE the CTA's slices of x and dy are copied to shared memory first, every copy in
// flight at once; with relu dy is then zeroed there where y <= 0 (y read once, four loads in
// flight), and the passes read x and dz there.  Without CACHE each pass reads memory (from L2
// after the first pass) with several loads in flight per thread.
template <typename T, bool CACHE>
__global__ void __cluster_dims__(kLnSplit, 1, 1) __launch_bounds__(kLnThreads)
k_lng_cols(const T *__restrict__ x, const T *__restrict__ y, const float *__restrict__ g, const T *dy, T *dx,
           float *__restrict__ ws, int C, int N, float eps, int relu)
{
    extern __shared__ __align__(16) uint8_t ln_smem[];
    constexpr int TPR = kLngCols / 8, RG = kLnThreads / TPR;          // threads per row, row groups
    __shared__ float acc[RG][kLngCols];
    __shared__ float part_u[kLngCols], part_v[kLngCols];
    __shared__ float stat[4][kLngCols];                               // sum x, sum sq, sum a, sum a xh
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    const uint32_t rank = tc::cluster_ctarank();
    const int tile = blockIdx.x / kLnSplit;
    const int rg = threadIdx.x / TPR, cc = threadIdx.x % TPR;
    const int n0 = tile * kLngCols + cc * 8;
    const bool has = n0 < N;                                           // N % 8 == 0: all 8 or none
    const int rows = (C + kLnSplit - 1) / kLnSplit;
    const int r0 = (int)rank * rows, r1 = min(C, r0 + rows);
    const int nr = max(0, r1 - r0);
    const int nsl = CACHE ? 2 : 0;                                     // cached slices: x, dz
    Vec8<T> *sl = reinterpret_cast<Vec8<T> *>(ln_smem);              // [nsl][rows][TPR] (CACHE)
    float *sg = reinterpret_cast<float *>(ln_smem + (CACHE ? (size_t)nsl * rows * sizeof(Vec8<T>) * TPR : 0));
    for (int i = threadIdx.x; i < nr; i += kLnThreads) sg[i] = g[r0 + i];
    const T *src[3] = {x, dy, y};
    if (CACHE) {
        if (has)
            for (int q = 0; q < nsl; ++q)
                for (int i = rg; i < nr; i += RG) {
                    const T *p = src[q] + (size_t)(r0 + i) * N + n0;
#pragma unroll
                    for (int h = 0; h < (int)(sizeof(Vec8<T>) / 16); ++h)
                        cp_async16(reinterpret_cast<uint8_t *>(&sl[((size_t)q * rows + i) * TPR + cc]) + 16 * h,
                                   reinterpret_cast<const uint8_t *>(p) + 16 * h);
                }
        cp_async_wait_all();                           // each thread reads back only its own copies
        if (relu && has) {                             // dz = dy where y > 0, in place (own elements)
            int i = rg;
            auto mask = [&](int ii, const Vec8<T> &yv) {
                float yf[8], d[8];
                unpack8<T>(yv, yf);
                Vec8<T> &slot = sl[((size_t)rows + ii) * TPR + cc];
                unpack8<T>(slot, d);
                T *e = reinterpret_cast<T *>(&slot);
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = st1<T>(yf[j] > 0.f ? d[j] : 0.f);
            };
            for (; i + 3 * RG < nr; i += 4 * RG) {
                Vec8<T> yv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    yv[u] = *reinterpret_cast<const Vec8<T> *>(y + (size_t)(r0 + i + u * RG) * N + n0);
#pragma unroll
                for (int u = 0; u < 4; ++u) mask(i + u * RG, yv[u]);
            }
            for (; i < nr; i += RG) mask(i, *reinterpret_cast<const Vec8<T> *>(y + (size_t)(r0 + i) * N + n0));
        }
    }
    // slice q (0 x, 1 dy, 2 y) of row i of this CTA, 8 samples (x and dz from shared memory with CACHE)
    auto ld8 = [&](int q, int i, float (&f)[8]) {
        if (CACHE && q < nsl) unpack8<T>(sl[((size_t)q * rows + i) * TPR + cc], f);
        else unpack8<T>(*reinterpret_cast<const Vec8<T> *>(src[q] + (size_t)(r0 + i) * N + n0), f);
    };
    auto dz8 = [&](int i, float (&dz)[8]) {
        ld8(1, i, dz);
        if (relu && !CACHE) {
            float yv[8];
            ld8(2, i, yv);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (!(yv[j] > 0.f)) dz[j] = 0.f;
        }
    };
    const float zero8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};

    // pass 1: sums of x
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (has) {
        int i = rg;
        if (!CACHE)
            for (; i + 3 * RG < nr; i += 4 * RG) {                    // four loads in flight
                float f[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u) ld8(0, i + u * RG, f[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int j = 0; j < 8; ++j) s[j] += f[u][j];
            }
        for (; i < nr; i += RG) {
            float f[8];
            ld8(0, i, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] += f[j];
        }
    }
    cluster_col_sums2<kLngCols>(s, zero8, acc, part_u, part_v, stat[0], stat[2]);
    float mean[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mean[j] = stat[0][cc * 8 + j] / (float)C;

    // pass 2: squared deviations
    float q2[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (has) {
        int i = rg;
        if (!CACHE)
            for (; i + 3 * RG < nr; i += 4 * RG) {
                float f[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u) ld8(0, i + u * RG, f[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float d = f[u][j] - mean[j];
                        q2[j] += d * d;
                    }
            }
        for (; i < nr; i += RG) {
            float f[8];
            ld8(0, i, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float d = f[j] - mean[j];
                q2[j] += d * d;
            }
        }
    }
    tc::cluster_sync();                                // the peers have read this CTA's part_u / part_v
    cluster_col_sums2<kLngCols>(q2, zero8, acc, part_u, part_v, stat[1], stat[2]);
    float rstd[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rstd[j] = rsqrtf(stat[1][cc * 8 + j] / (float)C + eps);

    // pass 3: sums of a = g * dz and of a * xh
    float sa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, sx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (has) {
        int i = rg;
        if (!CACHE)
            for (; i + RG < nr; i += 2 * RG) {                        // two rows (4-6 loads) in flight
                float f[2][8], dz[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    ld8(0, i + u * RG, f[u]);
                    dz8(i + u * RG, dz[u]);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float gf = sg[i + u * RG];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float av = gf * dz[u][j];
                        sa[j] += av;
                        sx[j] += av * ((f[u][j] - mean[j]) * rstd[j]);
                    }
                }
            }
        for (; i < nr; i += RG) {
            float f[8], dz[8];
            ld8(0, i, f);
            dz8(i, dz);
            const float gf = sg[i];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float av = gf * dz[j];
                sa[j] += av;
                sx[j] += av * ((f[j] - mean[j]) * rstd[j]);
            }
        }
    }
    tc::cluster_sync();
    cluster_col_sums2<kLngCols>(sa, sx, acc, part_u, part_v, stat[2], stat[3]);
    float ma[8], mx[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        ma[j] = stat[2][cc * 8 + j] / (float)C;
        mx[j] = stat[3][cc * 8 + j] / (float)C;
    }

    // pass 4: dx, and this tile's partial dg, db of each of the CTA's rows
    float *w0 = ws + (size_t)tile * 2 * C;
    for (int ib = 0; ib < nr; ib += RG) {
        const int i = ib + rg;
        float pg = 0.f, pb = 0.f;
        if (has && i < nr) {
            float f[8], dz[8];
            ld8(0, i, f);
            dz8(i, dz);
            const float gf = sg[i];
            Vec8<T> o;
            T *e = reinterpret_cast<T *>(&o);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float h = (f[j] - mean[j]) * rstd[j];
                pg += dz[j] * h;
                pb += dz[j];
                e[j] = st1<T>(rstd[j] * (gf * dz[j] - ma[j] - h * mx[j]));
            }
            *reinterpret_cast<Vec8<T> *>(dx + (size_t)(r0 + i) * N + n0) = o;
        }
        // the TPR threads of a row (consecutive lanes of a warp) add their 8-sample sums
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
            pg += __shfl_xor_sync(0xffffffffu, pg, o);
            pb += __shfl_xor_sync(0xffffffffu, pb, o);
        }
        if (cc == 0 && i < nr) {
            w0[r0 + i] = pg;
            w0[C + r0 + i] = pb;
        }
    }
    tc::cluster_sync();                                // no CTA leaves while a peer reads its partials
}

// dg[f] = sum_p ws[p][f], db[f] = sum_p ws[p][C + f] over P partial rows of 2C floats: a CTA of
// kLngRedThreads owns 128 consecutive entries of the 2C (32 lanes x 4); warp w adds rows
// p = w, w + 32, ... and the 32 warp sums are added in warp order (fixed order: deterministic).
constexpr int kLngRedThreads = 1024;

__global__ void __launch_bounds__(kLngRedThreads) k_lng_reduce(const float *__restrict__ ws, float *dg, float *db,
                                                               int P, int C)
{
    constexpr int W = kLngRedThreads / 32;
    __shared__ float4 part[W][32];
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int k = (blockIdx.x * 32 + lane) * 4;                        // 4 entries of 0 .. 2C - 1
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < 2 * C) {
        int p = warp;
        for (; p + 3 * W < P; p += 4 * W) {                             // four rows in flight
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4 *>(ws + (size_t)(p + u * W) * 2 * C + k);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                s.x += v[u].x;
                s.y += v[u].y;
                s.z += v[u].z;
                s.w += v[u].w;
            }
        }
        for (; p < P; p += W) {
            const float4 v = *reinterpret_cast<const float4 *>(ws + (size_t)p * 2 * C + k);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
    }
    part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && k < 2 * C) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < W; ++w) {
            const float4 v = part[w][lane];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        // C is a multiple of 4, so the four entries are all dg or all db
        float *dst = k < C ? dg + k : db + (k - C);
        dst[0] = t.x;
        dst[1] = t.y;
        dst[2] = t.z;
        dst[3] = t.w;
    }
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

// Rows per CTA: several when the rows are short enough for their registers and the grid still
// gives every SM a few CTAs (BSMM_LN_RPC pins 1, 2 or 4 for tuning).
inline int ln_rows_per_cta(int N, int it)
{
    if (const char *e = getenv("BSMM_LN_RPC")) {
        const int v = atoi(e);
        if (v == 1 || v == 2 || v == 4) return it <= 4 || v == 1 ? v : 1;
    }
    if (it > 4) return 1;
    return N >= 1024 ? 4 : 1;                          // measured: 2 rows per CTA was slower than 1 at N = 1024
}

template <typename T, int IT>
cudaError_t launch_rows(const void *x, const float *g, const float *b, void *y, int N, int C, float eps, int relu,
                        cudaStream_t s)
{
    const int rpc = ln_rows_per_cta(N, IT);
    const T *xt = static_cast<const T *>(x);
    T *yt = static_cast<T *>(y);
    if (IT <= 4 && rpc == 4)
        return launch_pdl_ln(k_ln_rows<T, IT, (IT <= 4 ? 4 : 1)>, (N + 3) / 4, 0, s, xt, g, b, yt, N, C, eps, relu);
    if (IT <= 4 && rpc == 2)
        return launch_pdl_ln(k_ln_rows<T, IT, (IT <= 4 ? 2 : 1)>, (N + 1) / 2, 0, s, xt, g, b, yt, N, C, eps, relu);
    return launch_pdl_ln(k_ln_rows<T, IT, 1>, N, 0, s, xt, g, b, yt, N, C, eps, relu);
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
            auto kern = k_ln_cols<T, true, kLnCols>;
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
            auto kern = k_ln_cols<T, false, kLnCols>;
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

// axis = 1: samples per chunk of the column-sum kernel; the partial sets are the chunks
// (axis = 1) or the 32-sample tiles of k_lng_cols (axis = 0).
int lng_chunk_rows(int N) { return std::max(kLngChunkRows, (N + kLngChunks - 1) / kLngChunks); }

int lng_parts(int N, int axis)
{
    return axis == 1 ? (N + lng_chunk_rows(N) - 1) / lng_chunk_rows(N) : (N + kLngCols - 1) / kLngCols;
}

// Floats ahead of the partial sets in the workspace: the per-sample statistics (axis = 1),
// rounded up to 16 bytes.
size_t lng_stats_floats(int N, int axis) { return axis == 1 ? ((size_t)2 * N + 3) / 4 * 4 : 0; }

template <typename T, int IT>
cudaError_t launch_lng_rows(const void *x, const void *y, const float *g, const void *dy, void *dx, float *stats,
                            int N, int C, float eps, int relu, cudaStream_t s)
{
    return launch_pdl_ln(k_lng_rows<T, IT>, N, 0, s, static_cast<const T *>(x), static_cast<const T *>(y), g,
                         static_cast<const T *>(dy), static_cast<T *>(dx), stats, C, eps, relu);
}

template <typename T>
cudaError_t launch_lng(const void *x, const void *y, const float *g, const void *dy, void *dx, float *dg, float *db,
                       float *ws, int N, int C, int axis, float eps, int relu, cudaStream_t s)
{
    cudaError_t le;
    float *parts = ws + lng_stats_floats(N, axis);
    if (axis == 1) {
        const int vec = 16 / (int)sizeof(T);
        const int need = (C + kLnThreads * vec - 1) / (kLnThreads * vec);
        // rows of at most 4 vectors per thread: one pass for dx and the chunk partials (the same
        // chunks as the column-sum kernel); BSMM_LNG_SPLIT=1 forces the three-kernel form
        const bool fused = need <= 4 && !getenv("BSMM_LNG_SPLIT");
        if (fused) {
            const int R = lng_chunk_rows(N), P = lng_parts(N, 1);
            const T *xt = static_cast<const T *>(x), *yt = static_cast<const T *>(y), *dyt = static_cast<const T *>(dy);
            T *dxt = static_cast<T *>(dx);
            if (need <= 1) le = launch_pdl_ln(k_lng_rows_fused<T, 1>, P, 0, s, xt, yt, g, dyt, dxt, parts, N, C, R, eps, relu);
            else if (need <= 2) le = launch_pdl_ln(k_lng_rows_fused<T, 2>, P, 0, s, xt, yt, g, dyt, dxt, parts, N, C, R, eps, relu);
            else le = launch_pdl_ln(k_lng_rows_fused<T, 4>, P, 0, s, xt, yt, g, dyt, dxt, parts, N, C, R, eps, relu);
        } else if (need <= 1) le = launch_lng_rows<T, 1>(x, y, g, dy, dx, ws, N, C, eps, relu, s);
        else if (need <= 2) le = launch_lng_rows<T, 2>(x, y, g, dy, dx, ws, N, C, eps, relu, s);
        else if (need <= 4) le = launch_lng_rows<T, 4>(x, y, g, dy, dx, ws, N, C, eps, relu, s);
        else if (need <= 8) le = launch_lng_rows<T, 8>(x, y, g, dy, dx, ws, N, C, eps, relu, s);
        else le = launch_lng_rows<T, 16>(x, y, g, dy, dx, ws, N, C, eps, relu, s);
        if (!fused) {
            g_bsmm_launches += 1;
            if (le != cudaSuccess) return le;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)need, (unsigned)lng_parts(N, 1));
            cfg.blockDim = dim3(kLnThreads);
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            le = cudaLaunchKernelEx(&cfg, k_lng_colsum<T>, static_cast<const T *>(x), static_cast<const T *>(y),
                                    static_cast<const T *>(dy), (const float *)ws, parts, N, C, lng_chunk_rows(N),
                                    relu);
        }
    } else {
        const int tiles = lng_parts(N, 0);
        const int rows = (C + kLnSplit - 1) / kLnSplit;
        const size_t slice = (size_t)rows * kLngCols * sizeof(T);
        const size_t gsz = (size_t)rows * sizeof(float);                 // staged g
        const bool cache = 2 * slice + gsz <= (size_t)kLngCacheMax;     // x and dz slices kept in shared memory
        auto kern = cache ? k_lng_cols<T, true> : k_lng_cols<T, false>;
        static std::atomic<int> attr_set[2] = {{-1}, {-1}};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (attr_set[cache].load() != dev) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLnCacheMax);
            if (e != cudaSuccess) return e;
            attr_set[cache].store(dev);
        }
        le = launch_pdl_ln(kern, tiles * kLnSplit, (cache ? 2 * slice : 0) + gsz, s, static_cast<const T *>(x),
                           static_cast<const T *>(y), g, static_cast<const T *>(dy), static_cast<T *>(dx), parts, C,
                           N, eps, relu);
    }
    g_bsmm_launches += 1;
    if (le != cudaSuccess) return le;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((2 * C + 127) / 128));
        cfg.blockDim = dim3(kLngRedThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        le = cudaLaunchKernelEx(&cfg, k_lng_reduce, (const float *)parts, dg, db, lng_parts(N, axis), C);
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

extern "C" size_t bsmm_layer_norm_grad_workspace(int N, int C, int axis)
{
    if (N < 0 || C < 1 || (axis != 0 && axis != 1)) return 0;
    return (lng_stats_floats(N, axis) + (size_t)lng_parts(N, axis) * 2 * (size_t)C) * sizeof(float);
}

extern "C" bsmm_status bsmm_layer_norm_grad(const void *x, const void *y, const float *g, const void *dy, void *dx,
                                            float *dg, float *db, int N, int C, int axis, float epsilon, int relu,
                                            bsmm_dtype t, void *workspace, size_t workspace_bytes, void *stream)
{
    if (N < 0 || C < 1 || (axis != 0 && axis != 1) || !(epsilon >= 0.f)) return BSMM_ERR_INVALID;
    if (t != BSMM_F32 && t != BSMM_F16 && t != BSMM_BF16) return BSMM_ERR_INVALID;
    if (!dg || !db || dg == db) return BSMM_ERR_INVALID;
    const uintptr_t mo = reinterpret_cast<uintptr_t>(dg) | reinterpret_cast<uintptr_t>(db);
    if (mo & 15u) return BSMM_ERR_ALIGN;
    if (axis == 1 && C > kLnMaxC) return BSMM_ERR_UNSUPPORTED;
    if (axis == 0 && (size_t)((C + kLnSplit - 1) / kLnSplit) * sizeof(float) > (size_t)kLnCacheMax)
        return BSMM_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {                                      // no samples: dg = db = 0, nothing else is read
        if (cudaMemsetAsync(dg, 0, (size_t)C * sizeof(float), s) != cudaSuccess ||
            cudaMemsetAsync(db, 0, (size_t)C * sizeof(float), s) != cudaSuccess)
            return BSMM_ERR_CUDA;
        return BSMM_OK;
    }
    if (!x || !g || !dy || !dx || (relu && !y) || !workspace) return BSMM_ERR_INVALID;
    if (dx == x || dx == dy || (relu && dx == y)) return BSMM_ERR_INVALID;   // inputs are read again after dx is written
    if (workspace_bytes < bsmm_layer_norm_grad_workspace(N, C, axis)) return BSMM_ERR_INVALID;
    const size_t e = t == BSMM_F32 ? 4 : 2;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dy) |
                          reinterpret_cast<uintptr_t>(dx) | reinterpret_cast<uintptr_t>(g) |
                          reinterpret_cast<uintptr_t>(workspace) | (relu ? reinterpret_cast<uintptr_t>(y) : 0u);
    if (mis & 15u) return BSMM_ERR_ALIGN;
    if (((size_t)(axis == 1 ? C : N) * e) % 16u) return BSMM_ERR_ALIGN;
    if (axis == 0 && N % 8) return BSMM_ERR_ALIGN;
    float *ws = static_cast<float *>(workspace);
    cudaError_t err;
    if (t == BSMM_F32) err = launch_lng<float>(x, y, g, dy, dx, dg, db, ws, N, C, axis, epsilon, relu, s);
    else if (t == BSMM_F16) err = launch_lng<__half>(x, y, g, dy, dx, dg, db, ws, N, C, axis, epsilon, relu, s);
    else err = launch_lng<__nv_bfloat16>(x, y, g, dy, dx, dg, db, ws, N, C, axis, epsilon, relu, s);
    return err == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}
