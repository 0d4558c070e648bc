// l2_normalize: weight normalisation of the block-sparse weight, and its gradient (README,
// "API Documentation: blocksparse.matmul", BlocksparseMatMul.l2_normalize(W, gain, epsilon,
// dtype)).  Every output feature f = k*bs + j owns one incoming weight vector, column f of the
// dense C x K weight: w[b][i][j] over all blocks b of block column k and all rows i.
//     s_f = sum w^2,  rho_f = 1 / sqrt(max(s_f, epsilon)),  y = gain[f] * rho_f * w   (gain 1 if absent)
// gradient, with D_f = sum dy * w over the same vector:
//     dw = gain[f] * rho_f * (dy - [s_f >= epsilon] * rho_f^2 * D_f * w),  dgain[f] = rho_f * D_f.
//
// A cluster of kWnSplit CTAs owns an output block column k.  CTA r of the cluster takes column
// entries r, r + kWnSplit, ... (the per-column table of the handle lists them, c increasing).
// Thread t handles 16-byte vectors t, t + 256, ... of the CTA's blocks; because a block is
// bs*bs/4 vectors and 1024 is a multiple of bs, every vector of thread t covers the same four
// features j0 .. j0 + 3, j0 = 4t mod bs, so each thread keeps four partial sums (two sets for the
// gradient).  The CTA's partials are added in shared memory, the kWnSplit CTA partials are
// exchanged through distributed shared memory and added in rank order by every CTA (identical
// totals in all of them), and the output pass scales the vectors the CTA still holds: w (and dy)
// are read from memory once.  Two forms:
//   k_l2n    one cluster per column, the vectors held in registers (V per thread; vectors beyond
//            that, in very long columns, are streamed and read a second time);
//   k_l2n_p  persistent clusters that walk the columns, the vectors staged in shared memory with
//            cp.async, double-buffered so the next column's copies overlap the current column's
//            reduction and output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "bsmm.h"
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

namespace {

constexpr int kWnThreads = 256;
constexpr int kWnSplit = 8;      // CTAs per cluster, one cluster per output block column
constexpr int kWnMaxV = 8;       // 16-byte vectors a thread keeps in registers (per operand)
constexpr int kWnSmemMax = 200 * 1024;   // persistent kernel: dynamic shared memory of a CTA, at most

// Kernel form.  By default the gradient takes the persistent kernel wherever a CTA's share of the
// longest column fits its shared memory, and l2_normalize itself the register kernel (measured on
// the 4096-wide, block 32, 50% dense weight: forward 17.3 us with registers against 20.4 us
// persistent; gradient 32.0 us persistent against 44.1 us with registers).
// BSMM_WN_KERNEL=registers or =persistent (read at every call) forces one form where it fits, for
// comparison and for testing both.
enum WnForm { kWnAuto, kWnRegisters, kWnPersistent };
WnForm wn_form()
{
    const char *e = getenv("BSMM_WN_KERNEL");
    if (e && strcmp(e, "registers") == 0) return kWnRegisters;
    if (e && strcmp(e, "persistent") == 0) return kWnPersistent;
    return kWnAuto;
}

// Four consecutive elements of type T as floats, from a 16-byte (float) or 8-byte (16-bit) load.
template <typename T> __device__ __forceinline__ float4 ld4(const T *p);
template <> __device__ __forceinline__ float4 ld4<float>(const float *p)
{
    return __ldg(reinterpret_cast<const float4 *>(p));
}
template <> __device__ __forceinline__ float4 ld4<__half>(const __half *p)
{
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <> __device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Store four floats rounded to T (round to nearest even).
template <typename T> __device__ __forceinline__ void st4(T *p, float4 v);
template <> __device__ __forceinline__ void st4<float>(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
template <> __device__ __forceinline__ void st4<__half>(__half *p, float4 v)
{
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 r;
    r.x = *reinterpret_cast<const uint32_t *>(&a);
    r.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = r;
}
template <> __device__ __forceinline__ void st4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v)
{
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 r;
    r.x = *reinterpret_cast<const uint32_t *>(&a);
    r.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = r;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cluster(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void fma4(float4 &acc, float4 a, float4 b)
{
    acc.x = fmaf(a.x, b.x, acc.x);
    acc.y = fmaf(a.y, b.y, acc.y);
    acc.z = fmaf(a.z, b.z, acc.z);
    acc.w = fmaf(a.w, b.w, acc.w);
}

// GRAD = false: out = y of type T (dy unused, dgain unused).
// GRAD = true:  out = dw (float), dy of type T, dgain (may be null).
// lq = log2(bs*bs/4), the number of 16-byte vectors of a block.
template <bool GRAD, typename T, int V>
__global__ void __cluster_dims__(kWnSplit, 1, 1) __launch_bounds__(kWnThreads)
k_l2n(const int32_t *__restrict__ col_ptr, const int32_t *__restrict__ col_ent, const float *w,
      const float *__restrict__ gain, const T *dy, void *out, float *__restrict__ dgain, int bs, int lq, float eps)
{
    __shared__ float4 part[2][kWnThreads];             // per-thread partial sums (s, D)
    __shared__ float csum[2][32];                      // this CTA's per-feature partials
    __shared__ __align__(16) float coef[2][32];        // per-feature output coefficients
    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    tc::pdl_wait();                                    // the previous kernel's writes are visible

    const int k = blockIdx.x / kWnSplit;
    const int rank = (int)tc::cluster_ctarank();
    const int e0 = col_ptr[k];
    const int n = col_ptr[k + 1] - e0;
    const int nb = n > rank ? (n - rank + kWnSplit - 1) / kWnSplit : 0;     // this CTA's blocks
    const int units = nb << lq;
    const int qmask = (1 << lq) - 1;
    const int t = threadIdx.x;
    const size_t bb = (size_t)bs * bs;

    // element offset of 16-byte vector u of this CTA's blocks
    auto offset = [&](int u) -> size_t {
        const int b = __ldg(col_ent + 2 * (e0 + rank + (u >> lq) * kWnSplit));
        return (size_t)b * bb + (size_t)(u & qmask) * 4;
    };

    float4 wr[V], gr[V];
    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = s4;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int u = t + v * kWnThreads;
        if (u < units) {
            const size_t o = offset(u);
            wr[v] = ld4<float>(w + o);
            if (GRAD) gr[v] = ld4<T>(dy + o);
        }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
        if (t + v * kWnThreads < units) {
            fma4(s4, wr[v], wr[v]);
            if (GRAD) fma4(d4, gr[v], wr[v]);
        }
    }
    for (int u = t + V * kWnThreads; u < units; u += kWnThreads) {   // long columns: streamed
        const size_t o = offset(u);
        const float4 a = ld4<float>(w + o);
        fma4(s4, a, a);
        if (GRAD) fma4(d4, ld4<T>(dy + o), a);
    }

    // CTA partials: feature j is component j % 4 of the threads t = j / 4 (mod bs / 4)
    part[0][t] = s4;
    if (GRAD) part[1][t] = d4;
    __syncthreads();
    if (t < bs) {
        const float *p0 = reinterpret_cast<const float *>(part[0]);
        const float *p1 = reinterpret_cast<const float *>(part[1]);
        float a = 0.f, d = 0.f;
        for (int i = t; i < kWnThreads * 4; i += bs) {  // float t of every (bs / 4)-th thread's vector
            a += p0[i];
            if (GRAD) d += p1[i];
        }
        csum[0][t] = a;
        if (GRAD) csum[1][t] = d;
    }
    tc::cluster_sync();                                // every CTA's csum is written
    if (t < bs) {
        float s = 0.f, d = 0.f;
        const uint32_t a0 = tc::smem_u32(&csum[0][t]), a1 = tc::smem_u32(&csum[1][t]);
#pragma unroll
        for (int r = 0; r < kWnSplit; ++r) {           // rank order: identical totals in every CTA
            s += ld_cluster(tc::map_to_rank(a0, (uint32_t)r));
            if (GRAD) d += ld_cluster(tc::map_to_rank(a1, (uint32_t)r));
        }
        const int f = k * bs + t;
        const float g = gain ? gain[f] : 1.f;
        const float rho = 1.f / sqrtf(fmaxf(s, eps));
        coef[0][t] = g * rho;
        if (GRAD) {
            coef[1][t] = s >= eps ? rho * rho * d : 0.f;
            if (dgain && rank == 0) dgain[f] = rho * d;
        }
    }
    cluster_arrive();                                  // remote reads done; peers may leave later
    __syncthreads();

    const int j0 = (4 * t) & (bs - 1);
    const float4 ca = *reinterpret_cast<const float4 *>(&coef[0][j0]);
    float4 cc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (GRAD) cc = *reinterpret_cast<const float4 *>(&coef[1][j0]);
    auto emit = [&](size_t o, float4 a, float4 g) {
        if (GRAD) {
            float4 r;
            r.x = ca.x * (g.x - cc.x * a.x);
            r.y = ca.y * (g.y - cc.y * a.y);
            r.z = ca.z * (g.z - cc.z * a.z);
            r.w = ca.w * (g.w - cc.w * a.w);
            st4<float>(static_cast<float *>(out) + o, r);
        } else {
            st4<T>(static_cast<T *>(out) + o, make_float4(ca.x * a.x, ca.y * a.y, ca.z * a.z, ca.w * a.w));
        }
    };
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int u = t + v * kWnThreads;
        if (u < units) emit(offset(u), wr[v], GRAD ? gr[v] : wr[v]);
    }
    for (int u = t + V * kWnThreads; u < units; u += kWnThreads) {
        const size_t o = offset(u);
        const float4 a = ld4<float>(w + o);
        emit(o, a, GRAD ? ld4<T>(dy + o) : a);
    }
    cluster_wait();                                    // no CTA leaves while a peer reads its csum
}


// 16-, 8- and 4-byte asynchronous global -> shared copies; completion: cp.async.wait_group.
__device__ __forceinline__ void cpa16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa8(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <typename T> __device__ __forceinline__ float4 sh4(const uint8_t *p);
template <> __device__ __forceinline__ float4 sh4<float>(const uint8_t *p) { return *reinterpret_cast<const float4 *>(p); }
template <> __device__ __forceinline__ float4 sh4<__half>(const uint8_t *p)
{
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <> __device__ __forceinline__ float4 sh4<__nv_bfloat16>(const uint8_t *p)
{
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Persistent form of k_l2n: gridDim.x / kWnSplit clusters walk the output block columns
// k = cluster, cluster + clusters, ...  A CTA's share of a column (at most cap blocks) is staged
// in shared memory with cp.async, double-buffered: the copies of the next column are in flight
// while the current one is reduced, exchanged and written.  The block ids of a column are copied
// two columns ahead (three slots), so no copy waits on a table lookup.  Each thread copies and
// later reads the same 16-byte vectors (u = t, t + 256, ...), so its own cp.async.wait_group
// orders them; the ids, read by every thread, are published by the barrier after the wait.
// Shared memory: 2 x cap blocks of w (and dy), then 3 x cap block ids.
template <bool GRAD, typename T>
__global__ void __cluster_dims__(kWnSplit, 1, 1) __launch_bounds__(kWnThreads)
k_l2n_p(const int32_t *__restrict__ col_ptr, const int32_t *__restrict__ col_ent, const float *w,
        const float *__restrict__ gain, const T *dy, void *out, float *__restrict__ dgain, int S, int bs, int lq,
        int cap, float eps)
{
    extern __shared__ __align__(16) uint8_t wn_smem[];
    __shared__ float4 part[2][kWnThreads];
    __shared__ float csum[2][2][32];                   // [column parity][s, D][feature]
    __shared__ __align__(16) float coef[2][32];
    constexpr int DSZ = 4 * sizeof(T);                 // bytes of 4 dy elements
    const size_t wbytes = (size_t)cap << (lq + 4);     // one buffer of w: cap blocks
    const size_t dbytes = GRAD ? ((size_t)cap << lq) * DSZ : 0;
    // buffer b of w at wn_smem + b * wbytes, of dy at wn_smem + 2 * wbytes + b * dbytes
    auto wb = [&](int b) { return wn_smem + b * wbytes; };
    auto db = [&](int b) { return wn_smem + 2 * wbytes + b * dbytes; };
    int32_t *ids = reinterpret_cast<int32_t *>(wn_smem + 2 * (wbytes + dbytes));   // [3][cap]

    tc::pdl_launch_dependents();                       // holds no tensor memory: the next kernel may start
    const int t = threadIdx.x;
    const int rank = (int)tc::cluster_ctarank();
    const int clusters = gridDim.x / kWnSplit;
    const int k0 = blockIdx.x / kWnSplit;
    const int qmask = (1 << lq) - 1;
    const size_t bb = (size_t)bs * bs;
    // (first entry, this CTA's block count) of column k; k >= S gives no blocks
    auto span = [&](int k, int &e, int &nb) {
        e = 0;
        nb = 0;
        if (k < S) {
            const int a = __ldg(col_ptr + k), n = __ldg(col_ptr + k + 1) - a;
            e = a;
            nb = n > rank ? (n - rank + kWnSplit - 1) / kWnSplit : 0;
        }
    };
    auto copy_ids = [&](int slot, int e, int nb) {
        for (int m = t; m < nb; m += kWnThreads) cpa4(ids + slot * cap + m, col_ent + 2 * (e + rank + m * kWnSplit));
    };
    auto copy_data = [&](int slot, int buf, int nb) {
        const int units = nb << lq;
        for (int u = t; u < units; u += kWnThreads) {
            const size_t o = (size_t)ids[slot * cap + (u >> lq)] * bb + (size_t)(u & qmask) * 4;
            cpa16(wb(buf) + (size_t)u * 16, w + o);
            if (GRAD) {
                if (DSZ == 16) cpa16(db(buf) + (size_t)u * DSZ, dy + o);
                else cpa8(db(buf) + (size_t)u * DSZ, dy + o);
            }
        }
    };

    // the tables are fixed after creation: read them before waiting on the previous kernel
    int e_a, nb_a, e_b, nb_b, e_c, nb_c;               // columns i, i + 1, i + 2 of this cluster
    span(k0, e_a, nb_a);
    span(k0 + clusters, e_b, nb_b);
    for (int m = t; m < nb_a; m += kWnThreads) ids[m] = __ldg(col_ent + 2 * (e_a + rank + m * kWnSplit));
    copy_ids(1, e_b, nb_b);
    cpa_commit();
    tc::pdl_wait();                                    // w (and dy) may be the previous kernel's output
    __syncthreads();                                   // ids of column 0 published
    copy_data(0, 0, nb_a);
    cpa_commit();

    const int j0 = (4 * t) & (bs - 1);
    int i = 0;
    for (int k = k0; k < S; k += clusters, ++i) {
        const int p = i & 1;
        span(k + 2 * clusters, e_c, nb_c);
        cpa_wait_all();                                // column i's vectors, column i + 1's ids
        __syncthreads();
        copy_data((i + 1) % 3, p ^ 1, nb_b);           // column i + 1
        copy_ids((i + 2) % 3, e_c, nb_c);              // ids of column i + 2
        cpa_commit();

        const int units = nb_a << lq;
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = s4;
        for (int u = t; u < units; u += kWnThreads) {
            const float4 a = sh4<float>(wb(p) + (size_t)u * 16);
            fma4(s4, a, a);
            if (GRAD) fma4(d4, sh4<T>(db(p) + (size_t)u * DSZ), a);
        }
        part[0][t] = s4;
        if (GRAD) part[1][t] = d4;
        __syncthreads();
        if (t < bs) {
            const float *p0 = reinterpret_cast<const float *>(part[0]);
            const float *p1 = reinterpret_cast<const float *>(part[1]);
            float a = 0.f, d = 0.f;
            for (int q = t; q < kWnThreads * 4; q += bs) {
                a += p0[q];
                if (GRAD) d += p1[q];
            }
            csum[p][0][t] = a;
            if (GRAD) csum[p][1][t] = d;
        }
        tc::cluster_sync();                            // every CTA's csum[p] is written
        if (t < bs) {
            float s = 0.f, d = 0.f;
            const uint32_t a0 = tc::smem_u32(&csum[p][0][t]), a1 = tc::smem_u32(&csum[p][1][t]);
#pragma unroll
            for (int r = 0; r < kWnSplit; ++r) {       // rank order: identical totals in every CTA
                s += ld_cluster(tc::map_to_rank(a0, (uint32_t)r));
                if (GRAD) d += ld_cluster(tc::map_to_rank(a1, (uint32_t)r));
            }
            const int f = k * bs + t;
            const float g = gain ? gain[f] : 1.f;
            const float rho = 1.f / sqrtf(fmaxf(s, eps));
            coef[0][t] = g * rho;
            if (GRAD) {
                coef[1][t] = s >= eps ? rho * rho * d : 0.f;
                if (dgain && rank == 0) dgain[f] = rho * d;
            }
        }
        __syncthreads();
        const float4 ca = *reinterpret_cast<const float4 *>(&coef[0][j0]);
        float4 cc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (GRAD) cc = *reinterpret_cast<const float4 *>(&coef[1][j0]);
        const int32_t *cid = ids + (i % 3) * cap;
        for (int u = t; u < units; u += kWnThreads) {
            const size_t o = (size_t)cid[u >> lq] * bb + (size_t)(u & qmask) * 4;
            const float4 a = sh4<float>(wb(p) + (size_t)u * 16);
            if (GRAD) {
                const float4 g = sh4<T>(db(p) + (size_t)u * DSZ);
                float4 r;
                r.x = ca.x * (g.x - cc.x * a.x);
                r.y = ca.y * (g.y - cc.y * a.y);
                r.z = ca.z * (g.z - cc.z * a.z);
                r.w = ca.w * (g.w - cc.w * a.w);
                st4<float>(static_cast<float *>(out) + o, r);
            } else {
                st4<T>(static_cast<T *>(out) + o, make_float4(ca.x * a.x, ca.y * a.y, ca.z * a.z, ca.w * a.w));
            }
        }
        e_a = e_b;
        nb_a = nb_b;
        e_b = e_c;
        nb_b = nb_c;
    }
    cpa_wait_all();                                    // no copy outlives the CTA
    tc::cluster_sync();                                // no CTA leaves while a peer reads its csum
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_wn(void (*kern)(KArgs...), int grid, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWnThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <bool GRAD, typename T, int V>
cudaError_t launch_v(bsmm_ctx *h, const float *w, const float *gain, const void *dy, void *out, float *dgain,
                     int lq, float eps, cudaStream_t s)
{
    return launch_pdl_wn(k_l2n<GRAD, T, V>, h->S * kWnSplit, s, (const int32_t *)h->d_col_ptr,
                         (const int32_t *)h->d_col_ent, w, gain, static_cast<const T *>(dy), out, dgain, h->bs, lq,
                         eps);
}

// Dynamic shared memory of the persistent kernel: both buffers of w (and dy) plus three id slots.
size_t persistent_smem(bool grad, int esz, int bs, int cap)
{
    const size_t blk = (size_t)bs * bs * (4 + (grad ? esz : 0));
    return 2 * blk * cap + 3 * sizeof(int32_t) * cap;
}

template <bool GRAD, typename T>
cudaError_t launch_persistent(bsmm_ctx *h, const float *w, const float *gain, const void *dy, void *out,
                              float *dgain, int lq, int cap, size_t smem, float eps, cudaStream_t s)
{
    auto kern = k_l2n_p<GRAD, T>;
    static std::atomic<int> attr_dev{-1};              // device whose shared-memory limit has been raised
    static std::atomic<long long> occ{-1};             // device << 48 | smem << 16 | resident clusters
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (attr_dev.load() != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kWnSmemMax);
        if (e != cudaSuccess) return e;
        attr_dev.store(dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kWnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    const long long key = ((long long)dev << 48) | ((long long)smem << 16);
    int clusters = 0;
    const long long c = occ.load();
    if (c >= 0 && (c & ~0xffffll) == key) {
        clusters = (int)(c & 0xffff);
    } else {
        cfg.gridDim = dim3(h->S * kWnSplit);           // cluster shape: the kernel's __cluster_dims__
        e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        occ.store(key | (long long)std::min(clusters, 0xffff));
    }
    clusters = std::max(1, std::min(clusters, h->S));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(clusters * kWnSplit);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, (const int32_t *)h->d_col_ptr, (const int32_t *)h->d_col_ent, w, gain,
                              static_cast<const T *>(dy), out, dgain, h->S, h->bs, lq, cap, eps);
}

template <bool GRAD, typename T>
cudaError_t launch_wn(bsmm_ctx *h, const float *w, const float *gain, const void *dy, void *out, float *dgain,
                      float eps, cudaStream_t s)
{
    int maxcol = 0;
    for (int k = 0; k < h->S; ++k) maxcol = std::max(maxcol, h->h_col_ptr[k + 1] - h->h_col_ptr[k]);
    const int lq = h->bs == 32 ? 8 : h->bs == 16 ? 6 : 4;
    const int cap = std::max(1, (maxcol + kWnSplit - 1) / kWnSplit);                // blocks per CTA, at most
    cudaError_t e;
    const size_t smem = persistent_smem(GRAD, (int)sizeof(T), h->bs, cap);
    const WnForm form = wn_form();
    const bool persistent = form == kWnPersistent || (form == kWnAuto && GRAD);
    if (persistent && smem <= (size_t)kWnSmemMax) {
        e = launch_persistent<GRAD, T>(h, w, gain, dy, out, dgain, lq, cap, smem, eps, s);
    } else {
        const int64_t need = (((int64_t)cap << lq) + kWnThreads - 1) / kWnThreads; // vectors per thread
        if (need <= 1) e = launch_v<GRAD, T, 1>(h, w, gain, dy, out, dgain, lq, eps, s);
        else if (need <= 2) e = launch_v<GRAD, T, 2>(h, w, gain, dy, out, dgain, lq, eps, s);
        else if (need <= 4) e = launch_v<GRAD, T, 4>(h, w, gain, dy, out, dgain, lq, eps, s);
        else e = launch_v<GRAD, T, kWnMaxV>(h, w, gain, dy, out, dgain, lq, eps, s);
    }
    g_bsmm_launches += 1;
    return e;
}

bool a16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bsmm_status wn_prologue(bsmm_ctx *h, bsmm_dtype t, float eps)
{
    if (!h) return BSMM_ERR_INVALID;
    if (t != BSMM_F32 && t != BSMM_F16 && t != BSMM_BF16) return BSMM_ERR_INVALID;
    if (!(eps >= 0.f)) return BSMM_ERR_INVALID;                        // negative or NaN
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSMM_ERR_CUDA;
    if (dev != h->device && cudaSetDevice(h->device) != cudaSuccess) return BSMM_ERR_CUDA;
    return BSMM_OK;
}

} // namespace

extern "C" bsmm_status bsmm_l2_normalize(bsmm_t h, const float *w, const float *gain, void *y, float epsilon,
                                         bsmm_dtype t, void *stream)
{
    bsmm_status st = wn_prologue(h, t, epsilon);
    if (st != BSMM_OK) return st;
    if (h->nnz == 0) return BSMM_OK;                   // no blocks: nothing is read or written
    if (!w || !y) return BSMM_ERR_INVALID;
    if (!a16(w) || !a16(y)) return BSMM_ERR_ALIGN;
    if ((const void *)y == (const void *)w && t != BSMM_F32) return BSMM_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (t == BSMM_F32) e = launch_wn<false, float>(h, w, gain, nullptr, y, nullptr, epsilon, s);
    else if (t == BSMM_F16) e = launch_wn<false, __half>(h, w, gain, nullptr, y, nullptr, epsilon, s);
    else e = launch_wn<false, __nv_bfloat16>(h, w, gain, nullptr, y, nullptr, epsilon, s);
    return e == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

extern "C" bsmm_status bsmm_l2_normalize_grad(bsmm_t h, const float *w, const float *gain, const void *dy,
                                              float *dw, float *dgain, float epsilon, bsmm_dtype t, void *stream)
{
    bsmm_status st = wn_prologue(h, t, epsilon);
    if (st != BSMM_OK) return st;
    if (h->nnz == 0 && !dgain) return BSMM_OK;         // nothing to read or write
    if (h->nnz > 0 && (!w || !dy || !dw)) return BSMM_ERR_INVALID;
    if (h->nnz > 0 && (!a16(w) || !a16(dy) || !a16(dw))) return BSMM_ERR_ALIGN;
    if (h->nnz > 0 && ((const void *)dw == (const void *)w || (const void *)dw == dy)) return BSMM_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (t == BSMM_F32) e = launch_wn<true, float>(h, w, gain, dy, dw, dgain, epsilon, s);
    else if (t == BSMM_F16) e = launch_wn<true, __half>(h, w, gain, dy, dw, dgain, epsilon, s);
    else e = launch_wn<true, __nv_bfloat16>(h, w, gain, dy, dw, dgain, epsilon, s);
    return e == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}
