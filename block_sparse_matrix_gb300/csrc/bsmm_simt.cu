// IEEE-float SIMT kernels for all three passes, every dtype and block size.
//
// These are the fp32 path (FFMA, no TF32, so float32 results stay within a
// few ulps of the exact product) and a plain second implementation of the
// 16-bit passes.  Accumulation is float32; 16-bit outputs are rounded to
// nearest-even once at the store.
//
// fprop  (README "__call__(I, W)"):      y[:, k blk]  = sum_{b in column k} x[:, c_b blk] . w[b]
// bprop  (gradient w.r.t. I):            dx[:, c blk] = sum_{b in row c} dy[:, k_b blk] . w[b]^T
// updat  (gradient w.r.t. W, dw_dtype):  dw[b] = sum_t x_t[:, c_b blk]^T . dy_t[:, k_b blk]
//        (t over the G <= 8 timesteps of group_param_grads; G = 1 for a plain updat)
#include "bsmm_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kTN = 64;   // minibatch rows per CTA (fprop/bprop) and per reduction chunk (updat)

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Activation element (n, f) of an (N, F) [FA=1] or (F, N) [FA=0] array.
template <int FA>
__device__ __forceinline__ size_t aidx(int64_t n, int64_t f, int64_t N, int64_t F)
{
    return FA ? (size_t)(n * F + f) : (size_t)(f * N + n);
}

// Output (n, j) handled by slot r of thread tid: feature-fastest for (N,F)
// storage, minibatch-fastest for (F,N) storage, so stores coalesce.
template <int BS, int FA, int TN>
__device__ __forceinline__ void out_coord(int idx, int &n, int &j)
{
    if (FA) { n = idx / BS; j = idx % BS; }
    else    { n = idx % TN; j = idx / TN; }
}

// BWD=false: fprop over the column LUT.  BWD=true: bprop over the row LUT.
// The operands of entry e + 1 (weight block and input panel) are loaded into registers while
// entry e is multiplied out of shared memory, so each entry costs one compute phase instead of a
// memory round trip followed by it.
template <typename T, int BS, int FA, bool BWD, int TN>
__global__ void __launch_bounds__(kThreads)
k_simt_fwd_bwd(const T *__restrict__ in, const T *__restrict__ w, T *__restrict__ out,
               const int32_t *__restrict__ ptr, const int32_t *__restrict__ ent,
               int N, int Fin, int Fout)
{
    constexpr int OUT = TN * BS / kThreads;
    constexpr int NW = (BS * BS + kThreads - 1) / kThreads;   // weight elements per thread
    constexpr int NA = TN * BS / kThreads;                     // panel elements per thread
    __shared__ float sw[BS][BS + 1];
    __shared__ float sa[TN][BS + 1];
    const int tid = threadIdx.x;
    const int blk = blockIdx.x;         // output block column (fprop) / row (bprop)
    const int n0 = blockIdx.y * TN;
    float acc[OUT];
#pragma unroll
    for (int r = 0; r < OUT; ++r) acc[r] = 0.f;

    const int e0 = ptr[blk], e1 = ptr[blk + 1];
    float rw[NW], ra[NA];
    auto load = [&](int e) {
        int b, src;                     // weight block id, source block index of the input panel
        if (BWD) { b = e; src = ent[e]; }
        else     { b = ent[2 * e]; src = ent[2 * e + 1]; }
        const T *wb = w + (size_t)b * BS * BS;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int q = tid + k * kThreads;
            rw[k] = q < BS * BS ? to_f<T>(wb[q]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < NA; ++k) {
            const int q = tid + k * kThreads;
            int n, i;
            if (FA) { n = q / BS; i = q % BS; }
            else    { i = q / TN; n = q % TN; }
            ra[k] = n0 + n < N ? to_f<T>(in[aidx<FA>(n0 + n, (int64_t)src * BS + i, N, Fin)]) : 0.f;
        }
    };
    if (e0 < e1) load(e0);
    for (int e = e0; e < e1; ++e) {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int q = tid + k * kThreads;
            if (q < BS * BS) sw[q / BS][q % BS] = rw[k];
        }
#pragma unroll
        for (int k = 0; k < NA; ++k) {
            const int q = tid + k * kThreads;
            int n, i;
            if (FA) { n = q / BS; i = q % BS; }
            else    { i = q / TN; n = q % TN; }
            sa[n][i] = ra[k];
        }
        __syncthreads();
        if (e + 1 < e1) load(e + 1);    // in flight during the multiply below
#pragma unroll
        for (int r = 0; r < OUT; ++r) {
            int n, j;
            out_coord<BS, FA, TN>(tid + kThreads * r, n, j);
            float s = acc[r];
#pragma unroll
            for (int i = 0; i < BS; ++i)
                s = fmaf(sa[n][i], BWD ? sw[j][i] : sw[i][j], s);
            acc[r] = s;
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < OUT; ++r) {
        int n, j;
        out_coord<BS, FA, TN>(tid + kThreads * r, n, j);
        if (n0 + n < N) out[aidx<FA>(n0 + n, (int64_t)blk * BS + j, N, Fout)] = from_f<T>(acc[r]);
    }
}

// Weight gradient, one CTA per block.  Outputs (i, j) are spread over the
// threads; for bs=8 the 64 outputs are replicated over 4 thread groups that
// split the minibatch and are summed at the end.
template <typename T, typename TD, int BS, int FA>
__global__ void __launch_bounds__(kThreads)
k_simt_updat(GroupPtrs g, TD *__restrict__ dw, const int32_t *__restrict__ coord,
             int N, int C, int K, int accumulate)
{
    constexpr int NOUT = BS * BS;
    constexpr int OUT = NOUT >= kThreads ? NOUT / kThreads : 1;
    constexpr int SPLIT = NOUT >= kThreads ? 1 : kThreads / NOUT;
    __shared__ float sx[kTN][BS + 1];
    __shared__ float sd[kTN][BS + 1];
    __shared__ float red[SPLIT > 1 ? kThreads : 1];
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int c = coord[2 * b], k = coord[2 * b + 1];
    const int part = SPLIT > 1 ? tid / NOUT : 0;   // minibatch split index
    float acc[OUT];
#pragma unroll
    for (int r = 0; r < OUT; ++r) acc[r] = 0.f;

    for (int t = 0; t < g.G; ++t) {
        const T *x = (const T *)g.x[t];
        const T *dy = (const T *)g.dy[t];
        for (int n0 = 0; n0 < N; n0 += kTN) {
            for (int q = tid; q < kTN * BS; q += kThreads) {
                int n, i;
                if (FA) { n = q / BS; i = q % BS; }
                else    { i = q / kTN; n = q % kTN; }
                float vx = 0.f, vd = 0.f;
                if (n0 + n < N) {
                    vx = to_f<T>(x[aidx<FA>(n0 + n, (int64_t)c * BS + i, N, C)]);
                    vd = to_f<T>(dy[aidx<FA>(n0 + n, (int64_t)k * BS + i, N, K)]);
                }
                sx[n][i] = vx;
                sd[n][i] = vd;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < OUT; ++r) {
                int o = (SPLIT > 1 ? tid % NOUT : tid + kThreads * r);
                int i = o / BS, j = o % BS;
                float s = acc[r];
                for (int n = part; n < kTN; n += SPLIT) s = fmaf(sx[n][i], sd[n][j], s);
                acc[r] = s;
            }
            __syncthreads();
        }
    }
    if (SPLIT > 1) {
        red[tid] = acc[0];
        __syncthreads();
        if (tid < NOUT) {
            float s = 0.f;
            for (int p = 0; p < SPLIT; ++p) s += red[tid + p * NOUT];
            acc[0] = s;
        }
    }
#pragma unroll
    for (int r = 0; r < OUT; ++r) {
        int o = tid + kThreads * r;
        if (o >= NOUT) break;
        TD *p = dw + b * NOUT + o;
        float v = acc[r];
        if (accumulate) v += to_f<TD>(*p);
        *p = from_f<TD>(v);
    }
}

template <typename T, int BS>
bsmm_status fwd_bwd_bs(bsmm_ctx *h, const void *in, const void *w, void *out, int N, bool bwd, cudaStream_t s)
{
    const int C = h->R * BS, K = h->S * BS;
    // 64 minibatch rows per CTA, or 256 / BS when that still leaves the GPU short of CTAs (each
    // CTA then walks its column's blocks with a quarter of the work per block)
    const int blocks = bwd ? h->R : h->S;
    const bool small = (int64_t)blocks * ((N + kTN - 1) / kTN) < h->sm_count;
    constexpr int TNS = kThreads / BS;
    dim3 grid(blocks, small ? (N + TNS - 1) / TNS : (N + kTN - 1) / kTN);
    const int32_t *ptr = bwd ? h->d_row_ptr : h->d_col_ptr;
    const int32_t *ent = bwd ? h->d_row_ent : h->d_col_ent;
    int Fin = bwd ? K : C, Fout = bwd ? C : K;
    const T *i_ = (const T *)in;
    const T *w_ = (const T *)w;
    T *o_ = (T *)out;
#define SIMT_FB(TN_)                                                                                     \
    if (h->fa) {                                                                                         \
        if (bwd) k_simt_fwd_bwd<T, BS, 1, true, TN_><<<grid, kThreads, 0, s>>>(i_, w_, o_, ptr, ent, N, Fin, Fout); \
        else     k_simt_fwd_bwd<T, BS, 1, false, TN_><<<grid, kThreads, 0, s>>>(i_, w_, o_, ptr, ent, N, Fin, Fout); \
    } else {                                                                                             \
        if (bwd) k_simt_fwd_bwd<T, BS, 0, true, TN_><<<grid, kThreads, 0, s>>>(i_, w_, o_, ptr, ent, N, Fin, Fout); \
        else     k_simt_fwd_bwd<T, BS, 0, false, TN_><<<grid, kThreads, 0, s>>>(i_, w_, o_, ptr, ent, N, Fin, Fout); \
    }
    if (small) { SIMT_FB(TNS) } else { SIMT_FB(kTN) }
#undef SIMT_FB
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <typename T>
bsmm_status fwd_bwd_t(bsmm_ctx *h, const void *in, const void *w, void *out, int N, bool bwd, cudaStream_t s)
{
    switch (h->bs) {
    case 32: return fwd_bwd_bs<T, 32>(h, in, w, out, N, bwd, s);
    case 16: return fwd_bwd_bs<T, 16>(h, in, w, out, N, bwd, s);
    default: return fwd_bwd_bs<T, 8>(h, in, w, out, N, bwd, s);
    }
}

bsmm_status fwd_bwd(bsmm_ctx *h, const void *in, const void *w, void *out, int N, bsmm_dtype t, bool bwd,
                    cudaStream_t s)
{
    if (t == BSMM_F32) return fwd_bwd_t<float>(h, in, w, out, N, bwd, s);
    if (t == BSMM_F16) return fwd_bwd_t<__half>(h, in, w, out, N, bwd, s);
    return fwd_bwd_t<__nv_bfloat16>(h, in, w, out, N, bwd, s);
}

template <typename T, typename TD, int BS>
bsmm_status updat_bs(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, int acc, cudaStream_t s)
{
    const int C = h->R * BS, K = h->S * BS;
    dim3 grid((unsigned)h->nnz);
    if (h->fa) k_simt_updat<T, TD, BS, 1><<<grid, kThreads, 0, s>>>(g, (TD *)dw, h->d_coord, N, C, K, acc);
    else       k_simt_updat<T, TD, BS, 0><<<grid, kThreads, 0, s>>>(g, (TD *)dw, h->d_coord, N, C, K, acc);
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <typename T, typename TD>
bsmm_status updat_t(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, int acc, cudaStream_t s)
{
    switch (h->bs) {
    case 32: return updat_bs<T, TD, 32>(h, g, dw, N, acc, s);
    case 16: return updat_bs<T, TD, 16>(h, g, dw, N, acc, s);
    default: return updat_bs<T, TD, 8>(h, g, dw, N, acc, s);
    }
}

} // namespace

bsmm_status simt_fprop(bsmm_ctx *h, const void *x, const void *w, void *y, int N, bsmm_dtype t, cudaStream_t s)
{
    return fwd_bwd(h, x, w, y, N, t, false, s);
}

bsmm_status simt_bprop(bsmm_ctx *h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t, cudaStream_t s)
{
    return fwd_bwd(h, dy, w, dx, N, t, true, s);
}

bsmm_status simt_updat(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, bsmm_dtype t, bsmm_dtype dw_t,
                       int accumulate, cudaStream_t s)
{
    if (h->nnz == 0) return BSMM_OK;
    if (t == BSMM_F32) return updat_t<float, float>(h, g, dw, N, accumulate, s);
    if (t == BSMM_F16) {
        if (dw_t == BSMM_F32) return updat_t<__half, float>(h, g, dw, N, accumulate, s);
        return updat_t<__half, __half>(h, g, dw, N, accumulate, s);
    }
    if (dw_t == BSMM_F32) return updat_t<__nv_bfloat16, float>(h, g, dw, N, accumulate, s);
    return updat_t<__nv_bfloat16, __nv_bfloat16>(h, g, dw, N, accumulate, s);
}
