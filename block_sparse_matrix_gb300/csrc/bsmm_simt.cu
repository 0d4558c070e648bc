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
#include "tc_common.cuh"

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
// A CTA walks its LUT entries D at a time.  The schedule (LUT entries: fixed once the handle
// exists) is read before the wait on the previous kernel; the D weight blocks and input panels of
// a group are then loaded into registers together, so a group costs one memory round trip, and
// the next group's loads are in flight while the current group is multiplied out of shared memory.
// Panel rows have a 16-byte pitch, so a thread reads four reduction terms with one vector load.
// Every output sums its entries in LUT order and each entry's terms in increasing index order.
template <typename T, int BS, int FA, bool BWD, int TN, int D>
__global__ void __launch_bounds__(kThreads, 1)
k_simt_fwd_bwd(const T *__restrict__ in, const T *__restrict__ w, T *__restrict__ out,
               const int32_t *__restrict__ ptr, const int32_t *__restrict__ ent,
               int N, int Fin, int Fout)
{
    constexpr int OUT = TN * BS / kThreads;
    constexpr int NW = (BS * BS + kThreads - 1) / kThreads;   // weight elements per thread and entry
    constexpr int NA = TN * BS / kThreads;                     // panel elements per thread and entry
    constexpr int PA = BS + 4;                                 // panel row pitch (floats)
    __shared__ float sw[D][BS][BS + 1];
    __shared__ __align__(16) float sa[D][TN][PA];
    tc::pdl_launch_dependents();        // holds no tensor memory: the next kernel may start
    const int tid = threadIdx.x;
    const int blk = blockIdx.x;         // output block column (fprop) / row (bprop)
    const int n0 = blockIdx.y * TN;
    const int e0 = ptr[blk], e1 = ptr[blk + 1];

    int bid[D], src[D];                 // weight block id and source block index of each entry
    auto sched = [&](int e) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            bid[d] = 0;
            src[d] = 0;
            if (e + d < e1) {
                if (BWD) { bid[d] = e + d; src[d] = ent[e + d]; }
                else     { bid[d] = ent[2 * (e + d)]; src[d] = ent[2 * (e + d) + 1]; }
            }
        }
    };
    float rw[D][NW], ra[D][NA];
    auto load = [&](int e) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const bool live = e + d < e1;
            const T *wb = w + (size_t)bid[d] * BS * BS;
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const int q = tid + k * kThreads;
                rw[d][k] = live && q < BS * BS ? to_f<T>(wb[q]) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < NA; ++k) {
                const int q = tid + k * kThreads;
                int n, i;
                if (FA) { n = q / BS; i = q % BS; }
                else    { i = q / TN; n = q % TN; }
                ra[d][k] = live && n0 + n < N
                               ? to_f<T>(in[aidx<FA>(n0 + n, (int64_t)src[d] * BS + i, N, Fin)]) : 0.f;
            }
        }
    };

    float acc[OUT];
#pragma unroll
    for (int r = 0; r < OUT; ++r) acc[r] = 0.f;

    sched(e0);
    tc::pdl_wait();                     // the previous kernel's writes (in, w, out) are settled
    if (e0 < e1) load(e0);
    for (int e = e0; e < e1; e += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const int q = tid + k * kThreads;
                if (q < BS * BS) sw[d][q / BS][q % BS] = rw[d][k];
            }
#pragma unroll
            for (int k = 0; k < NA; ++k) {
                const int q = tid + k * kThreads;
                int n, i;
                if (FA) { n = q / BS; i = q % BS; }
                else    { i = q / TN; n = q % TN; }
                sa[d][n][i] = ra[d][k];
            }
        }
        __syncthreads();
        if (e + D < e1) {               // the next group, in flight during the multiply below
            sched(e + D);
            load(e + D);
        }
#pragma unroll
        for (int d = 0; d < D; ++d) {
            if (e + d >= e1) break;     // uniform over the CTA
#pragma unroll
            for (int i = 0; i < BS; i += 4) {
#pragma unroll
                for (int r = 0; r < OUT; ++r) {
                    int n, j;
                    out_coord<BS, FA, TN>(tid + kThreads * r, n, j);
                    const float4 a = *reinterpret_cast<const float4 *>(&sa[d][n][i]);
                    float s = acc[r];
                    s = fmaf(a.x, BWD ? sw[d][j][i + 0] : sw[d][i + 0][j], s);
                    s = fmaf(a.y, BWD ? sw[d][j][i + 1] : sw[d][i + 1][j], s);
                    s = fmaf(a.z, BWD ? sw[d][j][i + 2] : sw[d][i + 2][j], s);
                    s = fmaf(a.w, BWD ? sw[d][j][i + 3] : sw[d][i + 3][j], s);
                    acc[r] = s;
                }
            }
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
// split the minibatch and are summed at the end.  For bs=32 a thread owns four
// consecutive i of one j, so one vector read of x serves four outputs.  Every
// output sums over the timesteps and the minibatch in increasing order.
template <typename T, typename TD, int BS, int FA>
__global__ void __launch_bounds__(kThreads)
k_simt_updat(GroupPtrs g, TD *__restrict__ dw, const int32_t *__restrict__ coord,
             int N, int C, int K, int accumulate)
{
    constexpr int NOUT = BS * BS;
    constexpr int OUT = NOUT >= kThreads ? NOUT / kThreads : 1;
    constexpr int SPLIT = NOUT >= kThreads ? 1 : kThreads / NOUT;
    constexpr bool QUAD = OUT % 4 == 0;
    constexpr int PX = BS + 4;                   // x row pitch (floats): rows start on 16 bytes
    __shared__ __align__(16) float sx[kTN][PX];
    __shared__ float sd[kTN][BS + 1];
    __shared__ float red[SPLIT > 1 ? kThreads : 1];
    tc::pdl_launch_dependents();                 // holds no tensor memory: the next kernel may start
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    const int c = coord[2 * b], k = coord[2 * b + 1];
    const int part = SPLIT > 1 ? tid / NOUT : 0;   // minibatch split index
    int oi[OUT], oj[OUT];
#pragma unroll
    for (int r = 0; r < OUT; ++r) {
        const int o = QUAD ? (tid / BS) * OUT * BS + r * BS + tid % BS
                           : (SPLIT > 1 ? tid % NOUT : tid + kThreads * r);
        oi[r] = o / BS;
        oj[r] = o % BS;
    }
    float acc[OUT];
#pragma unroll
    for (int r = 0; r < OUT; ++r) acc[r] = 0.f;
    tc::pdl_wait();                              // the previous kernel's writes (x, dy, dw) are settled

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
            if (QUAD) {
                const int i0 = oi[0], j = oj[0];
#pragma unroll 4
                for (int n = 0; n < kTN; ++n) {
                    const float d = sd[n][j];
#pragma unroll
                    for (int r = 0; r < OUT; r += 4) {
                        const float4 a = *reinterpret_cast<const float4 *>(&sx[n][i0 + r]);
                        acc[r + 0] = fmaf(a.x, d, acc[r + 0]);
                        acc[r + 1] = fmaf(a.y, d, acc[r + 1]);
                        acc[r + 2] = fmaf(a.z, d, acc[r + 2]);
                        acc[r + 3] = fmaf(a.w, d, acc[r + 3]);
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < OUT; ++r) {
                    float s = acc[r];
                    for (int n = part; n < kTN; n += SPLIT) s = fmaf(sx[n][oi[r]], sd[n][oj[r]], s);
                    acc[r] = s;
                }
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
        if (SPLIT > 1 && tid >= NOUT) break;
        TD *p = dw + b * NOUT + oi[r] * BS + oj[r];
        float v = acc[r];
        if (accumulate) v += to_f<TD>(*p);
        *p = from_f<TD>(v);
    }
}

// Every SIMT pass launches with programmatic dependent launch: it reads its schedule while the
// previous kernel on the stream finishes, and waits in pdl_wait() before touching activations,
// weights or outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_simt(void (*kern)(KArgs...), dim3 grid, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// LUT entries staged per group: as many as fit in 45 KB of static shared memory, at most 8 for
// the short tiles (few CTAs: a block column should take one round trip) and 4 for 64-row tiles
// (enough CTAs to hide the latency).
template <int BS, int TN>
constexpr int simt_group()
{
    return (45 * 1024) / ((BS * (BS + 1) + TN * (BS + 4)) * 4) >= (TN == kTN ? 4 : 8)
               ? (TN == kTN ? 4 : 8)
               : (45 * 1024) / ((BS * (BS + 1) + TN * (BS + 4)) * 4);
}

template <typename T, int BS, int TN>
cudaError_t launch_fb(bsmm_ctx *h, dim3 grid, bool bwd, const T *in, const T *w, T *out, int N, int Fin, int Fout,
                      cudaStream_t s)
{
    constexpr int D = simt_group<BS, TN>();
    static_assert(D >= 1, "one LUT entry must fit in shared memory");
    const int32_t *ptr = bwd ? h->d_row_ptr : h->d_col_ptr;
    const int32_t *ent = bwd ? h->d_row_ent : h->d_col_ent;
    if (h->fa) {
        if (bwd) return launch_simt(k_simt_fwd_bwd<T, BS, 1, true, TN, D>, grid, s, in, w, out, ptr, ent, N, Fin, Fout);
        return launch_simt(k_simt_fwd_bwd<T, BS, 1, false, TN, D>, grid, s, in, w, out, ptr, ent, N, Fin, Fout);
    }
    if (bwd) return launch_simt(k_simt_fwd_bwd<T, BS, 0, true, TN, D>, grid, s, in, w, out, ptr, ent, N, Fin, Fout);
    return launch_simt(k_simt_fwd_bwd<T, BS, 0, false, TN, D>, grid, s, in, w, out, ptr, ent, N, Fin, Fout);
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
    const int Fin = bwd ? K : C, Fout = bwd ? C : K;
    const T *i_ = (const T *)in;
    const T *w_ = (const T *)w;
    T *o_ = (T *)out;
    const cudaError_t le = small ? launch_fb<T, BS, TNS>(h, grid, bwd, i_, w_, o_, N, Fin, Fout, s)
                                 : launch_fb<T, BS, kTN>(h, grid, bwd, i_, w_, o_, N, Fin, Fout, s);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
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
    const dim3 grid((unsigned)h->nnz);
    const cudaError_t le =
        h->fa ? launch_simt(k_simt_updat<T, TD, BS, 1>, grid, s, g, (TD *)dw, (const int32_t *)h->d_coord, N, C, K, acc)
              : launch_simt(k_simt_updat<T, TD, BS, 0>, grid, s, g, (TD *)dw, (const int32_t *)h->d_coord, N, C, K, acc);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
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
