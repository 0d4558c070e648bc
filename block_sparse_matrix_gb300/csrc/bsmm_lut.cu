// Lookup-table construction and weight initialisation on the device.
//
// BlocksparseMatMul(layout, ...) in the blocksparse README ("API Documentation:
// blocksparse.matmul") keeps a 0/1 block layout; block_coord(block) maps a block
// id to its (c, k) layout coordinates.  Block ids follow the row-major scan of
// the layout.  From the layout these kernels build:
//   row_ptr/row_ent  per input block row c: the k of each block (ids are contiguous)
//   col_ptr/col_ent  per output block column k: (block id, c) pairs, c increasing
//   coord            per block id: (c, k)
// One thread owns one row or one column and scans it serially, so the tables
// are deterministic and need no atomics.
#include "bsmm_internal.cuh"

namespace {

__global__ void k_row_count(const uint8_t *__restrict__ L, int R, int S, int32_t *__restrict__ cnt)
{
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= R) return;
    int n = 0;
    for (int k = 0; k < S; ++k) n += L[(size_t)c * S + k] != 0;
    cnt[c] = n;
}

__global__ void k_col_count(const uint8_t *__restrict__ L, int R, int S, int32_t *__restrict__ cnt)
{
    int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= S) return;
    int n = 0;
    for (int c = 0; c < R; ++c) n += L[(size_t)c * S + k] != 0;
    cnt[k] = n;
}

// Exclusive scan of cnt[0..n) into ptr[0..n] by one block (setup only).
__global__ void k_scan(const int32_t *__restrict__ cnt, int32_t *__restrict__ ptr, int n)
{
    __shared__ int32_t carry;
    __shared__ int32_t part[1024];
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        int i = base + threadIdx.x;
        int v = i < n ? cnt[i] : 0;
        part[threadIdx.x] = v;
        __syncthreads();
        // Hillis-Steele inclusive scan in shared memory
        for (int off = 1; off < (int)blockDim.x; off <<= 1) {
            int t = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
            __syncthreads();
            part[threadIdx.x] += t;
            __syncthreads();
        }
        if (i < n) ptr[i] = carry + part[threadIdx.x] - v;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry += part[threadIdx.x];
        __syncthreads();
    }
    if (threadIdx.x == 0) ptr[n] = carry;
}

__global__ void k_row_fill(const uint8_t *__restrict__ L, int R, int S, const int32_t *__restrict__ row_ptr,
                           int32_t *__restrict__ row_ent, int32_t *__restrict__ coord, int32_t *__restrict__ bid)
{
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= R) return;
    int e = row_ptr[c];
    for (int k = 0; k < S; ++k) {
        if (L[(size_t)c * S + k]) {
            row_ent[e] = k;
            coord[2 * e] = c;
            coord[2 * e + 1] = k;
            bid[(size_t)c * S + k] = e;
            ++e;
        } else {
            bid[(size_t)c * S + k] = -1;
        }
    }
}

__global__ void k_col_fill(const uint8_t *__restrict__ L, int R, int S, const int32_t *__restrict__ col_ptr,
                           const int32_t *__restrict__ bid, int32_t *__restrict__ col_ent)
{
    int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= S) return;
    int e = col_ptr[k];
    for (int c = 0; c < R; ++c) {
        if (L[(size_t)c * S + k]) {
            col_ent[2 * e] = bid[(size_t)c * S + k];
            col_ent[2 * e + 1] = c;
            ++e;
        }
    }
}

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// identity_init: w[b][i][j] = (c_b == k_b && i == j) ? 1 : 0.
template <typename T>
__global__ void k_identity(T *__restrict__ w, const int32_t *__restrict__ coord, int64_t nnz, int bs)
{
    int64_t total = nnz * bs * bs;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total;
         q += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = q / (bs * bs);
        int r = (int)(q % (bs * bs));
        int i = r / bs, j = r % bs;
        bool one = coord[2 * b] == coord[2 * b + 1] && i == j;
        w[q] = from_f<T>(one ? 1.0f : 0.0f);
    }
}

} // namespace

bsmm_status lut_build(bsmm_ctx *h, const uint8_t *layout_host, cudaStream_t s)
{
    const int R = h->R, S = h->S;
    const size_t RS = (size_t)R * S;
    int32_t *d_cnt = nullptr;
    if (cudaMalloc(&h->d_layout, RS) != cudaSuccess) return BSMM_ERR_OOM;
    if (cudaMalloc(&h->d_bid, RS * sizeof(int32_t)) != cudaSuccess) return BSMM_ERR_OOM;
    if (cudaMalloc(&h->d_row_ptr, (R + 1) * sizeof(int32_t)) != cudaSuccess) return BSMM_ERR_OOM;
    if (cudaMalloc(&h->d_col_ptr, (S + 1) * sizeof(int32_t)) != cudaSuccess) return BSMM_ERR_OOM;
    if (cudaMalloc(&d_cnt, (size_t)(R > S ? R : S) * sizeof(int32_t)) != cudaSuccess) return BSMM_ERR_OOM;

    bsmm_status st = BSMM_OK;
    do {
        if (cudaMemcpyAsync(h->d_layout, layout_host, RS, cudaMemcpyHostToDevice, s) != cudaSuccess) {
            st = BSMM_ERR_CUDA;
            break;
        }
        const int tb = 128;
        k_row_count<<<(R + tb - 1) / tb, tb, 0, s>>>(h->d_layout, R, S, d_cnt);
        k_scan<<<1, 1024, 0, s>>>(d_cnt, h->d_row_ptr, R);
        k_col_count<<<(S + tb - 1) / tb, tb, 0, s>>>(h->d_layout, R, S, d_cnt);
        k_scan<<<1, 1024, 0, s>>>(d_cnt, h->d_col_ptr, S);
        g_bsmm_launches += 4;
        int32_t nnz32 = 0;
        if (cudaMemcpyAsync(&nnz32, h->d_row_ptr + R, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            st = BSMM_ERR_CUDA;
            break;
        }
        h->nnz = nnz32;
        size_t ne = (size_t)(nnz32 > 0 ? nnz32 : 1);
        if (cudaMalloc(&h->d_row_ent, ne * sizeof(int32_t)) != cudaSuccess ||
            cudaMalloc(&h->d_col_ent, 2 * ne * sizeof(int32_t)) != cudaSuccess ||
            cudaMalloc(&h->d_coord, 2 * ne * sizeof(int32_t)) != cudaSuccess) {
            st = BSMM_ERR_OOM;
            break;
        }
        k_row_fill<<<(R + tb - 1) / tb, tb, 0, s>>>(h->d_layout, R, S, h->d_row_ptr, h->d_row_ent, h->d_coord,
                                                     h->d_bid);
        k_col_fill<<<(S + tb - 1) / tb, tb, 0, s>>>(h->d_layout, R, S, h->d_col_ptr, h->d_bid, h->d_col_ent);
        g_bsmm_launches += 2;
        if (cudaGetLastError() != cudaSuccess) {
            st = BSMM_ERR_CUDA;
            break;
        }
        // Host mirrors
        h->h_row_ptr.resize(R + 1);
        h->h_col_ptr.resize(S + 1);
        h->h_row_ent.resize(nnz32);
        h->h_col_ent.resize(2 * (size_t)nnz32);
        h->h_coord.resize(2 * (size_t)nnz32);
        if (cudaMemcpyAsync(h->h_row_ptr.data(), h->d_row_ptr, (R + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, s) ||
            cudaMemcpyAsync(h->h_col_ptr.data(), h->d_col_ptr, (S + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, s)) {
            st = BSMM_ERR_CUDA;
            break;
        }
        if (nnz32 > 0 &&
            (cudaMemcpyAsync(h->h_row_ent.data(), h->d_row_ent, nnz32 * sizeof(int32_t), cudaMemcpyDeviceToHost, s) ||
             cudaMemcpyAsync(h->h_col_ent.data(), h->d_col_ent, 2 * (size_t)nnz32 * sizeof(int32_t),
                             cudaMemcpyDeviceToHost, s) ||
             cudaMemcpyAsync(h->h_coord.data(), h->d_coord, 2 * (size_t)nnz32 * sizeof(int32_t),
                             cudaMemcpyDeviceToHost, s))) {
            st = BSMM_ERR_CUDA;
            break;
        }
        if (cudaStreamSynchronize(s) != cudaSuccess) st = BSMM_ERR_CUDA;
    } while (0);
    cudaFree(d_cnt);
    return st;
}

bsmm_status launch_identity_init(bsmm_ctx *h, void *w, bsmm_dtype t, cudaStream_t s)
{
    if (h->nnz == 0) return BSMM_OK;
    int64_t total = h->nnz * h->bs * h->bs;
    int grid = (int)((total + 255) / 256);
    int cap = h->sm_count * 8;
    if (grid > cap) grid = cap;
    if (t == BSMM_F32)
        k_identity<float><<<grid, 256, 0, s>>>((float *)w, h->d_coord, h->nnz, h->bs);
    else if (t == BSMM_F16)
        k_identity<__half><<<grid, 256, 0, s>>>((__half *)w, h->d_coord, h->nnz, h->bs);
    else
        k_identity<__nv_bfloat16><<<grid, 256, 0, s>>>((__nv_bfloat16 *)w, h->d_coord, h->nnz, h->bs);
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}
