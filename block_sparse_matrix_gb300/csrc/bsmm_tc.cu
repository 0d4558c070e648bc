// tcgen05 tensor-core kernels for 16-bit inputs (fp16 / bf16), float32 accumulation in
// Tensor Memory, operands staged in shared memory by TMA.
//
// The passes are those of BlocksparseMatMul in the blocksparse README ("API
// Documentation: blocksparse.matmul"): fprop y = x.W (__call__), bprop dx = dy.W^T,
// updat dw[b] = x[:, c_b blk]^T . dy[:, k_b blk] and its grouped form
// (group_param_grads) summed over up to 8 timesteps.
//
// Mapping onto the MMA (D[M x N] += A[M x K] . B[K x N], M = 128):
//   fprop/bprop: M = 128 minibatch rows, N = one output block (bs), K = one input
//     block (bs).  A is the activation panel (K-major for (N,C) activations,
//     MN-major for (C,N)), B is the weight block (MN-major for fprop, K-major for
//     bprop, i.e. W^T is read in place).  A CTA owns a window of up to 256/bs output
//     blocks (fprop: block columns, bprop: block rows) for one 128-row minibatch
//     tile; it walks the union of their source blocks, loads each activation panel
//     once and multiplies it with every weight block of the window that uses it.
//     Each output block has its own accumulator columns in TMEM, so bprop needs no
//     atomics, and output blocks without any weight block are written as zeros.
//   updat: M = 128 = up to 128/bs blocks of one block column stacked, N = bs,
//     K = the minibatch (and the timesteps of a group).  The dy panel of the column
//     is shared by the whole stack.
//   bs = 8 runs on 16 x 16 coarse blocks: each coarse block is assembled in shared
//     memory from its four 8 x 8 weight blocks, absent ones loaded from a zero tile,
//     because an M = 128 MMA needs N >= 16 and K = 16.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 issues MMAs (one lane),
// warps 2..5 drain TMEM and write the outputs.  Every mbarrier wait is bounded.
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

#include <algorithm>
#include <cstring>
#include <mutex>

using namespace tc;

namespace {

// ---------------------------------------------------------------------------------------
// Host-side schedules
// ---------------------------------------------------------------------------------------

// One entry of a fprop/bprop window: the source block index (coarse c for fprop,
// coarse k for bprop) and the range of its (slot, ids) records.
struct FbSched {
    int W = 0;                 // output slots per window
    int nwin = 0;              // windows
    int Fslots = 0;            // output blocks (coarse) of the pass
    int32_t *d_win_ptr = nullptr;   // nwin+1, into ents
    int32_t *d_ents = nullptr;      // 3 per entry: src, rec_off, nrec
    int32_t *d_recs = nullptr;      // 5 per record: slot, id(0,0), id(0,1), id(1,0), id(1,1)
    int32_t *d_win_order = nullptr; // nwin, windows by decreasing work
    uint32_t *d_win_mask = nullptr; // nwin, slots that receive at least one block
    size_t bytes = 0;
    bool built = false;
};

struct UpSched {
    int nunits = 0;
    int32_t *d_units = nullptr;     // 3 per unit: coarse column k', rec_off, nrec
    int32_t *d_recs = nullptr;      // 5 per record: coarse c', id(0,0), id(0,1), id(1,0), id(1,1)
    bool built = false;
};

struct TcState {
    FbSched fb[2][6]; // [pass: 0 fprop, 1 bprop][log2 of the window size]
    UpSched up;
    void *d_zero = nullptr;   // 16x16 bf16 zeros for absent 8x8 sub-blocks
    std::mutex mu;
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D tensor map over a row-major [rows][cols] 16-bit array.
bool make_map2d(CUtensorMap *m, const void *base, bsmm_dtype t, uint64_t cols, uint64_t rows, uint32_t box_cols,
                uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUtensorMapDataType dt = t == BSMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

CUtensorMapSwizzle swz_for_row_bytes(int bytes)
{
    return bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                                 : CU_TENSOR_MAP_SWIZZLE_NONE;
}

int pow2_at_least(int v)
{
    int p = 32;
    while (p < v) p <<= 1;
    return p;
}

template <typename T> bool upload(T **d, const std::vector<T> &h)
{
    size_t n = std::max<size_t>(h.size(), 1);
    if (cudaMalloc(d, n * sizeof(T)) != cudaSuccess) return false;
    if (!h.empty() && cudaMemcpy(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
        return false;
    return true;
}

// Block id of fine layout entry (c, k) or -1, from the host row tables.
struct BidLookup {
    const bsmm_ctx *h;
    int32_t operator()(int c, int k) const
    {
        if (c < 0 || c >= h->R || k < 0 || k >= h->S) return -1;
        const int32_t *b = h->h_row_ent.data() + h->h_row_ptr[c];
        const int32_t *e = h->h_row_ent.data() + h->h_row_ptr[c + 1];
        const int32_t *p = std::lower_bound(b, e, k);
        if (p != e && *p == k) return h->h_row_ptr[c] + (int32_t)(p - b);
        return -1;
    }
};

// Output blocks of a pass and their (coarse) edge.
void fb_shape(const bsmm_ctx *h, bool bwd, int &Fslots, int &Fsrc, int &bse)
{
    const int f = h->bs == 8 ? 2 : 1;
    const int Rc = (h->R + f - 1) / f, Sc = (h->S + f - 1) / f;
    bse = h->bs == 8 ? 16 : h->bs;
    Fslots = bwd ? Rc : Sc;
    Fsrc = bwd ? Sc : Rc;
}

// Window size (log2): at most 256 TMEM columns, shrunk until windows x minibatch tiles
// give about two CTAs per SM.
int choose_wlog(const bsmm_ctx *h, bool bwd, int n_tiles)
{
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    int wl = 0;
    while ((2 << wl) * bse <= 256 && (1 << wl) < Fslots) ++wl;
    const int64_t target = 2 * (int64_t)std::max(1, h->sm_count);
    while (wl > 0 && (int64_t)((Fslots + (1 << wl) - 1) >> wl) * n_tiles < target) --wl;
    return wl;
}

// Builds the window schedule of fprop (bwd=false) or bprop (bwd=true) for windows of W slots.
bool build_fb(bsmm_ctx *h, FbSched &fs, bool bwd, int W)
{
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;                       // fine blocks per coarse block edge
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    W = std::min(W, Fslots);
    const int nwin = (Fslots + W - 1) / W;
    BidLookup bid{h};

    std::vector<int32_t> win_ptr(nwin + 1, 0), ents, recs, order(nwin);
    std::vector<uint32_t> mask(nwin, 0);
    std::vector<int64_t> work(nwin, 0);
    std::vector<int32_t> ids(4);
    for (int w = 0; w < nwin; ++w) {
        win_ptr[w] = (int32_t)(ents.size() / 3);
        for (int src = 0; src < Fsrc; ++src) {
            int nrec = 0;
            int rec_off = (int)(recs.size() / 5);
            for (int s = 0; s < W; ++s) {
                int o = w * W + s;
                if (o >= Fslots) break;
                // coarse (c', k') of this (src, out) pair
                int cc = bwd ? o : src, kc = bwd ? src : o;
                bool any = false;
                for (int cs = 0; cs < f; ++cs)
                    for (int ks = 0; ks < f; ++ks) {
                        int b = bid(cc * f + cs, kc * f + ks);
                        ids[cs * 2 + ks] = b;
                        any |= b >= 0;
                    }
                if (!coarse) ids[1] = ids[2] = ids[3] = -1;
                if (!any) continue;
                recs.push_back(s);
                for (int q = 0; q < 4; ++q) recs.push_back(ids[q]);
                ++nrec;
                mask[w] |= 1u << s;
            }
            if (nrec) {
                ents.push_back(src);
                ents.push_back(rec_off);
                ents.push_back(nrec);
                work[w] += nrec + 2;
            }
        }
    }
    win_ptr[nwin] = (int32_t)(ents.size() / 3);
    for (int w = 0; w < nwin; ++w) order[w] = w;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return work[a] > work[b]; });
    fs.W = W;
    fs.nwin = nwin;
    fs.Fslots = Fslots;
    if (!upload(&fs.d_win_ptr, win_ptr) || !upload(&fs.d_ents, ents) || !upload(&fs.d_recs, recs) ||
        !upload(&fs.d_win_order, order) || !upload(&fs.d_win_mask, mask))
        return false;
    fs.built = true;
    return true;
}

bool build_up(bsmm_ctx *h, UpSched &us)
{
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;
    const int Rc = (h->R + f - 1) / f, Sc = (h->S + f - 1) / f;
    const int MS = coarse ? 8 : 128 / h->bs;           // blocks stacked along M
    BidLookup bid{h};
    std::vector<int32_t> units, recs;
    std::vector<int32_t> ids(4);
    for (int kc = 0; kc < Sc; ++kc) {
        std::vector<int32_t> col;   // records of this coarse column
        for (int cc = 0; cc < Rc; ++cc) {
            bool any = false;
            for (int cs = 0; cs < f; ++cs)
                for (int ks = 0; ks < f; ++ks) {
                    int b = bid(cc * f + cs, kc * f + ks);
                    ids[cs * 2 + ks] = b;
                    any |= b >= 0;
                }
            if (!coarse) ids[1] = ids[2] = ids[3] = -1;
            if (!any) continue;
            col.push_back(cc);
            for (int q = 0; q < 4; ++q) col.push_back(ids[q]);
        }
        int n = (int)col.size() / 5;
        for (int s0 = 0; s0 < n; s0 += MS) {
            units.push_back(kc);
            units.push_back((int)(recs.size() / 5) + s0);
            units.push_back(std::min(MS, n - s0));
        }
        recs.insert(recs.end(), col.begin(), col.end());
    }
    us.nunits = (int)units.size() / 3;
    if (!upload(&us.d_units, units) || !upload(&us.d_recs, recs)) return false;
    us.built = true;
    return true;
}

TcState *state(bsmm_ctx *h)
{
    if (!h->tc) {
        TcState *s = new TcState();
        h->tc = s;
    }
    return static_cast<TcState *>(h->tc);
}

// ---------------------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------------------

constexpr int kThreads = 192;

__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\telect.sync r|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

template <bool BF16> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<true>(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<false>(float a, float b)
{
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <bool BF16> __device__ __forceinline__ uint16_t cvt1(float a);
template <> __device__ __forceinline__ uint16_t cvt1<true>(float a)
{
    __nv_bfloat16 v = __float2bfloat16_rn(a);
    return *reinterpret_cast<uint16_t *>(&v);
}
template <> __device__ __forceinline__ uint16_t cvt1<false>(float a)
{
    __half v = __float2half_rn(a);
    return *reinterpret_cast<uint16_t *>(&v);
}

// Compile-time geometry of the fprop/bprop kernel for a (coarse) block edge BSE.
template <int BSE, int FA> struct FbGeo {
    static constexpr int A_BYTES = 128 * BSE * 2;                    // activation panel (128 rows x BSE)
    static constexpr int B_BYTES = BSE * BSE * 2;                    // one (coarse) weight block
    static constexpr int SA = BSE == 32 ? 6 : 8;                     // activation stages
    static constexpr int SB = BSE == 32 ? 24 : 32;                   // weight stages
    static constexpr int SMEM = SA * A_BYTES + SB * B_BYTES;
    static constexpr int KSTEPS = BSE / 16;
    // A operand descriptor parameters
    static constexpr uint32_t A_SWZ = FA ? (BSE == 32 ? SW_64 : SW_32) : SW_128;
    static constexpr uint32_t A_LBO = FA ? 16 : (BSE * 128);         // MN-major: distance of the two 64-row atoms
    static constexpr uint32_t A_SBO = FA ? (8 * BSE * 2) : 1024;
    static constexpr uint32_t A_KSTEP = FA ? 32 : (16 * 128);
};

struct FbParams {
    void *out;
    const int32_t *win_ptr, *ents, *recs, *win_order;
    const uint32_t *win_mask;
    int32_t *status;
    int N;          // minibatch
    int Fout;       // output features (C for bprop, K for fprop)
    int W;          // slots per window
    int Fslots;     // output (coarse) blocks
    int n_tiles;
};

// fprop (BWD=false) / bprop (BWD=true).  BS = fine block size, BSE = 16 when BS = 8.
template <int BS, int FA, bool BWD, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
k_tc_fb(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
        const __grid_constant__ CUtensorMap tm_zero, const FbParams p)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    using G = FbGeo<BSE, FA>;
    constexpr bool COARSE = BS == 8;
    // B operand: fprop reads w[b] as B[K=i][N=j] (MN-major), bprop as B[K=j][N=i] (K-major).
    constexpr uint32_t B_SWZ = COARSE ? SW_NONE : (BS == 32 ? SW_64 : SW_32);
    constexpr uint32_t B_LBO = COARSE ? 128 : 16;
    constexpr uint32_t B_SBO = COARSE ? 256 : 8 * BS * 2;
    constexpr uint32_t B_KSTEP = BWD ? 32 : 16 * BS * 2;
    constexpr uint32_t IDESC = idesc_f16(128, BSE, BF16, FA == 0, !BWD);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + G::SA * G::A_BYTES;
    __shared__ __align__(8) uint64_t fullA[G::SA], emptyA[G::SA], fullB[G::SB], emptyB[G::SB], acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int unit = blockIdx.x;
    const int win = p.win_order[unit / p.n_tiles];
    const int n0 = (unit % p.n_tiles) * 128;
    const int e_begin = p.win_ptr[win], e_end = p.win_ptr[win + 1];
    const int ncols = p.W * BSE;
    const uint32_t alloc_cols = ncols <= 32 ? 32 : ncols <= 64 ? 64 : ncols <= 128 ? 128 : 256;

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < G::SA; ++i) {
            mbar_init(&fullA[i], 1);
            mbar_init(&emptyA[i], 1);
        }
        for (int i = 0; i < G::SB; ++i) {
            mbar_init(&fullB[i], 1);
            mbar_init(&emptyB[i], 1);
        }
        mbar_init(&acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, alloc_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (elect_one()) {
            prefetch_tmap(&tm_act);
            prefetch_tmap(&tm_w);
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int ia = 0, ib = 0;
            for (int e = e_begin; e < e_end && !aborted; ++e) {
                const int src = p.ents[3 * e], roff = p.ents[3 * e + 1], nrec = p.ents[3 * e + 2];
                const int sa = ia % G::SA;
                if (ia >= G::SA && !mbar_wait(&emptyA[sa], ((ia / G::SA) - 1) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                mbar_arrive_expect_tx(&fullA[sa], G::A_BYTES);
                uint8_t *dstA = sA + sa * G::A_BYTES;
                if (FA) {
                    tma_load_2d(dstA, &tm_act, &fullA[sa], src * BSE, n0, pol_act);
                } else {
                    tma_load_2d(dstA, &tm_act, &fullA[sa], n0, src * BSE, pol_act);
                    tma_load_2d(dstA + BSE * 128, &tm_act, &fullA[sa], n0 + 64, src * BSE, pol_act);
                }
                ++ia;
                for (int r = 0; r < nrec; ++r) {
                    const int32_t *rec = p.recs + 5 * (roff + r);
                    const int sb = ib % G::SB;
                    if (ib >= G::SB && !mbar_wait(&emptyB[sb], ((ib / G::SB) - 1) & 1, p.status)) {
                        aborted = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&fullB[sb], G::B_BYTES);
                    uint8_t *dstB = sB + sb * G::B_BYTES;
                    if (!COARSE) {
                        tma_load_2d(dstB, &tm_w, &fullB[sb], 0, rec[1] * BS, pol_w);
                    } else {
                        // sub-block (cs, ks) -> core matrix at (N-group)*256 + (K-group)*128
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int cs = q >> 1, ks = q & 1;
                            const int ng = BWD ? cs : ks, kg = BWD ? ks : cs;
                            uint8_t *d = dstB + ng * 256 + kg * 128;
                            const int32_t id = rec[1 + q];
                            if (id >= 0) tma_load_2d(d, &tm_w, &fullB[sb], 0, id * 8, pol_w);
                            else tma_load_2d(d, &tm_zero, &fullB[sb], 0, 0, pol_w);
                        }
                    }
                    ++ib;
                }
            }
            // Drain: wait until every issued load has landed before the CTA may exit.
            for (int i = std::max(0, ia - G::SA); i < ia; ++i) mbar_wait(&fullA[i % G::SA], (i / G::SA) & 1, p.status);
            for (int i = std::max(0, ib - G::SB); i < ib; ++i) mbar_wait(&fullB[i % G::SB], (i / G::SB) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (elect_one()) {
            uint32_t inited = 0;
            int ia = 0, ib = 0;
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int e = e_begin; e < e_end && !aborted; ++e) {
                const int roff = p.ents[3 * e + 1], nrec = p.ents[3 * e + 2];
                const int sa = ia % G::SA;
                if (!mbar_wait(&fullA[sa], (ia / G::SA) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = a_base + sa * G::A_BYTES;
                for (int r = 0; r < nrec; ++r) {
                    const int slot = p.recs[5 * (roff + r)];
                    const int sb = ib % G::SB;
                    if (!mbar_wait(&fullB[sb], (ib / G::SB) & 1, p.status)) {
                        aborted = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_addr = b_base + sb * G::B_BYTES;
                    const uint32_t d = tmem + slot * BSE;
#pragma unroll
                    for (int ks = 0; ks < G::KSTEPS; ++ks) {
                        uint64_t ad = sdesc(a_addr + ks * G::A_KSTEP, G::A_LBO, G::A_SBO, G::A_SWZ);
                        uint64_t bd = sdesc(b_addr + ks * B_KSTEP, B_LBO, B_SBO, B_SWZ);
                        mma_ss(d, ad, bd, IDESC, ((inited >> slot) & 1u) | (ks > 0 ? 1u : 0u));
                    }
                    inited |= 1u << slot;
                    mma_commit(&emptyB[sb]);
                    ++ib;
                }
                mma_commit(&emptyA[sa]);
                ++ia;
            }
            mma_commit(&acc_full);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = q * 32 + (threadIdx.x & 31);
        const int n = n0 + row;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full, 0, p.status));
        tc_fence_after();
        const uint32_t mask = p.win_mask[win];
        uint16_t *out = static_cast<uint16_t *>(p.out);
        for (int s = 0; s < p.W; ++s) {
            const int o = win * p.W + s;
            if (o >= p.Fslots) break;
            float v[BSE];
            if (ok && ((mask >> s) & 1u)) {
#pragma unroll
                for (int c0 = 0; c0 < BSE; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + s * BSE + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < BSE; ++j) v[j] = 0.f;
            }
            if (n < p.N) {
                const int f0 = o * BSE;
                if (FA) {
                    uint16_t *dst = out + (size_t)n * p.Fout + f0;
                    if (f0 + BSE <= p.Fout) {
#pragma unroll
                        for (int j = 0; j < BSE; j += 8) {
                            uint4 pk;
                            pk.x = pack2<BF16>(v[j], v[j + 1]);
                            pk.y = pack2<BF16>(v[j + 2], v[j + 3]);
                            pk.z = pack2<BF16>(v[j + 4], v[j + 5]);
                            pk.w = pack2<BF16>(v[j + 6], v[j + 7]);
                            *reinterpret_cast<uint4 *>(dst + j) = pk;
                        }
                    } else {
                        for (int j = 0; j < BSE && f0 + j < p.Fout; ++j) dst[j] = cvt1<BF16>(v[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < BSE; ++j)
                        if (f0 + j < p.Fout) out[(size_t)(f0 + j) * p.N + n] = cvt1<BF16>(v[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, alloc_cols);
}

// ---------------------------------------------------------------------------------------
// updat
// ---------------------------------------------------------------------------------------

struct UpMaps {
    CUtensorMap x[8];
    CUtensorMap dy[8];
};

struct UpParams {
    float *dw;
    const int32_t *units, *recs;
    int32_t *status;
    int N, G, accumulate;
};

template <int BSE, int FA> struct UpGeo {
    static constexpr int TK = 64;                                   // minibatch rows per stage
    static constexpr int A_BYTES = 128 * TK * 2;                    // 8 stacked panels max (16 KB)
    static constexpr int B_BYTES = TK * BSE * 2;
    static constexpr int PANEL = TK * BSE * 2;                      // one stacked panel
    static constexpr int STAGES = BSE == 32 ? 5 : 6;
    static constexpr int SMEM = STAGES * (A_BYTES + B_BYTES);
    // fa=1: A MN-major (rows n, BSE features contiguous); fa=0: A K-major (rows = features, n contiguous).
    static constexpr uint32_t A_SWZ = FA ? (BSE == 32 ? SW_64 : SW_32) : SW_128;
    static constexpr uint32_t A_LBO = FA ? PANEL : 16;
    static constexpr uint32_t A_SBO = FA ? 8 * BSE * 2 : 1024;
    static constexpr uint32_t A_KSTEP = FA ? 16 * BSE * 2 : 32;
    static constexpr uint32_t B_SWZ = A_SWZ;
    static constexpr uint32_t B_LBO = FA ? PANEL : 16;
    static constexpr uint32_t B_SBO = A_SBO;
    static constexpr uint32_t B_KSTEP = A_KSTEP;
};

template <int BS, int FA, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
k_tc_updat(const __grid_constant__ UpMaps maps, const UpParams p)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    constexpr bool COARSE = BS == 8;
    constexpr int MS = 128 / BSE;
    using G = UpGeo<BSE, FA>;
    constexpr uint32_t IDESC = idesc_f16(128, BSE, BF16, FA == 1, FA == 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + G::STAGES * G::A_BYTES;
    __shared__ __align__(8) uint64_t full[G::STAGES], empty[G::STAGES], acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int kc = p.units[3 * blockIdx.x];
    const int roff = p.units[3 * blockIdx.x + 1];
    const int nrec = p.units[3 * blockIdx.x + 2];
    const int chunks = (p.N + G::TK - 1) / G::TK;
    const int total = chunks * p.G;

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < G::STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        if (elect_one()) {
            const uint64_t pol = policy_evict_last();
            const uint32_t bytes = nrec * G::PANEL + G::B_BYTES;
            int it = 0;
            for (; it < total && !aborted; ++it) {
                const int t = it / chunks, n0 = (it % chunks) * G::TK;
                const int s = it % G::STAGES;
                if (it >= G::STAGES && !mbar_wait(&empty[s], ((it / G::STAGES) - 1) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], bytes);
                uint8_t *a = sA + s * G::A_BYTES;
                for (int r = 0; r < nrec; ++r) {
                    const int cc = p.recs[5 * (roff + r)];
                    if (FA) tma_load_2d(a + r * G::PANEL, &maps.x[t], &full[s], cc * BSE, n0, pol);
                    else tma_load_2d(a + r * G::PANEL, &maps.x[t], &full[s], n0, cc * BSE, pol);
                }
                uint8_t *b = sB + s * G::B_BYTES;
                if (FA) tma_load_2d(b, &maps.dy[t], &full[s], kc * BSE, n0, pol);
                else tma_load_2d(b, &maps.dy[t], &full[s], n0, kc * BSE, pol);
            }
            for (int i = std::max(0, it - G::STAGES); i < it; ++i)
                mbar_wait(&full[i % G::STAGES], (i / G::STAGES) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
            for (int it = 0; it < total && !aborted; ++it) {
                const int s = it % G::STAGES;
                if (!mbar_wait(&full[s], (it / G::STAGES) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < G::TK / 16; ++ks) {
                    uint64_t ad = sdesc(a_base + s * G::A_BYTES + ks * G::A_KSTEP, G::A_LBO, G::A_SBO, G::A_SWZ);
                    uint64_t bd = sdesc(b_base + s * G::B_BYTES + ks * G::B_KSTEP, G::B_LBO, G::B_SBO, G::B_SWZ);
                    mma_ss(tmem, ad, bd, IDESC, (it > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(&acc_full);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int row = q * 32 + (threadIdx.x & 31);
        const int slot = row / BSE, i = row % BSE;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full, 0, p.status));
        tc_fence_after();
        float v[BSE];
        if (ok && total > 0) {
#pragma unroll
            for (int c0 = 0; c0 < BSE; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < BSE; ++j) v[j] = 0.f;
        }
        if (slot < nrec && ok) {
            const int32_t *rec = p.recs + 5 * (roff + slot);
            if (!COARSE) {
                float *dst = p.dw + ((size_t)rec[1] * BS + i) * BS;
#pragma unroll
                for (int j = 0; j < BS; j += 4) {
                    float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    if (p.accumulate) {
                        float4 a = *reinterpret_cast<float4 *>(dst + j);
                        o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
                    }
                    *reinterpret_cast<float4 *>(dst + j) = o;
                }
            } else {
                const int cs = i / 8, i8 = i % 8;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int32_t id = rec[1 + cs * 2 + ks];
                    if (id < 0) continue;
                    float *dst = p.dw + ((size_t)id * 8 + i8) * 8;
#pragma unroll
                    for (int j = 0; j < 8; j += 4) {
                        float4 o = make_float4(v[ks * 8 + j], v[ks * 8 + j + 1], v[ks * 8 + j + 2], v[ks * 8 + j + 3]);
                        if (p.accumulate) {
                            float4 a = *reinterpret_cast<float4 *>(dst + j);
                            o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
                        }
                        *reinterpret_cast<float4 *>(dst + j) = o;
                    }
                }
            }
        }
        (void)MS;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 32);
}

// ---------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------

template <int BS, int FA, bool BWD, bool BF16>
bsmm_status launch_fb(bsmm_ctx *h, FbSched &fs, const void *act, const void *w, void *out, int N, bsmm_dtype t,
                      cudaStream_t s)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    using G = FbGeo<BSE, FA>;
    TcState *st = state(h);
    const int C = h->R * BS, K = h->S * BS;
    const int Fin = BWD ? K : C, Fout = BWD ? C : K;
    CUtensorMap m_act, m_w, m_zero;
    bool ok;
    if (FA) ok = make_map2d(&m_act, act, t, Fin, N, BSE, 128, swz_for_row_bytes(BSE * 2));
    else ok = make_map2d(&m_act, act, t, N, Fin, 64, BSE, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint64_t wrows = (uint64_t)std::max<int64_t>(h->nnz, 1) * BS;
    const void *wp = h->nnz > 0 ? w : st->d_zero;
    if (BS == 8) ok = ok && make_map2d(&m_w, wp, t, 8, h->nnz > 0 ? wrows : 16, 8, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    else ok = ok && make_map2d(&m_w, wp, t, BS, h->nnz > 0 ? wrows : BS, BS, BS, swz_for_row_bytes(BS * 2));
    ok = ok && make_map2d(&m_zero, st->d_zero, t, 8, 16, 8, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return BSMM_ERR_CUDA;
    FbParams p;
    p.out = out;
    p.win_ptr = fs.d_win_ptr;
    p.ents = fs.d_ents;
    p.recs = fs.d_recs;
    p.win_order = fs.d_win_order;
    p.win_mask = fs.d_win_mask;
    p.status = h->d_status;
    p.N = N;
    p.Fout = Fout;
    p.W = fs.W;
    p.Fslots = fs.Fslots;
    p.n_tiles = (N + 127) / 128;
    const int smem = G::SMEM + 1024;
    auto kern = k_tc_fb<BS, FA, BWD, BF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSMM_ERR_CUDA;
    dim3 grid(fs.nwin * p.n_tiles);
    kern<<<grid, kThreads, smem, s>>>(m_act, m_w, m_zero, p);
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int BS, int FA, bool BF16>
bsmm_status launch_up(bsmm_ctx *h, UpSched &us, const GroupPtrs &g, float *dw, int N, bsmm_dtype t, int acc,
                      cudaStream_t s)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    using G = UpGeo<BSE, FA>;
    const int C = h->R * BS, K = h->S * BS;
    UpMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int i = 0; i < g.G; ++i) {
        bool ok;
        if (FA) {
            ok = make_map2d(&maps.x[i], g.x[i], t, C, N, BSE, G::TK, swz_for_row_bytes(BSE * 2)) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, K, N, BSE, G::TK, swz_for_row_bytes(BSE * 2));
        } else {
            ok = make_map2d(&maps.x[i], g.x[i], t, N, C, G::TK, BSE, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, N, K, G::TK, BSE, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return BSMM_ERR_CUDA;
    }
    UpParams p;
    p.dw = dw;
    p.units = us.d_units;
    p.recs = us.d_recs;
    p.status = h->d_status;
    p.N = N;
    p.G = g.G;
    p.accumulate = acc;
    const int smem = G::SMEM + 1024;
    auto kern = k_tc_updat<BS, FA, BF16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSMM_ERR_CUDA;
    kern<<<us.nunits, kThreads, smem, s>>>(maps, p);
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <bool BWD>
bsmm_status fb_dispatch(bsmm_ctx *h, const void *act, const void *w, void *out, int N, bsmm_dtype t, cudaStream_t s)
{
    TcState *st = state(h);
    const int wl = choose_wlog(h, BWD, (N + 127) / 128);
    FbSched &fs = st->fb[BWD ? 1 : 0][wl];
    {
        std::lock_guard<std::mutex> lk(st->mu);
        if (!st->d_zero) {
            if (cudaMalloc(&st->d_zero, 4096) != cudaSuccess) return BSMM_ERR_OOM;
            if (cudaMemset(st->d_zero, 0, 4096) != cudaSuccess) return BSMM_ERR_CUDA;
        }
        if (!fs.built && !build_fb(h, fs, BWD, 1 << wl)) return BSMM_ERR_OOM;
    }
    const bool bf = t == BSMM_BF16;
#define FB_CASE(BS_, FA_)                                                                                   \
    if (h->bs == BS_ && h->fa == FA_)                                                                       \
        return bf ? launch_fb<BS_, FA_, BWD, true>(h, fs, act, w, out, N, t, s)                            \
                  : launch_fb<BS_, FA_, BWD, false>(h, fs, act, w, out, N, t, s);
    FB_CASE(32, 1)
    FB_CASE(32, 0)
    FB_CASE(16, 1)
    FB_CASE(16, 0)
    FB_CASE(8, 1)
    FB_CASE(8, 0)
#undef FB_CASE
    return BSMM_ERR_UNSUPPORTED;
}

} // namespace

bool tc_supported(bsmm_ctx *h, bsmm_dtype t)
{
    if (t != BSMM_F16 && t != BSMM_BF16) return false;
    if (!encode_fn()) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
    return major == 10 && minor == 3;
}

bsmm_status tc_fprop(bsmm_ctx *h, const void *x, const void *w, void *y, int N, bsmm_dtype t, cudaStream_t s)
{
    return fb_dispatch<false>(h, x, w, y, N, t, s);
}

bsmm_status tc_bprop(bsmm_ctx *h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t, cudaStream_t s)
{
    return fb_dispatch<true>(h, dy, w, dx, N, t, s);
}

bsmm_status tc_updat(bsmm_ctx *h, const GroupPtrs &g, float *dw, int N, bsmm_dtype t, int accumulate,
                     cudaStream_t s)
{
    TcState *st = state(h);
    {
        std::lock_guard<std::mutex> lk(st->mu);
        if (!st->up.built && !build_up(h, st->up)) return BSMM_ERR_OOM;
    }
    if (st->up.nunits == 0) return BSMM_OK;
    const bool bf = t == BSMM_BF16;
#define UP_CASE(BS_, FA_)                                                                         \
    if (h->bs == BS_ && h->fa == FA_)                                                             \
        return bf ? launch_up<BS_, FA_, true>(h, st->up, g, dw, N, t, accumulate, s)             \
                  : launch_up<BS_, FA_, false>(h, st->up, g, dw, N, t, accumulate, s);
    UP_CASE(32, 1)
    UP_CASE(32, 0)
    UP_CASE(16, 1)
    UP_CASE(16, 0)
    UP_CASE(8, 1)
    UP_CASE(8, 0)
#undef UP_CASE
    return BSMM_ERR_UNSUPPORTED;
}

void tc_release(bsmm_ctx *h)
{
    if (!h->tc) return;
    TcState *st = static_cast<TcState *>(h->tc);
    for (auto &pass : st->fb)
        for (auto &f : pass) {
        cudaFree(f.d_win_ptr);
        cudaFree(f.d_ents);
        cudaFree(f.d_recs);
        cudaFree(f.d_win_order);
        cudaFree(f.d_win_mask);
        }
    cudaFree(st->up.d_units);
    cudaFree(st->up.d_recs);
    cudaFree(st->d_zero);
    delete st;
    h->tc = nullptr;
}
