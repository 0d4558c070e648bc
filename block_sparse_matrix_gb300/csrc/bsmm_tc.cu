// tcgen05 tensor-core kernels for 16-bit inputs (fp16 / bf16), float32 accumulation in
// Tensor Memory, operands staged in shared memory by TMA.
//
// The passes are those of BlocksparseMatMul in the blocksparse README ("API
// Documentation: blocksparse.matmul"): fprop y = x.W (__call__), bprop dx = dy.W^T,
// updat dw[b] = x[:, c_b blk]^T . dy[:, k_b blk] and its grouped form
// (group_param_grads) summed over up to 8 timesteps.
//
// Kernel families (the dispatch is in fbd_try and tc_updat near the end of this file):
//   k_tc_fbd_pair    fprop/bprop, bs = 32, dense layouts, minibatch > 64: CTA pairs with
//                    two-SM MMAs (M256 x N256 x K16) on tiles of 8 output blocks x 256 rows,
//                    absent blocks as zero tiles.
//   k_tc_fbd_split   fprop/bprop, bs = 32, dense layouts, minibatch <= 64: clusters of 4 CTAs
//                    split a 4-block x 64-row tile's sources and reduce in distributed shared
//                    memory.
//   k_tc_fb          fprop/bprop, any block size: a CTA owns a window of output blocks for a
//                    128-row tile and issues one N = bs MMA per present block (bs = 8 runs on
//                    16 x 16 coarse blocks with zero tiles).
//   k_tc_updat_pair  updat, bs = 32, dense layouts: CTA pairs with two-SM MMAs on 256 x 256
//                    tiles of x^T.dy, persistent, double-buffered accumulators.
//   k_tc_updat       updat, any block size: 128/bs blocks of one block column stacked along M.
//   k_tc_fbd, k_tc_updat_dense   one-CTA forms of the dense tiles (fallback, and a second
//                    implementation the tests compare with bit for bit).
// All of them are warp-specialised (producer warps issue each stage's TMA loads as one
// instruction, one thread issues the MMAs, producer or epilogue warps drain TMEM), launch
// with programmatic dependent launch, and bound every mbarrier wait.
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

using namespace tc;

namespace {

// ---------------------------------------------------------------------------------------
// Host-side schedules
// ---------------------------------------------------------------------------------------

// Schedule of fprop/bprop: one packed word stream per window of W output blocks, cut
// into chunks; a chunk is what one pipeline stage holds.
//   chunk header: (ne << 8) | nr     -- ne entries then nr records follow; 0 ends the stream
//   entry word:   (src << 8) | nrec  -- src = source panel group whose activations are loaded
//                 into the stage; its nrec records are the next nrec records of the chunk.  With
//                 (N,C) activations a group is the 128/(2 bs) adjacent source blocks (coarse c for
//                 fprop, coarse k for bprop) that make one 128-byte row; with (C,N) it is one block
//   record (bs 32/16): ((block id + 1) << 7) | (sub << 5) | slot, sub = block within the group
//   record (bs 8, coarse 16x16 block): 4 words, ((id00 + 1) << 7) | (sub << 5) | slot,
//                 id01 + 1, id10 + 1, id11 + 1, where idXY is the 8x8 block (2c'+X, 2k'+Y),
//                 0 = absent
// Streams start on 16-byte boundaries and are padded to a multiple of 4 words so a CTA
// can bulk-copy its window into shared memory.
// (N,C) activation panels of the window kernel: row bytes and source blocks per row (a 32-feature
// block alone in a 64-byte row; 16-feature blocks four to a 128-byte row).
__host__ __device__ constexpr int fb_row_bytes(int bse) { return bse == 32 ? 64 : 128; }
__host__ __device__ constexpr int fb_row_sources(int fa, int bse) { return fa ? fb_row_bytes(bse) / (2 * bse) : 1; }

struct FbSched {
    int W = 0;                      // output slots per window
    int nwin = 0;                   // windows
    int Fslots = 0;                 // output blocks (coarse) of the pass
    int max_words = 0;              // longest window stream
    uint32_t *d_stream = nullptr;
    // nwin descriptors in launch order (windows by decreasing work): window, word offset of its
    // stream, padded length in words, slots that receive at least one block -- one 16-byte load
    // gives a CTA everything it needs before the stream's bulk copy
    int4 *d_win_desc = nullptr;
    // binned windows only: nwin * W output blocks (slot s of window w at w * W + s, -1 = unused);
    // null for windows of W consecutive output blocks
    int32_t *d_win_out = nullptr;
    bool built = false;
    bool too_big = false;           // a window stream exceeds the shared-memory budget
};

// Schedule of updat: units of up to 128/bs (coarse) blocks of one block column, dealt
// round-robin to persistent CTAs.  Each CTA's units sit in one fixed-size table that the
// CTA bulk-copies into shared memory:
//   table word 0: number of units; unit u at word 4 + u * kUnitWords:
//     k' (coarse block column), nrec, then nrec records of 5 words:
//     c' (coarse block row), id00, id01, id10, id11 (block ids of the 8x8 sub-blocks for
//     bs 8, id00 = the block for bs 32/16, -1 = absent)
constexpr int kUnitWords = 44;
constexpr int kUnitsPerCta = 64;
constexpr int kTableWords = 4 + kUnitsPerCta * kUnitWords;

struct UpSched {
    int ctas = 0;
    int32_t *d_table = nullptr;     // ctas * kTableWords
    bool built = false;
};

struct TcState {
    std::map<uint64_t, FbSched> fb;   // key: pass, window log2, chunk entries, chunk records
    UpSched up;
    struct UpDenseSched *upd = nullptr;
    struct UpPairSched *upp = nullptr;
    struct FbDenseSched *fbd[4] = {};   // dense-tile fprop / bprop; + 2: CTA-pair schedules
    void *d_zero = nullptr;   // zero buffer: 8x8 zero tiles for absent sub-blocks of 16x16 coarse blocks
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

// The same over any element type (float32 dW for the weight-gradient epilogue).
bool make_map2d_dt(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols,
                   uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * (uint64_t)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

CUtensorMapSwizzle swz_for_row_bytes(int bytes)
{
    return bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                                 : CU_TENSOR_MAP_SWIZZLE_NONE;
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
// give at least one CTA per SM.  Larger windows load each activation panel for more
// output blocks, smaller ones spread the work over more SMs.
int choose_wlog(const bsmm_ctx *h, bool bwd, int n_tiles)
{
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    int wl = 0;
    while ((2 << wl) * bse <= 256 && (1 << wl) < Fslots) ++wl;
    const int64_t target = (int64_t)std::max(1, h->sm_count);
    while (wl > 0 && (int64_t)((Fslots + (1 << wl) - 1) >> wl) * n_tiles < target) --wl;
    return wl;
}

// Builds the window schedule of fprop (bwd=false) or bprop (bwd=true) for windows of W
// slots.  A chunk holds at most e_max entries and r_max records and issues at most 32 TMA
// loads (a_ops per entry, b_ops per record), one per lane of the producer warp.  Sets
// too_big when a window's stream would exceed max_words.
bool build_fb(bsmm_ctx *h, FbSched &fs, bool bwd, int W, int e_max, int r_max, int a_ops, int b_ops,
              int max_words, const std::vector<std::vector<int>> *bins = nullptr)
{
    if (e_max < 1 || r_max < 1 || a_ops + r_max * b_ops > 32) return false;
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;                       // fine blocks per coarse block edge
    const int rw = coarse ? 4 : 1;                      // words per record
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    const int gc = fb_row_sources(h->fa, bse);         // source blocks per activation panel row
    W = std::min(W, Fslots);
    int nwin = (Fslots + W - 1) / W;
    std::vector<int32_t> win_out;
    if (bins) {
        nwin = (int)bins->size();
        W = 0;
        for (const auto &b : *bins) W = std::max(W, (int)b.size());
        if (W < 1 || W > 32) return false;
        win_out.assign((size_t)nwin * W, -1);
        for (int w = 0; w < nwin; ++w)
            for (size_t sl = 0; sl < (*bins)[w].size(); ++sl) win_out[(size_t)w * W + sl] = (*bins)[w][sl];
    }
    // output block of slot sl in window w, or -1
    auto slot_out = [&](int w, int sl) -> int {
        if (bins) return win_out[(size_t)w * W + sl];
        const int o = w * W + sl;
        return o < Fslots ? o : -1;
    };
    BidLookup bid{h};

    std::vector<uint32_t> stream, mask(nwin, 0);
    std::vector<int32_t> off(nwin), len(nwin), order(nwin);
    std::vector<int64_t> work(nwin, 0);
    int32_t ids[4];
    int longest = 0;
    struct Ent { int src; std::vector<uint32_t> recs; };
    for (int w = 0; w < nwin; ++w) {
        off[w] = (int32_t)stream.size();
        // entries of this window, each split so that no entry has more than r_max records
        std::vector<Ent> ents;
        for (int grp = 0; grp * gc < Fsrc; ++grp) {
            Ent e{grp, {}};
            // records by sub-block then slot, so every output sees its sources in increasing order
            for (int sub = 0; sub < gc; ++sub) {
                const int src = grp * gc + sub;
                if (src >= Fsrc) break;
                for (int sl = 0; sl < W; ++sl) {
                    const int o = slot_out(w, sl);
                    if (o < 0) continue;
                    const int cc = bwd ? o : src, kc = bwd ? src : o;   // coarse (c', k')
                    bool any = false;
                    for (int cs = 0; cs < f; ++cs)
                        for (int ks = 0; ks < f; ++ks) {
                            ids[cs * 2 + ks] = bid(cc * f + cs, kc * f + ks);
                            any |= ids[cs * 2 + ks] >= 0;
                        }
                    if (!any) continue;
                    e.recs.push_back(((uint32_t)(ids[0] + 1) << 7) | ((uint32_t)sub << 5) | (uint32_t)sl);
                    if (coarse)
                        for (int q = 1; q < 4; ++q) e.recs.push_back((uint32_t)(ids[q] + 1));
                    mask[w] |= 1u << sl;
                }
            }
            const int n = (int)e.recs.size() / rw;
            for (int r0 = 0; r0 < n; r0 += r_max) {
                const int r1 = std::min(n, r0 + r_max);
                ents.push_back(Ent{grp, std::vector<uint32_t>(e.recs.begin() + r0 * rw, e.recs.begin() + r1 * rw)});
            }
            work[w] += n ? n + 2 : 0;
        }
        // greedy packing into chunks
        size_t i = 0;
        while (i < ents.size()) {
            int ne = 0, nr = 0;
            size_t j = i;
            while (j < ents.size()) {
                const int er = (int)ents[j].recs.size() / rw;
                if (ne + 1 > e_max || nr + er > r_max || (ne + 1) * a_ops + (nr + er) * b_ops > 32) break;
                ++ne;
                nr += er;
                ++j;
            }
            if (ne == 0) return false;                           // limits admit no entry
            stream.push_back(((uint32_t)ne << 8) | (uint32_t)nr);
            for (size_t q = i; q < j; ++q)
                stream.push_back(((uint32_t)ents[q].src << 8) | (uint32_t)(ents[q].recs.size() / rw));
            for (size_t q = i; q < j; ++q) stream.insert(stream.end(), ents[q].recs.begin(), ents[q].recs.end());
            i = j;
        }
        stream.push_back(0);                                     // end marker
        while (stream.size() % 4) stream.push_back(0);
        len[w] = (int32_t)(stream.size() - off[w]);
        longest = std::max(longest, len[w]);
    }
    fs.too_big = longest > max_words;
    if (fs.too_big) return true;
    for (int w = 0; w < nwin; ++w) order[w] = w;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return work[a] > work[b]; });
    fs.W = W;
    fs.nwin = nwin;
    fs.Fslots = Fslots;
    fs.max_words = longest;
    std::vector<int4> desc(nwin);
    for (int j = 0; j < nwin; ++j) {
        const int w = order[j];
        desc[j] = make_int4(w, off[w], len[w], (int)mask[w]);
    }
    if (!upload(&fs.d_stream, stream) || !upload(&fs.d_win_desc, desc)) return false;
    if (bins && !upload(&fs.d_win_out, win_out)) return false;
    fs.built = true;
    return true;
}

// BSMM_UP_TEST_BAD_ID (tests only): the block id at table word `word` (the first record of
// the first CTA's first unit) becomes nnz + 5, which the weight-gradient epilogue must refuse
// (no store, BSMM_ERR_BOUNDS).  `packed` ids keep their sub-block position in bits 24..31.
void up_test_bad_id(const bsmm_ctx *h, std::vector<int32_t> &table, size_t word, bool packed)
{
    if (!getenv("BSMM_UP_TEST_BAD_ID") || table.size() <= word || table[0] == 0) return;
    const int32_t bad = h->nnz + 5;
    table[word] = packed ? (int32_t)(((uint32_t)table[word] & 0xFF000000u) | ((uint32_t)bad & 0xFFFFFFu)) : bad;
}

bool build_up(bsmm_ctx *h, UpSched &us)
{
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;
    const int Rc = (h->R + f - 1) / f, Sc = (h->S + f - 1) / f;
    const int MS = coarse ? 8 : 128 / h->bs;           // blocks stacked along M
    BidLookup bid{h};
    std::vector<std::vector<int32_t>> units;           // kUnitWords each
    int32_t ids[4];
    for (int kc = 0; kc < Sc; ++kc) {
        std::vector<int32_t> col;                      // 5 words per record of this coarse column
        for (int cc = 0; cc < Rc; ++cc) {
            bool any = false;
            for (int cs = 0; cs < f; ++cs)
                for (int ks = 0; ks < f; ++ks) {
                    ids[cs * 2 + ks] = bid(cc * f + cs, kc * f + ks);
                    any |= ids[cs * 2 + ks] >= 0;
                }
            if (!any) continue;
            col.push_back(cc);
            for (int q = 0; q < 4; ++q) col.push_back(ids[q]);
        }
        const int n = (int)col.size() / 5;
        for (int s0 = 0; s0 < n; s0 += MS) {
            std::vector<int32_t> u(kUnitWords, 0);
            const int m = std::min(MS, n - s0);
            u[0] = kc;
            u[1] = m;
            for (int q = 0; q < 5 * m; ++q) u[2 + q] = col[5 * s0 + q];
            units.push_back(u);
        }
    }
    const int nunits = (int)units.size();
    int ctas = std::max(1, std::min(nunits, 2 * std::max(1, h->sm_count)));
    ctas = std::max(ctas, (nunits + kUnitsPerCta - 1) / kUnitsPerCta);
    std::vector<int32_t> table((size_t)ctas * kTableWords, 0);
    for (int u = 0; u < nunits; ++u) {
        const int b = u % ctas, i = u / ctas;
        int32_t *t = table.data() + (size_t)b * kTableWords;
        t[0] = i + 1;
        std::copy(units[u].begin(), units[u].end(), t + 4 + i * kUnitWords);
    }
    us.ctas = nunits ? ctas : 0;
    up_test_bad_id(h, table, 4 + 2 + 1, false);
    if (!upload(&us.d_table, table)) return false;
    us.built = true;
    return true;
}

// Schedule of the dense-tile weight gradient (bs = 32): the 128 x 256 tiles of the dense
// gradient x^T.dy (4 block rows x 8 block columns) that contain at least one block, dealt
// round-robin to persistent CTAs.  Table word 0 = number of units; unit u at word
// 4 + u * kDUnitWords: c0 (first block row), k0 (first block column), count, then count
// words ((c_sub * 8 + k_sub) << 24) | block id.
constexpr int kDUnitWords = 36;
constexpr int kDUnitsPerCta = 48;
constexpr int kDTableWords = 4 + kDUnitsPerCta * kDUnitWords;

struct UpDenseSched {
    int ctas = 0;
    int32_t *d_table = nullptr;
    bool built = false;
};

bool build_up_dense(bsmm_ctx *h, UpDenseSched &us)
{
    const int Rt = (h->R + 3) / 4, St = (h->S + 7) / 8;
    std::vector<std::vector<int32_t>> units;
    for (int tc = 0; tc < Rt; ++tc)
        for (int tk = 0; tk < St; ++tk) {
            std::vector<int32_t> u(kDUnitWords, 0);
            int n = 0;
            for (int cs = 0; cs < 4; ++cs) {
                const int c = tc * 4 + cs;
                if (c >= h->R) break;
                const int32_t *b = h->h_row_ent.data() + h->h_row_ptr[c];
                const int32_t *e = h->h_row_ent.data() + h->h_row_ptr[c + 1];
                for (const int32_t *q = std::lower_bound(b, e, tk * 8); q != e && *q < tk * 8 + 8; ++q) {
                    const int32_t id = h->h_row_ptr[c] + (int32_t)(q - b);
                    u[3 + n++] = ((cs * 8 + (*q - tk * 8)) << 24) | id;
                }
            }
            if (!n) continue;
            u[0] = tc * 4;
            u[1] = tk * 8;
            u[2] = n;
            units.push_back(u);
        }
    const int nunits = (int)units.size();
    int ctas = std::max(1, std::min(nunits, std::max(1, h->sm_count)));
    ctas = std::max(ctas, (nunits + kDUnitsPerCta - 1) / kDUnitsPerCta);
    std::vector<int32_t> table((size_t)ctas * kDTableWords, 0);
    for (int u = 0; u < nunits; ++u) {
        const int b = u % ctas, i = u / ctas;
        int32_t *t = table.data() + (size_t)b * kDTableWords;
        t[0] = i + 1;
        std::copy(units[u].begin(), units[u].end(), t + 4 + i * kDUnitWords);
    }
    us.ctas = nunits ? ctas : 0;
    up_test_bad_id(h, table, 4 + 3, true);
    if (!upload(&us.d_table, table)) return false;
    us.built = true;
    return true;
}

// Schedule of the CTA-pair weight gradient (bs = 32): units are 256 x 256 tiles of x^T.dy
// (8 block rows x 8 block columns) with at least one block, dealt round-robin to the pairs.
// When the last round would leave most pairs idle (at most half of them busy), its tiles are
// split into two 256 x 128 units (nk = 4) so the tail is spread over twice as many pairs.
// Per pair: word 0 = number of units; unit u at 4 + u * kPUnitWords: c0, k0, nk, count, then
// count words ((c_sub * 8 + k_sub) << 24) | block id.
constexpr int kPUnitWords = 68;
constexpr int kPUnitsPerPair = 48;
constexpr int kPTableWords = 4 + kPUnitsPerPair * kPUnitWords;

struct UpPairSched {
    int ctas = 0;
    int32_t *d_table = nullptr;
    bool built = false, too_big = false;
};

bool build_up_pair(bsmm_ctx *h, UpPairSched &us)
{
    const int Rt = (h->R + 7) / 8, St = (h->S + 7) / 8;
    std::vector<std::vector<int32_t>> tiles;
    for (int tc = 0; tc < Rt; ++tc)
        for (int tk = 0; tk < St; ++tk) {
            std::vector<int32_t> u(kPUnitWords, 0);
            int n = 0;
            for (int cs = 0; cs < 8; ++cs) {
                const int c = tc * 8 + cs;
                if (c >= h->R) break;
                const int32_t *b = h->h_row_ent.data() + h->h_row_ptr[c];
                const int32_t *e = h->h_row_ent.data() + h->h_row_ptr[c + 1];
                for (const int32_t *q = std::lower_bound(b, e, tk * 8); q != e && *q < tk * 8 + 8; ++q) {
                    const int32_t id = h->h_row_ptr[c] + (int32_t)(q - b);
                    u[4 + n++] = ((cs * 8 + (*q - tk * 8)) << 24) | id;
                }
            }
            if (!n) continue;
            u[0] = tc * 8;
            u[1] = tk * 8;
            u[2] = 8;
            u[3] = n;
            tiles.push_back(u);
        }
    const int P = std::max(1, h->sm_count / 2);
    const int T = (int)tiles.size();
    const int full_rounds = T / P, rem = T - full_rounds * P;
    std::vector<std::vector<int32_t>> units(tiles.begin(), tiles.begin() + (size_t)full_rounds * P);
    for (int i = full_rounds * P; i < T; ++i) {
        const std::vector<int32_t> &t = tiles[i];
        if (full_rounds > 0 && 2 * rem <= P) {
            for (int half = 0; half < 2; ++half) {                 // block columns k0 + 4 half .. + 3
                std::vector<int32_t> u(kPUnitWords, 0);
                int n = 0;
                for (int e = 0; e < t[3]; ++e) {
                    const int ks = (t[4 + e] >> 24) & 7;
                    if ((ks >> 2) != half) continue;
                    const int cs = t[4 + e] >> 27;
                    u[4 + n++] = ((cs * 8 + (ks & 3)) << 24) | (t[4 + e] & 0xFFFFFF);
                }
                if (!n) continue;
                u[0] = t[0];
                u[1] = t[1] + 4 * half;
                u[2] = 4;
                u[3] = n;
                units.push_back(u);
            }
        } else {
            units.push_back(t);
        }
    }
    const int nunits = (int)units.size();
    const int pairs = std::max(1, std::min(nunits, P));
    if ((nunits + pairs - 1) / pairs > kPUnitsPerPair) {
        us.too_big = true;
        return true;
    }
    std::vector<int32_t> table((size_t)pairs * kPTableWords, 0);
    for (int u = 0; u < nunits; ++u) {
        const int b = u % pairs, i = u / pairs;
        int32_t *t = table.data() + (size_t)b * kPTableWords;
        t[0] = i + 1;
        std::copy(units[u].begin(), units[u].end(), t + 4 + i * kPUnitWords);
    }
    us.ctas = nunits ? 2 * pairs : 0;
    up_test_bad_id(h, table, 4 + 4, true);
    if (!upload(&us.d_table, table)) return false;
    us.built = true;
    return true;
}

// Schedule of the dense-tile fprop/bprop (bs = 32): for each group of 4 output blocks
// (fprop: block columns, bprop: block rows), the pairs of adjacent source blocks with at
// least one block among the group's outputs.  Per group a word stream:
//   entry: ((pair << 8) | mask), then 8 words id + 1 (0 = absent) in (sub, out) order,
//          mask bit sub*4 + out set when block (source 2*pair+sub, output out) is present
//   0xFFFFFFFF ends the stream; streams are padded to 4 words.
constexpr int kFbdSchedWords = 3072;

struct FbDenseSched {
    int ngroups = 0;
    uint32_t *d_stream = nullptr;
    int32_t *d_off = nullptr, *d_len = nullptr;
    bool built = false, too_big = false;
};

bool build_fb_dense(bsmm_ctx *h, FbDenseSched &fs, bool bwd)
{
    const int Fout = bwd ? h->R : h->S, Fsrc = bwd ? h->S : h->R;
    const int ng = (Fout + 3) / 4;
    BidLookup bid{h};
    std::vector<uint32_t> stream;
    std::vector<int32_t> off(ng), len(ng);
    for (int gi = 0; gi < ng; ++gi) {
        off[gi] = (int32_t)stream.size();
        for (int pr = 0; pr * 2 < Fsrc; ++pr) {
            uint32_t mask = 0, ids[8];
            for (int sub = 0; sub < 2; ++sub)
                for (int o = 0; o < 4; ++o) {
                    const int src = pr * 2 + sub, out = gi * 4 + o;
                    int32_t b = -1;
                    if (src < Fsrc && out < Fout) b = bwd ? bid(out, src) : bid(src, out);
                    ids[sub * 4 + o] = (uint32_t)(b + 1);
                    if (b >= 0) mask |= 1u << (sub * 4 + o);
                }
            if (!mask) continue;
            stream.push_back(((uint32_t)pr << 8) | mask);
            stream.insert(stream.end(), ids, ids + 8);
        }
        stream.push_back(0xFFFFFFFFu);
        while (stream.size() % 4) stream.push_back(0);
        len[gi] = (int32_t)(stream.size() - off[gi]);
        if (len[gi] > kFbdSchedWords) {
            fs.too_big = true;
            return true;
        }
    }
    fs.ngroups = ng;
    if (!upload(&fs.d_stream, stream) || !upload(&fs.d_off, off) || !upload(&fs.d_len, len)) return false;
    fs.built = true;
    return true;
}

// Schedule of the CTA-pair dense fprop/bprop (bs = 32): as build_fb_dense, for groups of 8
// output blocks.  Entry: ((pair << 16) | mask), mask bit sub * 8 + out, then 16 words id + 1
// in (sub, out) order; outputs 0-3 belong to the pair's even CTA, 4-7 to the odd one.
constexpr int kFbpSchedWords = 3072;

bool build_fb_dense_pair(bsmm_ctx *h, FbDenseSched &fs, bool bwd)
{
    const int Fout = bwd ? h->R : h->S, Fsrc = bwd ? h->S : h->R;
    const int ng = (Fout + 7) / 8;
    BidLookup bid{h};
    std::vector<uint32_t> stream;
    std::vector<int32_t> off(ng), len(ng);
    for (int gi = 0; gi < ng; ++gi) {
        off[gi] = (int32_t)stream.size();
        for (int pr = 0; pr * 2 < Fsrc; ++pr) {
            uint32_t mask = 0, ids[16];
            for (int sub = 0; sub < 2; ++sub)
                for (int o = 0; o < 8; ++o) {
                    const int src = pr * 2 + sub, out = gi * 8 + o;
                    int32_t b = -1;
                    if (src < Fsrc && out < Fout) b = bwd ? bid(out, src) : bid(src, out);
                    ids[sub * 8 + o] = (uint32_t)(b + 1);
                    if (b >= 0) mask |= 1u << (sub * 8 + o);
                }
            if (!mask) continue;
            stream.push_back(((uint32_t)pr << 16) | mask);
            stream.insert(stream.end(), ids, ids + 16);
        }
        stream.push_back(0xFFFFFFFFu);
        while (stream.size() % 4) stream.push_back(0);
        len[gi] = (int32_t)(stream.size() - off[gi]);
        if (len[gi] > kFbpSchedWords) {
            fs.too_big = true;
            return true;
        }
    }
    fs.ngroups = ng;
    if (!upload(&fs.d_stream, stream) || !upload(&fs.d_off, off) || !upload(&fs.d_len, len)) return false;
    fs.built = true;
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

constexpr int kProducers = 4;                    // fprop/bprop: producer+epilogue warps, then the MMA warp
constexpr int kFbThreads = 32 * (kProducers + 1);
constexpr int kUpThreads = 32 * (kProducers + 5);        // updat: producers, MMA warp, 4 epilogue warps
static_assert(16 % kProducers == 0, "stage counts must be multiples of the producer count");
constexpr int kFbpThreads = 32 * (kProducers + 5);      // CTA-pair fprop/bprop: + 4 epilogue warps
constexpr int kZeroTiles = 2048;                 // 8x8 zero tiles in the zero buffer (256 KB)
constexpr int kZeroBytes = kZeroTiles * 128;

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

// Compile-time descriptor geometry of the fprop/bprop kernel for a (coarse) block edge BSE.
template <int BSE, int FA> struct FbGeo {
    static constexpr int B_SLOT = BSE * BSE * 2;                     // one (coarse) weight block
    static constexpr int KSTEPS = BSE / 16;
    // A operand descriptor parameters.  (N,C) activations: K-major rows of ROW bytes holding
    // ROW / (2 BSE) adjacent source blocks (one 32-feature block for BSE = 32, so no panel carries
    // a neighbour the window may not need; four 16-feature blocks otherwise); block `sub` starts
    // sub*BSE*2 bytes into the row.  (C,N) activations: MN-major, two 64-row atoms of one block.
    static constexpr int ROW = fb_row_bytes(BSE);
    static constexpr uint32_t A_SWZ = FA ? (ROW == 64 ? SW_64 : SW_128) : SW_128;
    static constexpr uint32_t A_LBO = FA ? 16 : (BSE * 128);         // MN-major: distance of the two 64-row atoms
    static constexpr uint32_t A_SBO = FA ? 8 * ROW : 1024;
    static constexpr uint32_t A_KSTEP = FA ? 32 : (16 * 128);
    static constexpr uint32_t A_SUB = BSE * 2;                       // byte offset of block `sub` in a row
};

constexpr int kMaxStages = 16;                   // a multiple of kProducers
constexpr int kMaxSmem = 216 * 1024;         // largest dynamic request (static shared memory counts against 227 KB)
constexpr int kSchedWords = 3072;                                    // window stream budget (12 KB)

// Runtime stage geometry: a stage holds one chunk of up to e_slots activation panels
// (a_slot bytes each) and r_slots weight blocks.  With half = 1 (minibatch <= 64) a panel
// is 64 rows: the MMA still reads 128 rows, the upper 64 come from the next slot (or the
// padding after the last stage) and only feed accumulator rows that are never stored.
struct FbStages {
    int e_slots, r_slots, stages;
    int half;           // 1: 64-row minibatch tiles (activation panels of 64 rows), else 128
    int a_slot, stage_bytes, b_off;
    int producers;      // producer warps (1, 2 or 4), a divisor of stages
};

struct FbParams {
    void *out;
    const uint32_t *stream;
    const int4 *win_desc;       // per launch position: window, stream offset, length, slot mask
    const int32_t *win_out;     // binned windows: output block of each slot (-1 = unused); else null
    int32_t *status;
    int N;          // minibatch
    int Fout;       // output features (C for bprop, K for fprop)
    int W;          // slots per window
    int Fslots;     // output (coarse) blocks
    int n_tiles;
    FbStages g;
};

// fprop (BWD=false) / bprop (BWD=true).  BS = fine block size, BSE = 16 when BS = 8.
template <int BS, int FA, bool BWD, bool BF16>
__global__ void __launch_bounds__(kFbThreads, 1)
k_tc_fb(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
        const __grid_constant__ CUtensorMap tm_zero, const FbParams p)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    using G = FbGeo<BSE, FA>;
    constexpr bool COARSE = BS == 8;
    constexpr int RW = COARSE ? 4 : 1;                                // words per record
    constexpr int B_OPS = COARSE ? 4 : 1;                             // TMA boxes per record
    // B operand: fprop reads w[b] as B[K=i][N=j] (MN-major), bprop as B[K=j][N=i] (K-major).
    constexpr uint32_t B_SWZ = COARSE ? SW_NONE : (BS == 32 ? SW_64 : SW_32);
    constexpr uint32_t B_LBO = COARSE ? 128 : 16;
    constexpr uint32_t B_SBO = COARSE ? 256 : 8 * BS * 2;
    constexpr uint32_t B_KSTEP = BWD ? 32 : 16 * BS * 2;
    constexpr uint32_t IDESC = idesc_f16(128, BSE, BF16, FA == 0, !BWD);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const FbStages g = p.g;
    const int a_ops = (FA || g.half) ? 1 : 2;                         // TMA boxes per activation panel
    if (g.producers < 1 || g.producers > kProducers || g.stages % g.producers != 0 || g.stages > kMaxStages) {
        // the host guarantees this; refuse otherwise
        if (threadIdx.x == 0) atomicExch(p.status, (int32_t)BSMM_ERR_INVALID);
        return;
    }
    const uint32_t *sched = reinterpret_cast<const uint32_t *>(smem + g.stages * g.stage_bytes + g.a_slot);
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], acc_full, sched_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.x;
    const int4 desc = __ldg(p.win_desc + unit / p.n_tiles);
    const int win = desc.x;
    const int tile_rows = g.half ? 64 : 128;
    const int n0 = (unit % p.n_tiles) * tile_rows;
    const int ncols = p.W * BSE;
    const uint32_t alloc_cols = ncols <= 32 ? 32 : ncols <= 64 ? 64 : ncols <= 128 ? 128 : 256;

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < g.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&sched_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc(&tmem_base, alloc_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    // The window schedule belongs to the handle: fetch it before waiting for the previous kernel.
    if (warp == 0 && lane == 0) {
        const int len = desc.z;
        mbar_arrive_expect_tx(&sched_full, (uint32_t)len * 4u);
        if (len > 0) bulk_load((void *)sched, p.stream + desc.y, (uint32_t)len * 4u, &sched_full, policy_evict_last());
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_w);
    }
    pdl_wait();

    if (warp < kProducers) {
        // ---------------- TMA producers: warp w < P issues chunks w, w+P, ...; one load per lane ----
        const uint64_t pol_act = policy_evict_last();
        const uint64_t pol_w = policy_evict_first();
        if (!mbar_wait_warp(&sched_full, 0, p.status, 64)) aborted = 1;
        __syncwarp();
        int chunk = 0, last = -1;
        for (int pos = 0; !aborted; ++chunk) {
            const uint32_t hdr = sched[pos];
            const int ne = (int)(hdr >> 8), nr = (int)(hdr & 0xFFu);
            if (ne == 0) break;
            if (chunk % g.producers != warp) {
                pos += 1 + ne + nr * RW;
                continue;
            }
            const int st = chunk % g.stages;
            if (lane == 0) {
                if (chunk >= g.stages && !mbar_wait(&empty[st], ((chunk / g.stages) - 1) & 1, p.status))
                    aborted = 1;
                else
                    mbar_arrive_expect_tx(&full[st], (uint32_t)(ne * g.a_slot + nr * G::B_SLOT));
            }
            __syncwarp();
            if (aborted) break;
            last = chunk;
            uint8_t *stage = smem + st * g.stage_bytes;
            const int na = ne * a_ops;
            // One TMA instruction for the whole chunk (each issue costs a fixed few hundred ns
            // whatever the number of lanes): lanes < na load activation panels, the next
            // nr * B_OPS lanes weight blocks (or, for bs=8, 8x8 sub-blocks and zero tiles).
            if (lane < na + nr * B_OPS) {
                const bool isa = lane < na;
                const CUtensorMap *mp;
                uint8_t *dst;
                int cx, cy;
                uint64_t pol;
                if (isa) {
                    const int e = lane / a_ops, hf = lane % a_ops;
                    const int src = (int)(sched[pos + 1 + e] >> 8);
                    mp = &tm_act;
                    dst = stage + e * g.a_slot + (FA ? 0 : hf * BSE * 128);
                    cx = FA ? src * (G::ROW / 2) : n0 + 64 * hf;
                    cy = FA ? n0 : src * BSE;
                    pol = pol_act;
                } else {
                    const int q = lane - na, r = q / B_OPS, sub = q % B_OPS;
                    const uint32_t *rec = sched + pos + 1 + ne + r * RW;
                    dst = stage + g.b_off + r * G::B_SLOT;
                    pol = pol_w;
                    cx = 0;
                    if (!COARSE) {
                        mp = &tm_w;
                        cy = ((int)(rec[0] >> 7) - 1) * BS;
                    } else {
                        // sub-block (cs, ks) -> core matrix at (N-group)*256 + (K-group)*128;
                        // zero tiles are spread over the zero buffer so they hit many L2 lines
                        const int cs = sub >> 1, ks = sub & 1;
                        const int ng = BWD ? cs : ks, kg = BWD ? ks : cs;
                        const int id = (int)(sub == 0 ? (rec[0] >> 7) : rec[sub]) - 1;
                        const int zr = (int)((blockIdx.x * 61u + (unsigned)chunk * 32u + (unsigned)lane) % kZeroTiles) * 8;
                        mp = id >= 0 ? &tm_w : &tm_zero;
                        dst += ng * 256 + kg * 128;
                        cy = id >= 0 ? id * 8 : zr;
                    }
                }
                tma_load_2d(dst, mp, &full[st], cx, cy, pol);
            }
            pos += 1 + ne + nr * RW;
        }
        // After an abort, wait (bounded) for this warp's last loads before the CTA may exit.
        // Normally the MMA warp has waited on every stage, so nothing is left in flight.
        if (aborted && lane == 0 && last >= 0)
            mbar_wait(&full[last % g.stages], (last / g.stages) & 1, nullptr);
        __syncwarp();
    } else {
        // ---------------- MMA issuer ----------------
        if (elect_one()) {
            uint32_t inited = 0;
            const uint32_t s_base = smem_u32(smem);
            // Descriptors of the smem base; an operand at byte offset o is base + (o >> 4)
            // (the start address is the low 14-bit field, in 16-byte units).
            const uint64_t a_desc0 = sdesc(s_base, G::A_LBO, G::A_SBO, G::A_SWZ);
            const uint64_t b_desc0 = sdesc(s_base, B_LBO, B_SBO, B_SWZ);
            if (!mbar_wait(&sched_full, 0, p.status)) aborted = 1;
            int chunk = 0;
            for (int pos = 0; !aborted; ++chunk) {
                const uint32_t hdr = sched[pos];
                const int ne = (int)(hdr >> 8), nr = (int)(hdr & 0xFFu);
                if (ne == 0) break;
                const int st = chunk % g.stages;
                if (!mbar_wait(&full[st], (chunk / g.stages) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t stage_off = st * g.stage_bytes;
                const uint32_t *rec = sched + pos + 1 + ne;
                int r = 0;
                for (int e = 0; e < ne; ++e) {
                    const int nrec = (int)(sched[pos + 1 + e] & 0xFFu);
                    const uint32_t a_off = stage_off + e * g.a_slot;
                    for (int j = 0; j < nrec; ++j, ++r) {
                        const uint32_t rw0 = rec[r * RW];
                        const uint32_t slot = rw0 & 31u;
                        const uint64_t ad = a_desc0 + ((a_off + ((rw0 >> 5) & 3u) * G::A_SUB) >> 4);
                        const uint64_t bd = b_desc0 + ((stage_off + g.b_off + r * G::B_SLOT) >> 4);
                        const uint32_t d = tmem + slot * BSE;
                        const uint32_t acc = (inited >> slot) & 1u;
#pragma unroll
                        for (int ks = 0; ks < G::KSTEPS; ++ks)
                            mma_ss(d, ad + ((ks * G::A_KSTEP) >> 4), bd + ((ks * B_KSTEP) >> 4), IDESC,
                                   ks > 0 ? 1u : acc);
                        inited |= 1u << slot;
                    }
                }
                mma_commit(&empty[st]);
                pos += 1 + ne + nr * RW;
            }
            mma_commit(&acc_full);
        }
        __syncwarp();
    }
    if (warp < kProducers) {
        // ---------------- epilogue (producer warps 0..3, one TMEM lane quarter each) ----
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        // rows past a 64-row tile hold products of the neighbouring shared memory: never stored
        const int n = row < tile_rows ? n0 + row : p.N;
        const bool ok = mbar_wait_warp(&acc_full, 0, p.status, 256);
        tc_fence_after();
        const uint32_t mask = (uint32_t)desc.w;
        uint16_t *out = static_cast<uint16_t *>(p.out);
        for (int s = 0; s < p.W; ++s) {
            const int o = p.win_out ? __ldg(p.win_out + win * p.W + s) : win * p.W + s;
            if (o < 0 || o >= p.Fslots) continue;
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
#pragma unroll
                        for (int j = 0; j < BSE; ++j)
                            if (f0 + j < p.Fout) dst[j] = cvt1<BF16>(v[j]);
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
    if (warp == kProducers) tmem_dealloc(tmem, alloc_cols);
}

// ---------------------------------------------------------------------------------------
// updat
// ---------------------------------------------------------------------------------------

struct UpMaps {
    CUtensorMap x[8];
    CUtensorMap dy[8];
    CUtensorMap dw;             // [nnz * bs rows][bs] in dW's type, one block per box (TMA epilogue)
};

struct UpParams {
    void *dw;                   // dw_dtype: float32, or the inputs' 16-bit type
    const int32_t *table;
    int32_t *status;
    int N, G, accumulate;
    int dwt;                    // 0: float32 dW, 1: fp16, 2: bf16
    int nnz;                    // blocks in dW: every table id is checked against it before a store
    int tma;                    // 1: the epilogue writes dW blocks by TMA store (reduce-add to accumulate)
};

// True when block `id` lies inside dW; otherwise records BSMM_ERR_BOUNDS (sticky) and the
// caller skips the store, so a corrupted table never writes past dW.
__device__ __forceinline__ bool up_id_ok(int32_t id, const UpParams &p)
{
    if ((uint32_t)id < (uint32_t)p.nnz) return true;
    atomicExch(p.status, (int32_t)BSMM_ERR_BOUNDS);
    return false;
}


// Stores 4 consecutive dW values at element `off` in the output type; with accumulate, adds the
// stored values in float32 first and rounds the sum once.
__device__ __forceinline__ void up_store4(void *dw, size_t off, float4 v, int accumulate, int dwt)
{
    if (dwt == 0) {
        float *d = static_cast<float *>(dw) + off;
        if (accumulate) {
            const float4 a = *reinterpret_cast<const float4 *>(d);
            v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
        }
        *reinterpret_cast<float4 *>(d) = v;
        return;
    }
    uint16_t *d = static_cast<uint16_t *>(dw) + off;
    if (accumulate) {
        const uint2 a = *reinterpret_cast<const uint2 *>(d);
        float f[4];
        const uint16_t hs[4] = {(uint16_t)(a.x & 0xFFFFu), (uint16_t)(a.x >> 16), (uint16_t)(a.y & 0xFFFFu),
                                (uint16_t)(a.y >> 16)};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = dwt == 2 ? __uint_as_float((uint32_t)hs[i] << 16) : __half2float(__ushort_as_half(hs[i]));
        v.x += f[0]; v.y += f[1]; v.z += f[2]; v.w += f[3];
    }
    uint2 o;
    o.x = dwt == 2 ? pack2<true>(v.x, v.y) : pack2<false>(v.x, v.y);
    o.y = dwt == 2 ? pack2<true>(v.z, v.w) : pack2<false>(v.z, v.w);
    *reinterpret_cast<uint2 *>(d) = o;
}

// Writes one 32 x 32 dW block whose row `lane` this lane holds in v, through the warp's 4 KB
// staging tile stg (1024-byte aligned).  With p.tma the rows go into stg in the layout of the dW
// tensor map (16-byte piece c of row r at c ^ (r mod 8) for 128-byte float32 rows, at
// c ^ ((r / 2) mod 4) for 64-byte 16-bit rows) and lane 0 issues one TMA store, or a TMA
// reduce-add when accumulating (float32 sum in L2, one rounding); the tile is rewritten only after
// the previous store has read it.  Otherwise the tile is read back so that each store
// instruction writes 512 contiguous bytes.  Nothing is written when skip is set or id is out of range.
__device__ __forceinline__ void up_block32_out(const CUtensorMap *dwm, const UpParams &p, float *stg, int lane,
                                               int32_t id, const float (&v)[32], bool skip)
{
    if (p.tma) {
        uint8_t *sb = reinterpret_cast<uint8_t *>(stg);
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        if (p.dwt == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4 *>(sb + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                    make_float4(v[c * 4], v[c * 4 + 1], v[c * 4 + 2], v[c * 4 + 3]);
        } else {
            const bool b16 = p.dwt == 2;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 pk;
                pk.x = b16 ? pack2<true>(v[c * 8], v[c * 8 + 1]) : pack2<false>(v[c * 8], v[c * 8 + 1]);
                pk.y = b16 ? pack2<true>(v[c * 8 + 2], v[c * 8 + 3]) : pack2<false>(v[c * 8 + 2], v[c * 8 + 3]);
                pk.z = b16 ? pack2<true>(v[c * 8 + 4], v[c * 8 + 5]) : pack2<false>(v[c * 8 + 4], v[c * 8 + 5]);
                pk.w = b16 ? pack2<true>(v[c * 8 + 6], v[c * 8 + 7]) : pack2<false>(v[c * 8 + 6], v[c * 8 + 7]);
                *reinterpret_cast<uint4 *>(sb + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = pk;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && !skip && up_id_ok(id, p)) {
            if (p.accumulate) tma_reduce_add_2d(dwm, sb, 0, id * 32);
            else tma_store_2d(dwm, sb, 0, id * 32);
            bulk_commit();
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(stg + lane * 32 + ((c ^ (lane & 7)) * 4)) =
            make_float4(v[c * 4], v[c * 4 + 1], v[c * 4 + 2], v[c * 4 + 3]);
    __syncwarp();
    if (!skip && up_id_ok(id, p)) {
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
            const int o = k4 * 128 + lane * 4, r = o / 32, c = (o % 32) / 4;
            up_store4(p.dw, (size_t)id * 1024 + o, *reinterpret_cast<const float4 *>(stg + r * 32 + ((c ^ (r & 7)) * 4)),
                      p.accumulate, p.dwt);
        }
    }
    __syncwarp();                                   // reads done before the next block's writes
}

template <int BSE, int FA> struct UpGeo {
    static constexpr int TK = 64;                                   // minibatch rows per stage
    static constexpr int A_BYTES = 128 * TK * 2;                    // up to 128/BSE stacked panels (16 KB)
    static constexpr int B_BYTES = TK * BSE * 2;
    static constexpr int PANEL = TK * BSE * 2;                      // one stacked panel
    static constexpr int STAGES = 4;                                 // a multiple of kProducers
    static constexpr int TAB_OFF = STAGES * (A_BYTES + B_BYTES);
    static constexpr int OUT_OFF = (TAB_OFF + kTableWords * 4 + 1023) / 1024 * 1024;   // swizzled staging
    static constexpr int OUT_BYTES = 4 * 32 * 32 * 4;              // per epilogue warp: 32 rows of up to 32 fp32
    static constexpr int SMEM = OUT_OFF + OUT_BYTES;
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

// Persistent weight-gradient kernel: each CTA walks its unit table; TMA loads stream
// through the stage ring across unit boundaries; two TMEM accumulators let the epilogue of
// one unit overlap the MMAs of the next.
// Two CTAs share an SM: their 18 warps leave five on some SM sub-partitions, whose 16384 registers
// then allow at most 102 per thread, so the kernel is held to 96.
template <int BS, int FA, bool BF16>
__global__ void __maxnreg__(96)
k_tc_updat(const __grid_constant__ UpMaps maps, const UpParams p)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    constexpr bool COARSE = BS == 8;
    using G = UpGeo<BSE, FA>;
    static_assert(G::STAGES % kProducers == 0, "producer warp w must own stages w, w+4, ...");
    constexpr uint32_t IDESC = idesc_f16(128, BSE, BF16, FA == 1, FA == 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + G::STAGES * G::A_BYTES;
    int32_t *tab = reinterpret_cast<int32_t *>(smem + G::TAB_OFF);
    float *sout = reinterpret_cast<float *>(smem + G::OUT_OFF);
    __shared__ __align__(8) uint64_t full[G::STAGES], empty[G::STAGES], acc_full[2], acc_empty[2], tab_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int chunks = (p.N + G::TK - 1) / G::TK;
    const int total = chunks * p.G;                 // stages per unit

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < G::STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);            // one arrival per epilogue warp
        }
        mbar_init(&tab_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc(&tmem_base, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    const int32_t *gtab = p.table + (size_t)blockIdx.x * kTableWords;
    if (warp == 0 && lane == 0) {
        const int nu = gtab[0];
        const uint32_t bytes = (uint32_t)(4 + nu * kUnitWords) * 4u;
        mbar_arrive_expect_tx(&tab_full, bytes);
        bulk_load(tab, gtab, bytes, &tab_full, policy_evict_first());
    }
    pdl_wait();
    const bool tab_ok = mbar_wait_warp(&tab_full, 0, p.status, 64);
    const int nunits = tab_ok ? tab[0] : 0;

    if (warp < kProducers) {
        // TMA producers: warp w issues stage iterations w, w+4, ...; in each, lane r < nrec
        // loads stacked panel r and lane nrec the dy panel.
        const uint64_t pol = policy_evict_last();
        int it = 0, last = -1;
        for (int u = 0; u < nunits && !aborted; ++u) {
            const int32_t *ut = tab + 4 + u * kUnitWords;
            const int kc = ut[0], nrec = ut[1];
            const int cc = lane < nrec ? ut[2 + 5 * lane] : 0;
            const uint32_t bytes = nrec * G::PANEL + G::B_BYTES;
            for (int c = 0; c < total; ++c, ++it) {
                if (it % kProducers != warp) continue;
                const int t = c / chunks, n0 = (c % chunks) * G::TK;
                const int s = it % G::STAGES;
                if (lane == 0) {
                    if (it >= G::STAGES && !mbar_wait(&empty[s], ((it / G::STAGES) - 1) & 1, p.status)) aborted = 1;
                    else mbar_arrive_expect_tx(&full[s], bytes);
                }
                __syncwarp();
                if (aborted) break;
                last = it;
                // one TMA instruction: lanes < nrec the stacked x panels, lane nrec the dy panel
                if (lane <= nrec) {
                    const bool isx = lane < nrec;
                    const CUtensorMap *mp = isx ? &maps.x[t] : &maps.dy[t];
                    uint8_t *dst = isx ? sA + s * G::A_BYTES + lane * G::PANEL : sB + s * G::B_BYTES;
                    const int f = (isx ? cc : kc) * BSE;
                    tma_load_2d(dst, mp, &full[s], FA ? f : n0, FA ? n0 : f, pol);
                }
            }
        }
        // After an abort, wait (bounded) for this warp's last loads before the CTA may exit.
        if (aborted && lane == 0 && last >= 0)
            mbar_wait(&full[last % G::STAGES], (last / G::STAGES) & 1, nullptr);
        __syncwarp();
    } else if (warp == kProducers) {
        if (elect_one()) {
            const uint64_t a_desc0 = sdesc(smem_u32(sA), G::A_LBO, G::A_SBO, G::A_SWZ);
            const uint64_t b_desc0 = sdesc(smem_u32(sB), G::B_LBO, G::B_SBO, G::B_SWZ);
            int it = 0;
            for (int u = 0; u < nunits && !aborted; ++u) {
                const int buf = u & 1;
                if (u >= 2 && !mbar_wait(&acc_empty[buf], ((u >> 1) - 1) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * 32;
                for (int c = 0; c < total; ++c, ++it) {
                    const int s = it % G::STAGES;
                    if (!mbar_wait(&full[s], (it / G::STAGES) & 1, p.status)) {
                        aborted = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((s * G::A_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + ((s * G::B_BYTES) >> 4);
#pragma unroll
                    for (int ks = 0; ks < G::TK / 16; ++ks)
                        mma_ss(d, ad + ((ks * G::A_KSTEP) >> 4), bd + ((ks * G::B_KSTEP) >> 4), IDESC,
                               (c > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                mma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int slot = row / BSE, i = row % BSE;
        for (int u = 0; u < nunits; ++u) {
            const int buf = u & 1;
            const bool ok = mbar_wait_warp(&acc_full[buf], (u >> 1) & 1, p.status, 128);
            if (!ok) break;
            tc_fence_after();
            float v[BSE];
#pragma unroll
            for (int c0 = 0; c0 < BSE; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + buf * 32 + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            const int32_t *ut = tab + 4 + u * kUnitWords;
            if (!COARSE && p.tma) {
                // The warp's 32 rows are 32 / BSE whole blocks.  Each lane writes its row into the
                // warp's staging buffer in the layout of the dW tensor map (rows of ROWB bytes,
                // 16-byte piece c of a row at c ^ (row address bits 7..), as TMA reads it), and
                // lane 0 issues one TMA store per present block -- a reduce-add (float32 sum in
                // L2, one rounding) when accumulating.  The buffer is rewritten only after the
                // previous unit's stores have read it.
                uint8_t *stg = reinterpret_cast<uint8_t *>(sout + q * 32 * 32);
                const int eb = p.dwt == 0 ? 4 : 2, rowb = BS * eb;
                const uint32_t ro = (uint32_t)(lane * rowb);
                const uint32_t swm = rowb == 128 ? 7u : rowb == 64 ? 3u : 1u;
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                if (p.dwt == 0) {
#pragma unroll
                    for (int c = 0; c < BS / 4; ++c)
                        *reinterpret_cast<float4 *>(stg + ro + ((c ^ ((ro >> 7) & swm)) << 4)) =
                            make_float4(v[c * 4], v[c * 4 + 1], v[c * 4 + 2], v[c * 4 + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < BS / 8; ++c) {
                        uint4 pk;
                        const bool b16 = p.dwt == 2;
                        pk.x = b16 ? pack2<true>(v[c * 8], v[c * 8 + 1]) : pack2<false>(v[c * 8], v[c * 8 + 1]);
                        pk.y = b16 ? pack2<true>(v[c * 8 + 2], v[c * 8 + 3]) : pack2<false>(v[c * 8 + 2], v[c * 8 + 3]);
                        pk.z = b16 ? pack2<true>(v[c * 8 + 4], v[c * 8 + 5]) : pack2<false>(v[c * 8 + 4], v[c * 8 + 5]);
                        pk.w = b16 ? pack2<true>(v[c * 8 + 6], v[c * 8 + 7]) : pack2<false>(v[c * 8 + 6], v[c * 8 + 7]);
                        *reinterpret_cast<uint4 *>(stg + ro + ((c ^ ((ro >> 7) & swm)) << 4)) = pk;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && !aborted) {
#pragma unroll
                    for (int b = 0; b < 32 / BSE; ++b) {
                        const int sl = q * (32 / BSE) + b;
                        if (sl >= ut[1]) continue;
                        const int32_t id = ut[2 + 5 * sl + 1];
                        if (!up_id_ok(id, p)) continue;
                        const uint8_t *src = stg + b * BS * rowb;
                        if (p.accumulate) tma_reduce_add_2d(&maps.dw, src, 0, id * BS);
                        else tma_store_2d(&maps.dw, src, 0, id * BS);
                    }
                    bulk_commit();
                }
            } else if (!COARSE) {
                // The warp's 32 rows are 32 / BSE whole blocks, [row][BS] fp32 like the blocks in
                // dw.  Pass them through shared memory so that each store instruction writes 512
                // contiguous bytes of one block; 16-byte chunk c of row r sits at chunk
                // c ^ (r mod BS/4), which keeps both the row writes and the reads conflict-free.
                constexpr int CH = BS / 4;                      // 16-byte chunks per row
                float *stg = sout + q * 32 * 32;
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    *reinterpret_cast<float4 *>(stg + lane * BS + ((c ^ (lane & (CH - 1))) * 4)) =
                        make_float4(v[c * 4], v[c * 4 + 1], v[c * 4 + 2], v[c * 4 + 3]);
                __syncwarp();
                constexpr int BLK = BSE * BS;                   // floats per block
#pragma unroll
                for (int k4 = 0; k4 < BS / 4; ++k4) {
                    const int o = k4 * 128 + lane * 4;          // float offset in the warp's rows
                    const int sl = q * (32 / BSE) + o / BLK;
                    const int r = o / BS, c = (o % BS) / 4;
                    const float4 val = *reinterpret_cast<const float4 *>(stg + r * BS + ((c ^ (r & (CH - 1))) * 4));
                    if (sl < ut[1] && !aborted && up_id_ok(ut[2 + 5 * sl + 1], p))
                        up_store4(p.dw, (size_t)ut[2 + 5 * sl + 1] * (BS * BS) + (o % BLK), val, p.accumulate, p.dwt);
                }
                __syncwarp();                                   // reads done before the next unit's writes
            } else if (slot < ut[1] && !aborted) {
                const int32_t *rec = ut + 2 + 5 * slot;
                {
                    const int cs = i / 8, i8 = i % 8;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const int32_t id = rec[1 + cs * 2 + ks];
                        if (id < 0 || !up_id_ok(id, p)) continue;
#pragma unroll
                        for (int j = 0; j < 8; j += 4)
                            up_store4(p.dw, ((size_t)id * 8 + i8) * 8 + j,
                                      make_float4(v[ks * 8 + j], v[ks * 8 + j + 1], v[ks * 8 + j + 2], v[ks * 8 + j + 3]),
                                      p.accumulate, p.dwt);
                    }
                }
            }
        }
        if (p.tma && lane == 0) bulk_wait_all();        // every dW store has completed before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProducers) tmem_dealloc(tmem, 64);
}

// Dense-tile weight gradient, bs = 32.  A unit is a 128 x 256 tile of x^T.dy: block rows
// c0..c0+3 (M = 128) by block columns k0..k0+7 (N = 256), reduced over the minibatch in
// stages of 64 rows (4 MMAs of 128 x 256 x 16).  All loads are 128-byte rows: with (N,C)
// activations two 64-column boxes of x (MN-major A, two 64-row M atoms) and four of dy
// (MN-major B, four 64-column N atoms); with (C,N) one 128-row box of x (K-major A) and one
// 256-row box of dy (K-major B).  The epilogue warp for TMEM lane quarter q owns block row
// c0+q and writes every present block of that row.
struct UpDenseGeo {
    static constexpr int TK = 64;
    static constexpr int A_BYTES = 128 * TK * 2;                     // 16 KB
    static constexpr int B_BYTES = 256 * TK * 2;                     // 32 KB
    static constexpr int STAGES = 4;                                 // a multiple of kProducers
    static constexpr int TAB_OFF = STAGES * (A_BYTES + B_BYTES);
    static constexpr int OUT_OFF = (TAB_OFF + kDTableWords * 4 + 1023) / 1024 * 1024;  // swizzled staging
    static constexpr int SMEM = OUT_OFF + 4 * 32 * 32 * 4;           // + a 32 x 32 fp32 block per epilogue warp
};

template <int FA, bool BF16>
__global__ void __launch_bounds__(kUpThreads, 1)
k_tc_updat_dense(const __grid_constant__ UpMaps maps, const UpParams p)
{
    using G = UpDenseGeo;
    static_assert(G::STAGES % kProducers == 0, "producer warp w must own stages w, w+4, ...");
    // fa=1: A = x^T MN-major (M atoms of 64 at 8 KB), B = dy MN-major (N atoms of 64 at 8 KB);
    // fa=0: both K-major, 128-byte rows.
    constexpr uint32_t A_LBO = FA ? 8192 : 16, B_LBO = FA ? 8192 : 16;
    constexpr uint32_t KSTEP = FA ? 16 * 128 : 32;
    constexpr uint32_t IDESC = idesc_f16(128, 256, BF16, FA == 1, FA == 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + G::STAGES * G::A_BYTES;
    int32_t *tab = reinterpret_cast<int32_t *>(smem + G::TAB_OFF);
    float *sout = reinterpret_cast<float *>(smem + G::OUT_OFF);
    __shared__ __align__(8) uint64_t full[G::STAGES], empty[G::STAGES], acc_full[2], acc_empty[2], tab_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int chunks = (p.N + G::TK - 1) / G::TK;
    const int total = chunks * p.G;

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < G::STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(&tab_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    const int32_t *gtab = p.table + (size_t)blockIdx.x * kDTableWords;
    if (warp == 0 && lane == 0) {
        const int nu = gtab[0];
        const uint32_t bytes = (uint32_t)(4 + nu * kDUnitWords) * 4u;
        mbar_arrive_expect_tx(&tab_full, bytes);
        bulk_load(tab, gtab, bytes, &tab_full, policy_evict_first());
    }
    pdl_wait();
    const bool tab_ok = mbar_wait_warp(&tab_full, 0, p.status, 64);
    const int nunits = tab_ok ? tab[0] : 0;

    if (warp < kProducers) {
        const uint64_t pol = policy_evict_last();
        const uint32_t bytes = G::A_BYTES + G::B_BYTES;
        int it = 0, last = -1;
        for (int u = 0; u < nunits && !aborted; ++u) {
            const int32_t *ut = tab + 4 + u * kDUnitWords;
            const int f_c = ut[0] * 32, f_k = ut[1] * 32;        // first feature of the tile
            for (int c = 0; c < total; ++c, ++it) {
                if (it % kProducers != warp) continue;
                const int t = c / chunks, n0 = (c % chunks) * G::TK;
                const int s = it % G::STAGES;
                if (lane == 0) {
                    if (it >= G::STAGES && !mbar_wait(&empty[s], ((it / G::STAGES) - 1) & 1, p.status)) aborted = 1;
                    else mbar_arrive_expect_tx(&full[s], bytes);
                }
                __syncwarp();
                if (aborted) break;
                last = it;
                uint8_t *a = sA + s * G::A_BYTES;
                uint8_t *b = sB + s * G::B_BYTES;
                // one TMA instruction: the NA x boxes, then the NB dy boxes
                constexpr int NA = FA ? 2 : 1, NB = FA ? 4 : 1;
                if (lane < NA + NB) {
                    const bool isx = lane < NA;
                    const int j = isx ? lane : lane - NA;
                    const CUtensorMap *mp = isx ? &maps.x[t] : &maps.dy[t];
                    uint8_t *dst = (isx ? a : b) + j * 8192;
                    const int f = (isx ? f_c : f_k) + j * 64;
                    tma_load_2d(dst, mp, &full[s], FA ? f : n0, FA ? n0 : f, pol);
                }
            }
        }
        if (aborted && lane == 0 && last >= 0) mbar_wait(&full[last % G::STAGES], (last / G::STAGES) & 1, nullptr);
        __syncwarp();
    } else if (warp == kProducers) {
        if (elect_one()) {
            const uint64_t a_desc0 = sdesc(smem_u32(sA), A_LBO, 1024, SW_128);
            const uint64_t b_desc0 = sdesc(smem_u32(sB), B_LBO, 1024, SW_128);
            int it = 0;
            for (int u = 0; u < nunits && !aborted; ++u) {
                const int buf = u & 1;
                if (u >= 2 && !mbar_wait(&acc_empty[buf], ((u >> 1) - 1) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * 256;
                for (int c = 0; c < total; ++c, ++it) {
                    const int s = it % G::STAGES;
                    if (!mbar_wait(&full[s], (it / G::STAGES) & 1, p.status)) {
                        aborted = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((s * G::A_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + ((s * G::B_BYTES) >> 4);
#pragma unroll
                    for (int ks = 0; ks < G::TK / 16; ++ks)
                        mma_ss(d, ad + ((ks * KSTEP) >> 4), bd + ((ks * KSTEP) >> 4), IDESC,
                               (c > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                mma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else {
        const int q = warp & 3;                  // TMEM lane quarter = block row c0 + q
        for (int u = 0; u < nunits; ++u) {
            const int buf = u & 1;
            const bool ok = mbar_wait_warp(&acc_full[buf], (u >> 1) & 1, p.status, 128);
            if (!ok) break;
            tc_fence_after();
            const int32_t *ut = tab + 4 + u * kDUnitWords;
            const int cnt = ut[2];
            for (int e = 0; e < cnt; ++e) {
                const uint32_t wd = (uint32_t)ut[3 + e];
                const int sub = (int)(wd >> 24), id = (int)(wd & 0xFFFFFFu);
                if ((sub >> 3) != q) continue;
                float v[32];
#pragma unroll
                for (int c0 = 0; c0 < 32; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + buf * 256 + (sub & 7) * 32 + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
                }
                up_block32_out(&maps.dw, p, sout + q * 32 * 32, lane, id, v, aborted != 0);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (p.tma && lane == 0) bulk_wait_all();        // every dW store has completed before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProducers) tmem_dealloc(tmem, 512);
}

// Weight gradient on CTA pairs with two-SM MMAs, bs = 32.  A unit is a 256 x (32 nk) tile of
// x^T.dy (nk = 8, or 4 for split tail units): block rows c0..c0+7 by block columns
// k0..k0+nk-1, reduced over the minibatch in stages of 64 rows.  The even CTA holds tile rows
// 0-127 (block rows c0..c0+3) in its tensor memory, the odd CTA rows 128-255; each CTA loads
// its 128-feature slice of x (its half of A) and 128 dy features (its half of B, of which the
// MMA uses nk * 16), and the even CTA issues M256 x N x K16 MMAs over both CTAs' shared memory:
// 32 KB per CTA per stage for the MMA work that k_tc_updat_dense feeds with 48 KB.
// Accumulators are double-buffered (2 x 256 columns per CTA); the epilogue warps of both CTAs
// release a buffer to the even CTA's MMA warp, and epilogue warp q writes the present blocks
// of block row c0 + 4 rank + q with coalesced stores.
struct UpPairGeo {
    static constexpr int TK = 64;
    static constexpr int A_BYTES = 128 * TK * 2;                     // 16 KB
    static constexpr int B_BYTES = 128 * TK * 2;                     // 16 KB
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int PROD = 3;                                   // producer warps; warp w owns stages w, w + 3
    static constexpr int STAGES = 6;
    static constexpr int TAB_OFF = STAGES * STAGE;
    static constexpr int OUT_OFF = (TAB_OFF + kPTableWords * 4 + 1023) / 1024 * 1024;  // swizzled staging
    static constexpr int SMEM = OUT_OFF + 4 * 32 * 32 * 4;           // + a 32 x 32 fp32 block per epilogue warp
};

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

template <int FA, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kUpThreads, 1)
k_tc_updat_pair(const __grid_constant__ UpMaps maps, const UpParams p)
{
    using G = UpPairGeo;
    static_assert(G::STAGES % G::PROD == 0, "producer warp w must own stages w, w+PROD, ...");
    // fa=1: A = x^T MN-major (M atoms of 64 at 8 KB), B = dy MN-major (N atoms of 64 at 8 KB);
    // fa=0: both K-major, 128-byte rows.
    constexpr uint32_t A_LBO = FA ? 8192 : 16, B_LBO = FA ? 8192 : 16;
    constexpr uint32_t KSTEP = FA ? 16 * 128 : 32;
    constexpr uint32_t IDESC8 = idesc_f16(256, 256, BF16, FA == 1, FA == 1);
    constexpr uint32_t IDESC4 = idesc_f16(256, 128, BF16, FA == 1, FA == 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *tab = reinterpret_cast<int32_t *>(smem + G::TAB_OFF);
    float *sout = reinterpret_cast<float *>(smem + G::OUT_OFF);
    __shared__ __align__(8) uint64_t full[G::STAGES], empty[G::STAGES], acc_full[2], acc_empty[2], tab_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int chunks = (p.N + G::TK - 1) / G::TK;
    const int total = chunks * p.G;

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < G::STAGES; ++i) {
            mbar_init(&full[i], 1);                              // the even CTA's producer, + both halves' bytes
            mbar_init(&empty[i], 1);                             // one commit of the even CTA's MMA warp
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 8);                         // 4 epilogue warps in each CTA
        }
        mbar_init(&tab_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc_pair(&tmem_base, 512);
    tc_fence_before();
    cluster_sync();                                  // both CTAs' barriers and tensor memory exist
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    const int32_t *gtab = p.table + (size_t)pair * kPTableWords;
    if (warp == 0 && lane == 0) {
        const int nu = gtab[0];
        const uint32_t bytes = (uint32_t)(4 + nu * kPUnitWords) * 4u;
        mbar_arrive_expect_tx(&tab_full, bytes);
        bulk_load(tab, gtab, bytes, &tab_full, policy_evict_first());
    }
    pdl_wait();
    const bool tab_ok = mbar_wait_warp(&tab_full, 0, p.status, 64);
    const int nunits = tab_ok ? tab[0] : 0;
    const uint32_t full0 = map_to_rank(smem_u32(&full[0]), 0);       // the even CTA's barriers
    const uint32_t acc_empty0 = map_to_rank(smem_u32(&acc_empty[0]), 0);

    if (warp < G::PROD) {
        const uint64_t pol = policy_evict_last();
        int it = 0, last = -1;
        for (int u = 0; u < nunits && !aborted; ++u) {
            const int32_t *ut = tab + 4 + u * kPUnitWords;
            const int nk = ut[2];
            const int f_c = ut[0] * 32 + (int)rank * 128;         // this CTA's 128 tile rows
            const int f_k = ut[1] * 32 + (int)rank * nk * 16;     // this CTA's half of the tile columns
            for (int c = 0; c < total; ++c, ++it) {
                if (it % G::PROD != warp) continue;
                const int t = c / chunks, n0 = (c % chunks) * G::TK;
                const int s = it % G::STAGES;
                if (lane == 0) {
                    if (it >= G::STAGES && !mbar_wait(&empty[s], ((it / G::STAGES) - 1) & 1, p.status)) aborted = 1;
                    else if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * G::STAGE);
                }
                __syncwarp();
                if (aborted) break;
                last = it;
                uint8_t *a = smem + s * G::STAGE;
                uint8_t *b = a + G::A_BYTES;
                const uint32_t fb = full0 + (uint32_t)s * 8u;
                // one TMA instruction: the NB x boxes, then the NB dy boxes
                constexpr int NB = FA ? 2 : 1;
                if (lane < 2 * NB) {
                    const bool isx = lane < NB;
                    const int j = isx ? lane : lane - NB;
                    const CUtensorMap *mp = isx ? &maps.x[t] : &maps.dy[t];
                    uint8_t *dst = (isx ? a : b) + j * 8192;
                    const int f = (isx ? f_c : f_k) + j * 64;
                    tma_load_2d_pair(dst, mp, fb, FA ? f : n0, FA ? n0 : f, pol);
                }
            }
        }
        // The last release of this warp's stages comes from the even CTA's MMA warp: waiting for
        // it means no commit of the peer is still on its way to this CTA when it exits.
        if (!aborted && lane == 0 && last >= 0) {
            mbar_wait(&empty[last % G::STAGES], (last / G::STAGES) & 1, p.status);
            if (last >= G::PROD)
                mbar_wait(&empty[(last - G::PROD) % G::STAGES], ((last - G::PROD) / G::STAGES) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == kProducers) {
        if (rank == 0 && elect_one()) {
            const uint64_t a_desc0 = sdesc(smem_u32(smem), A_LBO, 1024, SW_128);
            const uint64_t b_desc0 = sdesc(smem_u32(smem) + G::A_BYTES, B_LBO, 1024, SW_128);
            int it = 0;
            for (int u = 0; u < nunits && !aborted; ++u) {
                const int buf = u & 1;
                const uint32_t idesc = tab[4 + u * kPUnitWords + 2] == 8 ? IDESC8 : IDESC4;
                if (u >= 2 && !mbar_wait(&acc_empty[buf], ((u >> 1) - 1) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * 256;
                for (int c = 0; c < total; ++c, ++it) {
                    const int s = it % G::STAGES;
                    if (!mbar_wait(&full[s], (it / G::STAGES) & 1, p.status)) {
                        aborted = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((s * G::STAGE) >> 4);
                    const uint64_t bd = b_desc0 + ((s * G::STAGE) >> 4);
#pragma unroll
                    for (int ks = 0; ks < G::TK / 16; ++ks)
                        mma_pair_ss(d, ad + ((ks * KSTEP) >> 4), bd + ((ks * KSTEP) >> 4), idesc,
                                    (c > 0 || ks > 0) ? 1u : 0u);
                    mma_pair_commit_mc(&empty[s], 3);             // releases the stage in both CTAs
                }
                mma_pair_commit_mc(&acc_full[buf], 3);
            }
        }
        __syncwarp();
    } else if (warp > kProducers) {
        const int q = warp & 3;                  // TMEM lane quarter = block row c0 + 4 rank + q
        const int row = (int)rank * 4 + q;
        for (int u = 0; u < nunits; ++u) {
            const int buf = u & 1;
            const bool ok = mbar_wait_warp(&acc_full[buf], (u >> 1) & 1, p.status, 128);
            if (!ok) break;
            tc_fence_after();
            const int32_t *ut = tab + 4 + u * kPUnitWords;
            const int cnt = ut[3];
            for (int e = 0; e < cnt; ++e) {
                const uint32_t wd = (uint32_t)ut[4 + e];
                const int sub = (int)(wd >> 24), id = (int)(wd & 0xFFFFFFu);
                if ((sub >> 3) != row) continue;
                float v[32];
#pragma unroll
                for (int c0 = 0; c0 < 32; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + buf * 256 + (sub & 7) * 32 + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
                }
                up_block32_out(&maps.dw, p, sout + q * 32 * 32, lane, id, v, aborted != 0);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)buf * 8u);
        }
        if (p.tma && lane == 0) bulk_wait_all();        // every dW store has completed before the CTA exits
    }
    if (aborted) {
        // copies of the pair may still be landing in this CTA: give them time (bounded)
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 20000u) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                  // both CTAs are done with the pair's tensor memory
    if (warp == kProducers) tmem_dealloc_pair(tmem, 512);
}

// Dense-tile fprop / bprop, bs = 32.  A CTA computes D[128 output features][256 minibatch
// rows] for a group of 4 output blocks: D += A[128 x 32] . B[32 x 256] for each present
// source block, A being the group's 4 weight blocks of that source (absent ones are zero
// tiles) and B the activation panel.  Sources are loaded in adjacent pairs so activation
// rows are 128 bytes.  Every MMA is M128 x N256 x K16.
//   fprop: A[(out, j)][i] = w(src, out)[i][j]  -> MN-major, 4 SW64 blocks 2 KB apart
//   bprop: A[(out, i)][j] = w(out, src)[i][j]  -> K-major, 128 rows of 64 bytes
//   (N,C) activations: B rows = minibatch rows of 128 bytes (K-major, SW128)
//   (C,N) activations: B = four 64-column MN-major SW128 atoms, 8 KB apart
struct FbdParams {
    void *out;
    const uint32_t *stream;
    const int32_t *off, *len;
    int32_t *status;
    int N, Fout, n_tiles;
};

template <int FA, bool BWD, bool BF16>
__global__ void __launch_bounds__(kFbThreads, 1)
k_tc_fbd(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
         const __grid_constant__ CUtensorMap tm_zero, const __grid_constant__ CUtensorMap tm_out, const FbdParams p)
{
    constexpr int STAGES = 4;                                    // = kProducers: warp w owns stage w
    static_assert(STAGES % kProducers == 0, "producer warp w must own stages w, w+4, ...");
    constexpr int A_BYTES = 16384, B_BYTES = 32768, STAGE = A_BYTES + B_BYTES;
    constexpr uint32_t A_LBO = BWD ? 16 : 2048, A_SBO = 512, A_KSTEP = BWD ? 32 : 1024;
    constexpr uint32_t B_LBO = FA ? 16 : 8192, B_KSTEP = FA ? 32 : 2048, B_SUB = FA ? 64 : 4096;
    constexpr uint32_t IDESC = idesc_f16(128, 256, BF16, !BWD, FA == 0);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t *sched = reinterpret_cast<const uint32_t *>(smem + STAGES * STAGE);
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], acc_full, sched_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int grp = blockIdx.x / p.n_tiles;
    const int n0 = (blockIdx.x % p.n_tiles) * 256;
    const int len = p.len[grp];

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&sched_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc(&tmem_base, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    // The tile schedule belongs to the handle: fetch it before waiting for the previous kernel.
    if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(&sched_full, (uint32_t)len * 4u);
        bulk_load((void *)sched, p.stream + p.off[grp], (uint32_t)len * 4u, &sched_full, policy_evict_last());
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_w);
    }
    pdl_wait();

    if (warp < kProducers) {
        const uint64_t pol_act = policy_evict_last();
        const uint64_t pol_w = policy_evict_first();
        if (!mbar_wait_warp(&sched_full, 0, p.status, 64)) aborted = 1;
        __syncwarp();
        int last = -1;
        for (int chunk = 0, pos = 0; !aborted; ++chunk, pos += 9) {
            const uint32_t hdr = sched[pos];
            if (hdr == 0xFFFFFFFFu) break;
            if (chunk % kProducers != warp) continue;
            const int st = chunk % STAGES;
            if (lane == 0) {
                if (chunk >= STAGES && !mbar_wait(&empty[st], ((chunk / STAGES) - 1) & 1, p.status)) aborted = 1;
                else mbar_arrive_expect_tx(&full[st], (uint32_t)STAGE);
            }
            __syncwarp();
            if (aborted) break;
            last = chunk;
            const int pr = (int)(hdr >> 8);
            uint8_t *a = smem + st * STAGE;
            uint8_t *b = a + A_BYTES;
            // one TMA instruction: lanes < NX the activation boxes, the next 8 lanes the weight
            // slots (sub * 4 + out), an absent block reading a zero tile
            constexpr int NX = FA ? 1 : 4;
            if (lane < NX + 8) {
                const bool isx = lane < NX;
                const int sl = lane - NX;
                const int id = isx ? 0 : (int)sched[pos + 1 + sl] - 1;
                const int zr = (int)((blockIdx.x * 13u + (unsigned)chunk * 8u + (unsigned)sl) % 128u) * 32;
                const CUtensorMap *mp = isx ? &tm_act : (id >= 0 ? &tm_w : &tm_zero);
                uint8_t *dst = isx ? b + lane * 8192 : a + (sl >> 2) * 8192 + (sl & 3) * 2048;
                const int cx = isx ? (FA ? pr * 64 : n0 + 64 * lane) : 0;
                const int cy = isx ? (FA ? n0 : pr * 64) : (id >= 0 ? id * 32 : zr);
                tma_load_2d(dst, mp, &full[st], cx, cy, isx ? pol_act : pol_w);
            }
        }
        if (aborted && lane == 0 && last >= 0) mbar_wait(&full[last % STAGES], (last / STAGES) & 1, nullptr);
        __syncwarp();
    } else {
        if (elect_one()) {
            const uint32_t s_base = smem_u32(smem);
            const uint64_t a_desc0 = sdesc(s_base, A_LBO, A_SBO, SW_64);
            const uint64_t b_desc0 = sdesc(s_base + A_BYTES, B_LBO, 1024, SW_128);
            uint32_t acc = 0;
            if (!mbar_wait(&sched_full, 0, p.status)) aborted = 1;
            for (int chunk = 0, pos = 0; !aborted; ++chunk, pos += 9) {
                const uint32_t hdr = sched[pos];
                if (hdr == 0xFFFFFFFFu) break;
                const int st = chunk % STAGES;
                if (!mbar_wait(&full[st], (chunk / STAGES) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t so = st * STAGE;
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    if (!((hdr >> (sub * 4)) & 0xFu)) continue;     // no block of this source in the group
                    const uint64_t ad = a_desc0 + ((so + sub * 8192) >> 4);
                    const uint64_t bd = b_desc0 + ((so + sub * B_SUB) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        mma_ss(tmem, ad + ((ks * A_KSTEP) >> 4), bd + ((ks * B_KSTEP) >> 4), IDESC, acc);
                        acc = 1;
                    }
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&acc_full);
        }
        __syncwarp();
    }
    if (warp < kProducers) {
        // epilogue: warp q holds output features 32q..32q+31 of the group, lane = feature
        const int q = warp & 3;
        const int f = grp * 128 + q * 32 + lane;
        const bool ok = mbar_wait_warp(&acc_full, 0, p.status, 256);
        tc_fence_after();
        const bool any = len > 4;                     // at least one entry (else the stream is the end marker)
        uint16_t *out = static_cast<uint16_t *>(p.out);
        // (N,C) outputs: the bf16 tile is staged as [256 minibatch rows][128 features] in the
        // idle stage memory and written by one TMA store; (C,N) outputs are row-contiguous.
        uint16_t *tile = reinterpret_cast<uint16_t *>(smem);
        for (int c0 = 0; c0 < 256; c0 += 32) {
            if (!FA && n0 + c0 >= p.N) break;
            float v[32];
            if (ok && any) {
#pragma unroll
                for (int h2 = 0; h2 < 32; h2 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0 + h2, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[h2 + j] = __uint_as_float(r[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (FA) {
#pragma unroll
                for (int j = 0; j < 32; ++j) tile[(c0 + j) * 128 + q * 32 + lane] = cvt1<BF16>(v[j]);
                continue;
            }
            if (f >= p.Fout) continue;
            const int nb = n0 + c0;
            uint16_t *dst = out + (size_t)f * p.N + nb;
            if (nb + 32 <= p.N) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 pk;
                    pk.x = pack2<BF16>(v[j], v[j + 1]);
                    pk.y = pack2<BF16>(v[j + 2], v[j + 3]);
                    pk.z = pack2<BF16>(v[j + 4], v[j + 5]);
                    pk.w = pack2<BF16>(v[j + 6], v[j + 7]);
                    *reinterpret_cast<uint4 *>(dst + j) = pk;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (nb + j < p.N) dst[j] = cvt1<BF16>(v[j]);
            }
        }
        if (FA) {
            fence_proxy_async_smem();
            named_sync(1, 32 * kProducers);
            if (warp == 0 && lane == 0) {
                tma_store_2d(&tm_out, tile, grp * 128, n0);
                bulk_commit();
                bulk_wait_read();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProducers) tmem_dealloc(tmem, 256);
}

// Dense-tile fprop / bprop on CTA pairs with two-SM MMAs, bs = 32.  A pair computes
// D[256 output features][256 minibatch rows] for a group of 8 output blocks.  M = 256 is split
// over the two CTAs' tensor memory (the even CTA holds the group's outputs 0-3, the odd one
// 4-7); each CTA loads only its own 4 weight blocks per source (its half of A) and 128 of the
// 256 activation rows (its half of B), and the even CTA issues M256 x N256 x K16 MMAs that
// read both CTAs' shared memory.  Per pair of sources a CTA thus streams 32 KB instead of the
// 48 KB of k_tc_fbd for the same MMA work per SM, which is what the L2 -> SM rate limits.
//   Loads of both CTAs complete on the even CTA's `full` barrier (which expects both halves);
//   the even CTA's commits release the stage in both CTAs and finally signal both
//   accumulators.  Operand layouts per CTA are those of k_tc_fbd with 128 activation rows.
template <int FA, bool BWD, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFbpThreads, 1)
k_tc_fbd_pair(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_zero, const __grid_constant__ CUtensorMap tm_out,
              const FbdParams p)
{
    constexpr int PROD = 3;                                      // producer warps; warp w owns stages w, w + 3
    constexpr int STAGES = 6;
    static_assert(STAGES % PROD == 0, "producer warp w must own stages w, w+PROD, ...");
    constexpr int A_BYTES = 16384, B_BYTES = 16384, STAGE = A_BYTES + B_BYTES;
    constexpr uint32_t A_LBO = BWD ? 16 : 2048, A_SBO = 512, A_KSTEP = BWD ? 32 : 1024;
    constexpr uint32_t B_LBO = FA ? 16 : 8192, B_KSTEP = FA ? 32 : 2048, B_SUB = FA ? 64 : 4096;
    constexpr uint32_t IDESC = idesc_f16(256, 256, BF16, !BWD, FA == 0);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t *sched = reinterpret_cast<const uint32_t *>(smem + STAGES * STAGE);
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], acc_full, sched_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int tile = blockIdx.x >> 1;
    const int grp = tile / p.n_tiles;                            // group of 8 output blocks
    const int n0 = (tile % p.n_tiles) * 256;
    const int len = p.len[grp];

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);                              // the even CTA's producer, + both halves' bytes
            mbar_init(&empty[i], 1);                             // one commit of the even CTA's MMA warp
        }
        mbar_init(&acc_full, 1);
        mbar_init(&sched_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc_pair(&tmem_base, 256);
    tc_fence_before();
    cluster_sync();                                  // both CTAs' barriers and tensor memory exist
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(&sched_full, (uint32_t)len * 4u);
        bulk_load((void *)sched, p.stream + p.off[grp], (uint32_t)len * 4u, &sched_full, policy_evict_last());
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_w);
    }
    pdl_wait();
    const uint32_t full0 = map_to_rank(smem_u32(&full[0]), 0);   // the even CTA's full[0]

    if (warp < PROD) {
        const uint64_t pol_act = policy_evict_last();
        const uint64_t pol_w = policy_evict_first();
        if (!mbar_wait_warp(&sched_full, 0, p.status, 64)) aborted = 1;
        __syncwarp();
        int last = -1;
        for (int chunk = 0, pos = 0; !aborted; ++chunk, pos += 17) {
            const uint32_t hdr = sched[pos];
            if (hdr == 0xFFFFFFFFu) break;
            if (chunk % PROD != warp) continue;
            const int st = chunk % STAGES;
            if (lane == 0) {
                if (chunk >= STAGES && !mbar_wait(&empty[st], ((chunk / STAGES) - 1) & 1, p.status)) aborted = 1;
                else if (rank == 0) mbar_arrive_expect_tx(&full[st], 2u * STAGE);
            }
            __syncwarp();
            if (aborted) break;
            last = chunk;
            const int pr = (int)(hdr >> 16);
            uint8_t *a = smem + st * STAGE;
            uint8_t *b = a + A_BYTES;
            const uint32_t fb = full0 + (uint32_t)st * 8u;
            // one TMA instruction: lanes < NX this CTA's activation boxes, the next 8 lanes its
            // weight slots (sub * 4 + out), an absent block reading a zero tile
            constexpr int NX = FA ? 1 : 2;
            if (lane < NX + 8) {
                const bool isx = lane < NX;
                const int sl = lane - NX, sub = sl >> 2, o = sl & 3;
                const int id = isx ? 0 : (int)sched[pos + 1 + sub * 8 + (int)rank * 4 + o] - 1;
                const int zr = (int)((blockIdx.x * 13u + (unsigned)chunk * 8u + (unsigned)sl) % 128u) * 32;
                const CUtensorMap *mp = isx ? &tm_act : (id >= 0 ? &tm_w : &tm_zero);
                uint8_t *dst = isx ? b + lane * 8192 : a + sub * 8192 + o * 2048;
                const int cx = isx ? (FA ? pr * 64 : n0 + 128 * (int)rank + 64 * lane) : 0;
                const int cy = isx ? (FA ? n0 + 128 * (int)rank : pr * 64) : (id >= 0 ? id * 32 : zr);
                tma_load_2d_pair(dst, mp, fb, cx, cy, isx ? pol_act : pol_w);
            }
        }
        // The last release of this warp's stages comes from the even CTA's MMA warp: waiting for
        // it means no commit of the peer is still on its way to this CTA when it exits.
        if (!aborted && lane == 0 && last >= 0) {
            mbar_wait(&empty[last % STAGES], (last / STAGES) & 1, p.status);
            if (last >= PROD) mbar_wait(&empty[(last - PROD) % STAGES], ((last - PROD) / STAGES) & 1, p.status);
        }
        __syncwarp();
    } else if (warp == kProducers) {
        if (rank == 0 && elect_one()) {
            const uint32_t s_base = smem_u32(smem);
            const uint64_t a_desc0 = sdesc(s_base, A_LBO, A_SBO, SW_64);
            const uint64_t b_desc0 = sdesc(s_base + A_BYTES, B_LBO, 1024, SW_128);
            uint32_t acc = 0;
            if (!mbar_wait(&sched_full, 0, p.status)) aborted = 1;
            for (int chunk = 0, pos = 0; !aborted; ++chunk, pos += 17) {
                const uint32_t hdr = sched[pos];
                if (hdr == 0xFFFFFFFFu) break;
                const int st = chunk % STAGES;
                if (!mbar_wait(&full[st], (chunk / STAGES) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t so = st * STAGE;
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    if (!((hdr >> (sub * 8)) & 0xFFu)) continue;  // no block of this source in the group
                    const uint64_t ad = a_desc0 + ((so + sub * 8192) >> 4);
                    const uint64_t bd = b_desc0 + ((so + sub * B_SUB) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        mma_pair_ss(tmem, ad + ((ks * A_KSTEP) >> 4), bd + ((ks * B_KSTEP) >> 4), IDESC, acc);
                        acc = 1;
                    }
                }
                mma_pair_commit_mc(&empty[st], 3);        // releases the stage in both CTAs
            }
            mma_pair_commit_mc(&acc_full, 3);
        }
        __syncwarp();
    }
    if (warp != kProducers) {
        // epilogue, 8 warps: warp w holds output features 32q..32q+31 (q = w mod 4, lane =
        // feature) of this CTA's half for minibatch columns 128h..128h+127 (h = 0 for warps
        // 0-3, 1 for warps 5-8)
        const int q = warp & 3;
        const int h = warp < kProducers ? 0 : 1;
        const int lead = h ? kProducers + 1 : 0;      // warp that stores the half's slices
        const int fbase = grp * 256 + (int)rank * 128;
        const int f = fbase + q * 32 + lane;
        const bool ok = mbar_wait_warp(&acc_full, 0, p.status, 256);
        tc_fence_after();
        const bool any = len > 4;                     // at least one entry (else the stream is the end marker)
        uint16_t *out = static_cast<uint16_t *>(p.out);
        // (N,C) outputs: the bf16 tile [256 rows][128 features] is staged in the idle stage
        // memory 32 rows at a time; each 32-row slice is stored by one TMA store as soon as the
        // half's four warps have written it, overlapping the stores with the remaining TMEM reads.
        uint16_t *tile_s = reinterpret_cast<uint16_t *>(smem);
        for (int c0 = h * 128; c0 < h * 128 + 128; c0 += 32) {
            if (!FA && n0 + c0 >= p.N) break;
            float v[32];
            if (ok && any) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, r0);
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0 + 16, r1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v[j] = __uint_as_float(r0[j]);
                    v[16 + j] = __uint_as_float(r1[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (FA) {
#pragma unroll
                for (int j = 0; j < 32; ++j) tile_s[(c0 + j) * 128 + q * 32 + lane] = cvt1<BF16>(v[j]);
                fence_proxy_async_smem();
                named_sync(1 + h, 128);
                if (warp == lead && lane == 0) {
                    tma_store_2d(&tm_out, tile_s + c0 * 128, fbase, n0 + c0);
                    bulk_commit();
                }
                continue;
            }
            if (f >= p.Fout) continue;
            const int nb = n0 + c0;
            uint16_t *dst = out + (size_t)f * p.N + nb;
            if (nb + 32 <= p.N) {
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 pk;
                    pk.x = pack2<BF16>(v[j], v[j + 1]);
                    pk.y = pack2<BF16>(v[j + 2], v[j + 3]);
                    pk.z = pack2<BF16>(v[j + 4], v[j + 5]);
                    pk.w = pack2<BF16>(v[j + 6], v[j + 7]);
                    *reinterpret_cast<uint4 *>(dst + j) = pk;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (nb + j < p.N) dst[j] = cvt1<BF16>(v[j]);
            }
        }
        if (FA && warp == lead && lane == 0) bulk_wait_read();   // the slices have left shared memory
    }
    if (aborted) {
        // copies of the pair may still be landing in this CTA: give them time (bounded)
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 20000u) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                  // both CTAs are done with the pair's tensor memory
    if (warp == kProducers) tmem_dealloc_pair(tmem, 256);
}

// Dense-tile fprop / bprop for a minibatch of at most 64 rows, bs = 32.  Same tiles and
// operands as k_tc_fbd with N = 64, but a 64-row minibatch gives too few tiles to fill the
// GPU, so a cluster of kSplit CTAs shares one tile: CTA r multiplies the r-th quarter of the
// tile's source pairs.  The partial tiles are then summed across the cluster in distributed
// shared memory, each CTA owning 32 of the tile's 128 output features: it receives the other
// three CTAs' fp32 partials of its features into its (then idle) stage memory, next to its
// own, and its four warps add them for 16 minibatch columns each, round once and store.  No
// atomics and no global scratch; with the reduction buffer inside the stage memory, 8 stages
// of 24 KB keep the weight stream from HBM in flight.
constexpr int kSplit = 4;

template <int FA, bool BWD, bool BF16>
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kFbThreads, 1)
k_tc_fbd_split(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_zero, const FbdParams p)
{
    constexpr int STAGES = 8;                                    // warp w owns stages w and w + 4
    static_assert(STAGES % kProducers == 0, "producer warp w must own stages w, w+4, ...");
    static_assert(kSplit == kProducers, "CTA r of the cluster owns the features of epilogue warp r");
    constexpr int A_BYTES = 16384, B_BYTES = 8192, STAGE = A_BYTES + B_BYTES;
    constexpr uint32_t A_LBO = BWD ? 16 : 2048, A_SBO = 512, A_KSTEP = BWD ? 32 : 1024;
    constexpr uint32_t B_LBO = FA ? 16 : 8192, B_KSTEP = FA ? 32 : 2048, B_SUB = FA ? 64 : 4096;
    constexpr uint32_t IDESC = idesc_f16(128, 64, BF16, !BWD, FA == 0);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // after the main loop: red[slot][j / 4][lane][4], the partials of this CTA's 32 features
    // from the three other CTAs (slots 0-2) and its own (slot 3)
    float *red = reinterpret_cast<float *>(smem);
    const uint32_t *sched = reinterpret_cast<const uint32_t *>(smem + STAGES * STAGE);
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], acc_full, sched_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int grp = blockIdx.x / kSplit;
    const int len = p.len[grp];

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&sched_full, 1);
        fence_barrier_init();
    }
    if (warp == kProducers) tmem_alloc(&tmem_base, 64);
    tc_fence_before();
    cluster_sync();                                  // every CTA of the cluster is running
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA of this grid holds its tensor memory before a dependent kernel may start, so a
    // dependent CTA that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();

    // this CTA's share of the tile's entries (the stream ends with 0xFFFFFFFF)
    int lo = 0, hi = 0;
    if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(&sched_full, (uint32_t)len * 4u);
        bulk_load((void *)sched, p.stream + p.off[grp], (uint32_t)len * 4u, &sched_full, policy_evict_last());
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_w);
    }
    pdl_wait();
    if (!mbar_wait(&sched_full, 0, p.status)) aborted = 1;
    {
        const int n = (len - 1) / 9;                 // 9-word entries, the end marker, < 4 words of padding
        lo = (int)(rank * n / kSplit);
        hi = (int)((rank + 1) * n / kSplit);
    }

    if (warp < kProducers) {
        const uint64_t pol_act = policy_evict_last();
        const uint64_t pol_w = policy_evict_first();
        int last = -1, prev = -1;
        for (int e = lo; e < hi && !aborted; ++e) {
            const int chunk = e - lo, pos = e * 9;
            if (chunk % kProducers != warp) continue;
            const uint32_t hdr = sched[pos];
            const int st = chunk % STAGES;
            if (lane == 0) {
                if (chunk >= STAGES && !mbar_wait(&empty[st], ((chunk / STAGES) - 1) & 1, p.status)) aborted = 1;
                else mbar_arrive_expect_tx(&full[st], (uint32_t)STAGE);
            }
            __syncwarp();
            if (aborted) break;
            prev = last;
            last = chunk;
            const int pr = (int)(hdr >> 8);
            uint8_t *a = smem + st * STAGE;
            uint8_t *b = a + A_BYTES;
            // one TMA instruction: lane 0 the activation panel, lanes 1..8 the weight slots
            // (sub * 4 + out), an absent block reading a zero tile
            if (lane < 9) {
                const bool isx = lane == 0;
                const int sl = lane - 1;
                const int id = isx ? 0 : (int)sched[pos + 1 + sl] - 1;
                const int zr = (int)((blockIdx.x * 13u + (unsigned)chunk * 8u + (unsigned)sl) % 128u) * 32;
                const CUtensorMap *mp = isx ? &tm_act : (id >= 0 ? &tm_w : &tm_zero);
                uint8_t *dst = isx ? b : a + (sl >> 2) * 8192 + (sl & 3) * 2048;
                const int cx = isx ? (FA ? pr * 64 : 0) : 0;
                const int cy = isx ? (FA ? 0 : pr * 64) : (id >= 0 ? id * 32 : zr);
                tma_load_2d(dst, mp, &full[st], cx, cy, isx ? pol_act : pol_w);
            }
        }
        if (aborted && lane == 0) {
            // let this warp's copies in flight land before the stage memory is reused
            if (last >= 0) mbar_wait(&full[last % STAGES], (last / STAGES) & 1, nullptr);
            if (prev >= 0) mbar_wait(&full[prev % STAGES], (prev / STAGES) & 1, nullptr);
        }
        __syncwarp();
    } else {
        if (elect_one()) {
            const uint32_t s_base = smem_u32(smem);
            const uint64_t a_desc0 = sdesc(s_base, A_LBO, A_SBO, SW_64);
            const uint64_t b_desc0 = sdesc(s_base + A_BYTES, B_LBO, 1024, SW_128);
            uint32_t acc = 0;
            for (int e = lo; e < hi && !aborted; ++e) {
                const int chunk = e - lo;
                const uint32_t hdr = sched[e * 9];
                const int st = chunk % STAGES;
                if (!mbar_wait(&full[st], (chunk / STAGES) & 1, p.status)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t so = st * STAGE;
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    if (!((hdr >> (sub * 4)) & 0xFu)) continue;
                    const uint64_t ad = a_desc0 + ((so + sub * 8192) >> 4);
                    const uint64_t bd = b_desc0 + ((so + sub * B_SUB) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        mma_ss(tmem, ad + ((ks * A_KSTEP) >> 4), bd + ((ks * B_KSTEP) >> 4), IDESC, acc);
                        acc = 1;
                    }
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&acc_full);
        }
        __syncwarp();
    }
    // partial tile: warp q holds output features 32q..32q+31 (lane = feature) for the 64
    // minibatch columns; CTA q of the cluster owns those features
    float v[64];
    const int q = warp & 3;
    if (warp < kProducers) {
        const bool ok = mbar_wait_warp(&acc_full, 0, p.status, 128);
        tc_fence_after();
        if (ok && hi > lo) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = 0.f;
        }
    }
    cluster_sync();                                  // every CTA's MMAs are done: stage memory is free
    if (warp < kProducers) {
        // warp q sends its partial to CTA q (slot = the sender's rank among the other three);
        // the owner's own partial goes to slot 3 of its own buffer
        const int slot = q == (int)rank ? 3 : ((int)rank < q ? (int)rank : (int)rank - 1);
        const uint32_t dst = map_to_rank(smem_u32(red + (slot * 16 * 32 + lane) * 4), (uint32_t)q);
#pragma unroll
        for (int j = 0; j < 64; j += 4) st_cluster_v4(dst + (j / 4) * 32 * 16, v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
    cluster_sync();                                  // all four partials of this CTA's features have landed
    if (warp < kProducers) {
        // warp w sums minibatch columns 16w .. 16w+15 of the CTA's 32 features (lane = feature):
        // own partial first, then the other CTAs' in rank order, rounded once
        const int f = grp * 128 + (int)rank * 32 + lane;
        float r16[16];
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4) {
            const int j4 = (warp * 16 + jj) / 4;
            float4 acc4 = *reinterpret_cast<const float4 *>(red + ((3 * 16 + j4) * 32 + lane) * 4);
#pragma unroll
            for (int sl = 0; sl < kSplit - 1; ++sl) {
                const float4 t4 = *reinterpret_cast<const float4 *>(red + ((sl * 16 + j4) * 32 + lane) * 4);
                acc4.x += t4.x;
                acc4.y += t4.y;
                acc4.z += t4.z;
                acc4.w += t4.w;
            }
            r16[jj] = acc4.x;
            r16[jj + 1] = acc4.y;
            r16[jj + 2] = acc4.z;
            r16[jj + 3] = acc4.w;
        }
        uint16_t *out = static_cast<uint16_t *>(p.out);
        const int j0 = warp * 16;
        if (f < p.Fout) {
            if (FA) {
                // (N, F) rows: each store writes 64 contiguous bytes of one minibatch row
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (j0 + jj < p.N) out[(size_t)(j0 + jj) * p.Fout + f] = cvt1<BF16>(r16[jj]);
            } else if (j0 + 16 <= p.N) {
                uint16_t *dst = out + (size_t)f * p.N + j0;
#pragma unroll
                for (int jj = 0; jj < 16; jj += 8) {
                    uint4 pk;
                    pk.x = pack2<BF16>(r16[jj], r16[jj + 1]);
                    pk.y = pack2<BF16>(r16[jj + 2], r16[jj + 3]);
                    pk.z = pack2<BF16>(r16[jj + 4], r16[jj + 5]);
                    pk.w = pack2<BF16>(r16[jj + 6], r16[jj + 7]);
                    *reinterpret_cast<uint4 *>(dst + jj) = pk;
                }
            } else {
                uint16_t *dst = out + (size_t)f * p.N + j0;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (j0 + jj < p.N) dst[jj] = cvt1<BF16>(r16[jj]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProducers) tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------

// Launches with programmatic stream serialization when `pdl` is set: the kernel may start
// while the previous kernel on the stream finishes; it fetches handle-owned schedules, then
// waits in pdl_wait() before it touches any caller buffer.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int BS, int FA, bool BWD, bool BF16>
bsmm_status launch_fb(bsmm_ctx *h, FbSched &fs, const FbStages &geo, const void *act, const void *w, void *out,
                      int N, bsmm_dtype t, cudaStream_t s)
{
    constexpr int BSE = BS == 8 ? 16 : BS;
    TcState *st = state(h);
    const int C = h->R * BS, K = h->S * BS;
    const int Fin = BWD ? K : C, Fout = BWD ? C : K;
    CUtensorMap m_act, m_w, m_zero;
    bool ok;
    if (FA)
        ok = make_map2d(&m_act, act, t, Fin, N, fb_row_bytes(BSE) / 2, geo.half ? 64 : 128,
                        fb_row_bytes(BSE) == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    else ok = make_map2d(&m_act, act, t, N, Fin, 64, BSE, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint64_t wrows = (uint64_t)std::max<int64_t>(h->nnz, 1) * BS;
    const void *wp = h->nnz > 0 ? w : st->d_zero;
    if (BS == 8) ok = ok && make_map2d(&m_w, wp, t, 8, h->nnz > 0 ? wrows : 16, 8, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    else ok = ok && make_map2d(&m_w, wp, t, BS, h->nnz > 0 ? wrows : BS, BS, BS, swz_for_row_bytes(BS * 2));
    ok = ok && make_map2d(&m_zero, st->d_zero, t, 8, kZeroTiles * 8, 8, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return BSMM_ERR_CUDA;
    FbParams p;
    p.out = out;
    p.stream = fs.d_stream;
    p.win_desc = fs.d_win_desc;
    p.win_out = fs.d_win_out;
    p.status = h->d_status;
    p.N = N;
    p.Fout = Fout;
    p.W = fs.W;
    p.Fslots = fs.Fslots;
    p.n_tiles = geo.half ? (N + 63) / 64 : (N + 127) / 128;
    p.g = geo;
    const int smem = geo.stages * geo.stage_bytes + geo.a_slot + kSchedWords * 4 + 1024;
    auto kern = k_tc_fb<BS, FA, BWD, BF16>;
    static std::atomic<int> attr_set{-1};     // device ordinal the attribute was last set for
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    dim3 grid(fs.nwin * p.n_tiles);
    const cudaError_t le = launch_pdl(kern, grid, dim3(kFbThreads), smem, s, true, m_act, m_w, m_zero, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

int dw_code(bsmm_dtype dw_t) { return dw_t == BSMM_F32 ? 0 : dw_t == BSMM_F16 ? 1 : 2; }

// bs 32 / 16: the weight-gradient epilogues write dW blocks by TMA store, or TMA reduce-add when
// accumulating a float32 dW (a 16-bit dW accumulates through registers: the sum is formed in
// float32, then rounded once); sets p.tma and the dW tensor map (one block per box, rows swizzled
// by their byte width).  BSMM_UP_EPI=stores keeps the per-thread stores.  p.dwt, p.accumulate set.
bool set_dw_map(const bsmm_ctx *h, UpMaps &maps, UpParams &p, void *dw, int BS)
{
    const char *ue = getenv("BSMM_UP_EPI");
    p.tma = BS != 8 && h->nnz > 0 && (p.dwt == 0 || !p.accumulate) && !(ue && !strcmp(ue, "stores")) ? 1 : 0;
    if (!p.tma) return true;
    const int eb = p.dwt == 0 ? 4 : 2;
    const CUtensorMapDataType dt = p.dwt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : p.dwt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int rowb = BS * eb;
    const CUtensorMapSwizzle sw = rowb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : swz_for_row_bytes(rowb);
    return make_map2d_dt(&maps.dw, dw, dt, eb, BS, (uint64_t)h->nnz * BS, BS, BS, sw);
}

template <int BS, int FA, bool BF16>
bsmm_status launch_up(bsmm_ctx *h, UpSched &us, const GroupPtrs &g, void *dw, int N, bsmm_dtype t, int acc,
                      cudaStream_t s, bsmm_dtype dw_t = BSMM_F32, bool pdl = true)
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
    p.table = us.d_table;
    p.status = h->d_status;
    p.N = N;
    p.G = g.G;
    p.accumulate = acc;
    p.dwt = dw_code(dw_t);
    p.nnz = h->nnz;
    if (!set_dw_map(h, maps, p, dw, BS)) return BSMM_ERR_CUDA;
    const int smem = G::SMEM + 1024;
    auto kern = k_tc_updat<BS, FA, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le = launch_pdl(kern, dim3(us.ctas), dim3(kUpThreads), smem, s, pdl, maps, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

// Stage geometry for a call.  P producer warps share the chunks (chunk c -> warp c mod P)
// and P divides the stage count: warp w then owns stages w, w+P, ... and waits on each
// stage's `empty` barrier one phase at a time, which is what a parity wait requires.
// Chunks hold the expected records of one activation entry (window size x blocks per
// panel group x layout density) so entries are rarely split.  Two CTAs share an SM when
// there are more units than SMs and two stages fit in half of shared memory (one CTA's
// prologue and epilogue then overlap the other's main loop); otherwise one CTA takes most
// of shared memory.
FbStages choose_stages(const bsmm_ctx *h, int N, int64_t units, int W, bool rows64)
{
    const int bse = h->bs == 8 ? 16 : h->bs;
    FbStages g;
    g.half = (N <= 64 || rows64) ? 1 : 0;
    g.a_slot = (g.half ? 64 : 128) * (h->fa ? fb_row_bytes(bse) : bse * 2);
    const int b_slot = bse * bse * 2;
    const int a_ops = (h->fa || g.half) ? 1 : 2, b_ops = h->bs == 8 ? 4 : 1;
    const int gc = fb_row_sources(h->fa, bse);
    const double density = (double)h->nnz / ((double)h->R * h->S);
    const double coarse_density = h->bs == 8 ? std::min(1.0, 4.0 * density) : density;
    const int expect_r = (int)(1.25 * W * gc * coarse_density) + 1;
    // Activation panels per chunk.  Fewer, larger chunks cost less per byte: each chunk is one TMA
    // issue of a few hundred ns and one barrier round trip.  Measured on the recurrent step (bs 32,
    // (N,C), N = 128), back to back: one CTA per SM (binned fprop) with 2 / 4 / 8 panels 7.93 /
    // 7.59 / 7.11 us; two CTAs per SM (bprop) with 2 / 4 panels 7.57 / 7.26 us, while 8 panels
    // leave room for one CTA per SM only (10.85 us).  (N,C) activations therefore take the largest
    // of 8, 4, 2, 1 panels that keeps two stages and, with more units than SMs, two CTAs per SM.
    // (C,N) activations keep 2 panels (bs 32) or 4, and any count (also one pinned for tests) is
    // halved while two stages do not fit.
    const bool want_two = units > h->sm_count;
    int e_first = h->fa ? 8 : (h->bs == 32 ? 2 : 4);
    if (h->tc_eslots >= 1 && h->tc_eslots <= 8) e_first = h->tc_eslots;
    const int budget_two = h->tc_stage_kb >= 32 ? std::min(h->tc_stage_kb, 196) * 1024 : 96 * 1024;
    const int budget_one = h->tc_stage_kb >= 32 ? std::min(h->tc_stage_kb, 196) * 1024 : 196 * 1024;
    for (g.e_slots = e_first;; g.e_slots = g.e_slots > 2 ? g.e_slots / 2 : g.e_slots - 1) {
        const int r_cap = (32 - g.e_slots * a_ops) / b_ops;
        g.r_slots = std::max(2, std::min(r_cap, g.e_slots * expect_r));
        bool two = false;
        for (;;) {
            g.b_off = g.e_slots * g.a_slot;
            g.stage_bytes = (g.b_off + g.r_slots * b_slot + 1023) & ~1023;
            two = want_two && 2 * g.stage_bytes + g.a_slot <= budget_two;
            const int budget = two ? budget_two : budget_one;
            g.stages = std::min(kMaxStages, (budget - g.a_slot) / g.stage_bytes);
            if (g.stages >= 2 || g.r_slots <= 1) break;
            --g.r_slots;                               // shrink the chunk until two stages fit
        }
        const bool fits = g.stages >= 2 && (two || !want_two);
        if (fits || g.e_slots <= 1) break;
        // (C,N) activations and a pinned panel count only need two stages to fit
        if (g.stages >= 2 && (!h->fa || h->tc_eslots >= 1)) break;
    }
    g.stages = std::max(g.stages, 2);
    if (g.stages >= kProducers) {
        g.stages = g.stages / kProducers * kProducers;
        g.producers = kProducers;
    } else {
        g.stages = g.stages / 2 * 2;
        g.producers = 2;
    }
    return g;
}

template <int FA, bool BF16>
bsmm_status launch_up_dense(bsmm_ctx *h, UpDenseSched &us, const GroupPtrs &g, void *dw, int N, bsmm_dtype t,
                            int acc, cudaStream_t s, bsmm_dtype dw_t)
{
    using G = UpDenseGeo;
    const int C = h->R * 32, K = h->S * 32;
    UpMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int i = 0; i < g.G; ++i) {
        bool ok;
        if (FA) {
            ok = make_map2d(&maps.x[i], g.x[i], t, C, N, 64, G::TK, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, K, N, 64, G::TK, CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            ok = make_map2d(&maps.x[i], g.x[i], t, N, C, G::TK, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, N, K, G::TK, 256, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return BSMM_ERR_CUDA;
    }
    UpParams p;
    p.dw = dw;
    p.table = us.d_table;
    p.status = h->d_status;
    p.N = N;
    p.G = g.G;
    p.accumulate = acc;
    p.dwt = dw_code(dw_t);
    p.nnz = h->nnz;
    if (!set_dw_map(h, maps, p, dw, 32)) return BSMM_ERR_CUDA;
    const int smem = G::SMEM + 1024;
    auto kern = k_tc_updat_dense<FA, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le = launch_pdl(kern, dim3(us.ctas), dim3(kUpThreads), smem, s, true, maps, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int FA, bool BF16>
bsmm_status launch_up_pair(bsmm_ctx *h, UpPairSched &us, const GroupPtrs &g, void *dw, int N, bsmm_dtype t,
                           int acc, cudaStream_t s, bsmm_dtype dw_t)
{
    using G = UpPairGeo;
    const int C = h->R * 32, K = h->S * 32;
    UpMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int i = 0; i < g.G; ++i) {
        bool ok;
        if (FA) {
            ok = make_map2d(&maps.x[i], g.x[i], t, C, N, 64, G::TK, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, K, N, 64, G::TK, CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            ok = make_map2d(&maps.x[i], g.x[i], t, N, C, G::TK, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map2d(&maps.dy[i], g.dy[i], t, N, K, G::TK, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return BSMM_ERR_CUDA;
    }
    UpParams p;
    p.dw = dw;
    p.table = us.d_table;
    p.status = h->d_status;
    p.N = N;
    p.G = g.G;
    p.accumulate = acc;
    p.dwt = dw_code(dw_t);
    p.nnz = h->nnz;
    if (!set_dw_map(h, maps, p, dw, 32)) return BSMM_ERR_CUDA;
    const int smem = G::SMEM + 1024;
    auto kern = k_tc_updat_pair<FA, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le = launch_pdl(kern, dim3(us.ctas), dim3(kUpThreads), smem, s, true, maps, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int FA, bool BWD, bool BF16>
bsmm_status launch_fbd(bsmm_ctx *h, FbDenseSched &fs, const void *act, const void *w, void *out, int N,
                       bsmm_dtype t, cudaStream_t s)
{
    TcState *st = state(h);
    const int C = h->R * 32, K = h->S * 32;
    const int Fin = BWD ? K : C, Fout = BWD ? C : K;
    CUtensorMap m_act, m_w, m_zero;
    bool ok;
    if (FA) ok = make_map2d(&m_act, act, t, Fin, N, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B);
    else ok = make_map2d(&m_act, act, t, N, Fin, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map2d(&m_w, w, t, 32, (uint64_t)h->nnz * 32, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map2d(&m_zero, st->d_zero, t, 32, kZeroBytes / 64, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    CUtensorMap m_out;
    if (FA) ok = ok && make_map2d(&m_out, out, t, Fout, N, 128, 256, CU_TENSOR_MAP_SWIZZLE_NONE);
    else m_out = m_act;                                  // unused for (C,N) outputs
    if (!ok) return BSMM_ERR_CUDA;
    FbdParams p;
    p.out = out;
    p.stream = fs.d_stream;
    p.off = fs.d_off;
    p.len = fs.d_len;
    p.status = h->d_status;
    p.N = N;
    p.Fout = Fout;
    p.n_tiles = (N + 255) / 256;
    const int smem = 4 * (16384 + 32768) + kFbdSchedWords * 4 + 1024;
    auto kern = k_tc_fbd<FA, BWD, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le =
        launch_pdl(kern, dim3(fs.ngroups * p.n_tiles), dim3(kFbThreads), smem, s, true, m_act, m_w, m_zero, m_out, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int FA, bool BWD, bool BF16>
bsmm_status launch_fbd_pair(bsmm_ctx *h, FbDenseSched &fs, const void *act, const void *w, void *out, int N,
                            bsmm_dtype t, cudaStream_t s)
{
    TcState *st = state(h);
    const int C = h->R * 32, K = h->S * 32;
    const int Fin = BWD ? K : C, Fout = BWD ? C : K;
    CUtensorMap m_act, m_w, m_zero, m_out;
    bool ok;
    // this CTA's half panel: 128 minibatch rows x 64 features, or 64 features x 64 minibatch columns
    if (FA) ok = make_map2d(&m_act, act, t, Fin, N, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    else ok = make_map2d(&m_act, act, t, N, Fin, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map2d(&m_w, w, t, 32, (uint64_t)h->nnz * 32, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map2d(&m_zero, st->d_zero, t, 32, kZeroBytes / 64, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (FA) ok = ok && make_map2d(&m_out, out, t, Fout, N, 128, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    else m_out = m_act;                                  // unused for (C,N) outputs
    if (!ok) return BSMM_ERR_CUDA;
    FbdParams p = {};
    p.out = out;
    p.stream = fs.d_stream;
    p.off = fs.d_off;
    p.len = fs.d_len;
    p.status = h->d_status;
    p.N = N;
    p.Fout = Fout;
    p.n_tiles = (N + 255) / 256;
    const int smem = 6 * (16384 + 16384) + kFbpSchedWords * 4 + 1024;
    auto kern = k_tc_fbd_pair<FA, BWD, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le = launch_pdl(kern, dim3(fs.ngroups * p.n_tiles * 2), dim3(kFbpThreads), smem, s, true, m_act,
                                      m_w, m_zero, m_out, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int FA, bool BWD, bool BF16>
bsmm_status launch_fbd_split(bsmm_ctx *h, FbDenseSched &fs, const void *act, const void *w, void *out, int N,
                             bsmm_dtype t, cudaStream_t s)
{
    TcState *st = state(h);
    const int C = h->R * 32, K = h->S * 32;
    const int Fin = BWD ? K : C, Fout = BWD ? C : K;
    CUtensorMap m_act, m_w, m_zero;
    bool ok;
    if (FA) ok = make_map2d(&m_act, act, t, Fin, N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    else ok = make_map2d(&m_act, act, t, N, Fin, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map2d(&m_w, w, t, 32, (uint64_t)h->nnz * 32, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map2d(&m_zero, st->d_zero, t, 32, kZeroBytes / 64, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return BSMM_ERR_CUDA;
    FbdParams p;
    p.out = out;
    p.stream = fs.d_stream;
    p.off = fs.d_off;
    p.len = fs.d_len;
    p.status = h->d_status;
    p.N = N;
    p.Fout = Fout;
    p.n_tiles = 1;
    const int smem = 8 * (16384 + 8192) + kFbdSchedWords * 4 + 1024;
    auto kern = k_tc_fbd_split<FA, BWD, BF16>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const cudaError_t le =
        launch_pdl(kern, dim3(fs.ngroups * kSplit), dim3(kFbThreads), smem, s, true, m_act, m_w, m_zero, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

// Dense tiles for bs = 32 layouts with at least a quarter of the blocks present and a
// minibatch of more than 128 rows (BSMM_TC_FB=dense / window overrides).  Returns
// BSMM_ERR_UNSUPPORTED when the window kernel should run instead.
template <bool BWD>
bsmm_status fbd_try(bsmm_ctx *h, const void *act, const void *w, void *out, int N, bsmm_dtype t, cudaStream_t s)
{
    if (h->bs != 32 || h->nnz == 0) return BSMM_ERR_UNSUPPORTED;
    const double density = (double)h->nnz / ((double)h->R * h->S);
    bool dense = density >= 0.25 && (N > 128 || N <= 64);
    bool pair = N > 64;                              // CTA-pair kernel unless one 64-row tile
    if (const char *e = getenv("BSMM_TC_FB")) {
        if (!strcmp(e, "window")) dense = false;
        if (!strcmp(e, "dense")) dense = true;
        if (!strcmp(e, "dense1")) dense = true, pair = false;
    }
    if (!dense) return BSMM_ERR_UNSUPPORTED;
    TcState *st = state(h);
    FbDenseSched *fs;
    {
        std::lock_guard<std::mutex> lk(st->mu);
        if (!st->d_zero) {
            if (cudaMalloc(&st->d_zero, kZeroBytes) != cudaSuccess) return BSMM_ERR_OOM;
            if (cudaMemset(st->d_zero, 0, kZeroBytes) != cudaSuccess) return BSMM_ERR_CUDA;
        }
        if (pair) {
            if (!st->fbd[2 + BWD]) st->fbd[2 + BWD] = new FbDenseSched();
            FbDenseSched *fp = st->fbd[2 + BWD];
            if (!fp->built && !fp->too_big && !build_fb_dense_pair(h, *fp, BWD)) return BSMM_ERR_OOM;
            if (!fp->built) pair = false;                // schedule too long: single-CTA tiles
        }
        if (!st->fbd[BWD]) st->fbd[BWD] = new FbDenseSched();
        fs = st->fbd[BWD];
        if (!pair && !fs->built && !fs->too_big && !build_fb_dense(h, *fs, BWD)) return BSMM_ERR_OOM;
        if (pair) fs = st->fbd[2 + BWD];
    }
    if (!fs->built) return BSMM_ERR_UNSUPPORTED;
    const bool bf = t == BSMM_BF16;
    if (N <= 64) {
        // minibatch of one 64-row tile: clusters of kSplit CTAs share each tile
        if (h->fa) return bf ? launch_fbd_split<1, BWD, true>(h, *fs, act, w, out, N, t, s)
                             : launch_fbd_split<1, BWD, false>(h, *fs, act, w, out, N, t, s);
        return bf ? launch_fbd_split<0, BWD, true>(h, *fs, act, w, out, N, t, s)
                  : launch_fbd_split<0, BWD, false>(h, *fs, act, w, out, N, t, s);
    }
    if (pair) {
        if (h->fa) return bf ? launch_fbd_pair<1, BWD, true>(h, *fs, act, w, out, N, t, s)
                             : launch_fbd_pair<1, BWD, false>(h, *fs, act, w, out, N, t, s);
        return bf ? launch_fbd_pair<0, BWD, true>(h, *fs, act, w, out, N, t, s)
                  : launch_fbd_pair<0, BWD, false>(h, *fs, act, w, out, N, t, s);
    }
    if (h->fa) return bf ? launch_fbd<1, BWD, true>(h, *fs, act, w, out, N, t, s)
                         : launch_fbd<1, BWD, false>(h, *fs, act, w, out, N, t, s);
    return bf ? launch_fbd<0, BWD, true>(h, *fs, act, w, out, N, t, s)
              : launch_fbd<0, BWD, false>(h, *fs, act, w, out, N, t, s);
}

// Work of output block o in a window pass: its source blocks (fine blocks for bs 8).
int64_t fb_block_work(const bsmm_ctx *h, bool bwd, int o)
{
    const int f = h->bs == 8 ? 2 : 1;
    int64_t w = 0;
    for (int q = 0; q < f; ++q) {
        const int fine = o * f + q;
        if (bwd && fine < h->R) w += h->h_row_ptr[fine + 1] - h->h_row_ptr[fine];
        if (!bwd && fine < h->S) w += h->h_col_ptr[fine + 1] - h->h_col_ptr[fine];
    }
    return w;
}

// Binned windows: output blocks dealt to one bin per SM (per minibatch tile), heaviest first,
// each to the bin with the least work so far; a bin's blocks are its window's slots.  Used when
// one-block windows give more CTAs than SMs but fewer than two per SM and the blocks' work is
// uneven (the heaviest at least 1.5 x the mean): the heaviest blocks then run alone on an SM
// with the deepest pipeline, and the light ones share bins instead of sharing those SMs.  With
// even work (every block the same number of sources) two CTAs per SM measured faster.
bool fb_binned(const bsmm_ctx *h, bool bwd, int n_tiles)
{
    if (h->tc_bins == 0) return false;
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    const int nbins = std::max(1, h->sm_count / n_tiles);
    if (Fslots <= nbins || (Fslots + nbins - 1) / nbins * bse > 256) return false;
    if (h->tc_bins == 1) return true;
    if (Fslots >= 2 * nbins) return false;
    int64_t total = 0, most = 0;
    for (int o = 0; o < Fslots; ++o) {
        const int64_t w = fb_block_work(h, bwd, o);
        total += w;
        most = std::max(most, w);
    }
    return 2 * most * Fslots >= 3 * total;
}

std::vector<std::vector<int>> fb_bins(const bsmm_ctx *h, bool bwd, int n_tiles)
{
    int Fslots, Fsrc, bse;
    fb_shape(h, bwd, Fslots, Fsrc, bse);
    const int nbins = std::min(Fslots, std::max(1, h->sm_count / n_tiles));
    const int wmax = std::min(256 / bse, 2 * ((Fslots + nbins - 1) / nbins));
    std::vector<int64_t> work(Fslots, 0);
    for (int o = 0; o < Fslots; ++o) work[o] = fb_block_work(h, bwd, o);
    std::vector<int> idx(Fslots);
    for (int o = 0; o < Fslots; ++o) idx[o] = o;
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return work[a] > work[b]; });
    std::vector<std::vector<int>> bins(nbins);
    std::vector<int64_t> load(nbins, 0);
    for (int o : idx) {
        int best = -1;
        for (int b = 0; b < nbins; ++b)
            if ((int)bins[b].size() < wmax && (best < 0 || load[b] < load[best])) best = b;
        bins[best].push_back(o);
        load[best] += work[o] + 2;
    }
    for (auto &b : bins) std::sort(b.begin(), b.end());
    return bins;
}

// Window kernel tile height for N > 64: 64-row tiles halve each CTA's activation bytes and
// double the units the hardware scheduler can balance over the SMs.
bool fb_rows64(const bsmm_ctx *h, int N)
{
    if (h->tc_rows == 64) return true;
    if (h->tc_rows == 128) return false;
    (void)N;
    return false;
}

template <bool BWD>
bsmm_status fb_dispatch(bsmm_ctx *h, const void *act, const void *w, void *out, int N, bsmm_dtype t, cudaStream_t s)
{
    TcState *st = state(h);
    const bool rows64 = N > 64 && fb_rows64(h, N);
    const int a_ops = (h->fa || N <= 64 || rows64) ? 1 : 2, b_ops = h->bs == 8 ? 4 : 1;
    const int wl_max = h->bs == 32 ? 3 : 4;
    const int n_tiles = rows64 ? (N + 63) / 64 : (N + 127) / 128;
    int wl = h->tc_wlog >= 0 ? std::min(h->tc_wlog, wl_max) : choose_wlog(h, BWD, n_tiles);
    bool binned = wl == 0 && fb_binned(h, BWD, n_tiles);
    FbSched *fs = nullptr;
    FbStages geo{};
    {
        std::lock_guard<std::mutex> lk(st->mu);
        if (!st->d_zero) {
            if (cudaMalloc(&st->d_zero, kZeroBytes) != cudaSuccess) return BSMM_ERR_OOM;
            if (cudaMemset(st->d_zero, 0, kZeroBytes) != cudaSuccess) return BSMM_ERR_CUDA;
        }
        // Shrink the window until its schedule stream fits the shared-memory budget.
        for (; wl >= 0; --wl) {
            int Fslots, Fsrc, bse;
            fb_shape(h, BWD, Fslots, Fsrc, bse);
            std::vector<std::vector<int>> bins;
            if (binned) bins = fb_bins(h, BWD, n_tiles);
            int W = std::min(1 << wl, Fslots), nwin = (Fslots + W - 1) / W;
            if (binned) {
                W = 0;
                for (const auto &b : bins) W = std::max(W, (int)b.size());
                nwin = (int)bins.size();
            }
            geo = choose_stages(h, N, (int64_t)nwin * n_tiles, W, rows64);
            const uint64_t key = (uint64_t)BWD | ((uint64_t)wl << 1) | ((uint64_t)geo.e_slots << 8) |
                                 ((uint64_t)geo.r_slots << 16) | ((uint64_t)a_ops << 24) |
                                 ((uint64_t)binned << 32);
            FbSched &c = st->fb[key];
            if (!c.built && !c.too_big &&
                !build_fb(h, c, BWD, 1 << wl, geo.e_slots, geo.r_slots, a_ops, b_ops, kSchedWords,
                          binned ? &bins : nullptr))
                return BSMM_ERR_OOM;
            if (c.built) {
                fs = &c;
                break;
            }
            if (binned) {                      // a bin's stream is too long: plain windows instead
                binned = false;
                ++wl;
            }
        }
    }
    if (!fs) return BSMM_ERR_UNSUPPORTED;     // caller falls back to the SIMT kernels
    const bool bf = t == BSMM_BF16;
#define FB_CASE(BS_, FA_)                                                                                   \
    if (h->bs == BS_ && h->fa == FA_)                                                                       \
        return bf ? launch_fb<BS_, FA_, BWD, true>(h, *fs, geo, act, w, out, N, t, s)                      \
                  : launch_fb<BS_, FA_, BWD, false>(h, *fs, geo, act, w, out, N, t, s);
    FB_CASE(32, 1)
    FB_CASE(32, 0)
    FB_CASE(16, 1)
    FB_CASE(16, 0)
    FB_CASE(8, 1)
    FB_CASE(8, 0)
#undef FB_CASE
    return BSMM_ERR_UNSUPPORTED;
}

// Self-test of the bounded waits: one warp waits on an mbarrier that nothing arrives on.
__global__ void k_wait_selftest(int32_t *status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, limit_ns);
}

// Launch-cost self-test: an empty kernel with the launch shape of the window kernel.  The
// TENSOR_MEMORY form allocates and frees 32 columns per CTA; a kernel that contains tcgen05
// instructions at all pays a larger fixed launch cost, which this form measures.
template <bool TENSOR_MEMORY>
__global__ void __launch_bounds__(kFbThreads, 1) k_empty_selftest(int32_t *status)
{
    __shared__ uint32_t tmem_base;
    if (TENSOR_MEMORY) {
        if (threadIdx.x < 32) tmem_alloc(&tmem_base, 32);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    pdl_launch_dependents();
    pdl_wait();
    if (TENSOR_MEMORY) {
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x < 32) tmem_dealloc(tmem_base, 32);
    }
    (void)status;
}

} // namespace

bsmm_status launch_wait_selftest(bsmm_ctx *h, uint64_t limit_ns, cudaStream_t s)
{
    k_wait_selftest<<<1, 32, 0, s>>>(h->d_status, limit_ns);
    g_bsmm_launches += 1;
    return cudaGetLastError() == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

bsmm_status launch_empty_selftest(bsmm_ctx *h, int ctas, bool tensor_memory, cudaStream_t s)
{
    const cudaError_t le = tensor_memory
                               ? launch_pdl(k_empty_selftest<true>, dim3(ctas), dim3(kFbThreads), 0, s, true, h->d_status)
                               : launch_pdl(k_empty_selftest<false>, dim3(ctas), dim3(kFbThreads), 0, s, true, h->d_status);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

bool tc_supported(bsmm_ctx *h, bsmm_dtype t)
{
    if (t != BSMM_F16 && t != BSMM_BF16) return false;
    if (!encode_fn()) return false;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
    return major == 10 && minor == 3;
}

// fprop/bprop dispatch: the dense-tile kernels (bs = 32, at least a quarter of the layout
// present); the sparse-window kernel for block sizes 16 and 8 (k_tc_sp, bsmm_sp.cu); else the
// window kernel, which is faster for sparse bs = 32 layouts at a minibatch of 128 (fewer, larger
// blocks per source).  BSMM_TC_FB = window | sp | dense | dense1 forces a family.
template <bool BWD>
bsmm_status fb_tc(bsmm_ctx *h, const void *act, const void *w, void *out, int N, bsmm_dtype t, cudaStream_t s)
{
    const char *e = getenv("BSMM_TC_FB");
    const bool force_window = e && !strcmp(e, "window");
    const bool force_sp = e && !strcmp(e, "sp");
    if (!force_window && !force_sp) {
        const bsmm_status st = fbd_try<BWD>(h, act, w, out, N, t, s);
        if (st != BSMM_ERR_UNSUPPORTED) return st;
    }
    if (force_sp || (!force_window && h->bs != 32)) {
        const bsmm_status st = sp_fb(h, BWD, act, w, out, N, t, s);
        if (st != BSMM_ERR_UNSUPPORTED) return st;
    }
    return fb_dispatch<BWD>(h, act, w, out, N, t, s);
}

bsmm_status tc_fprop(bsmm_ctx *h, const void *x, const void *w, void *y, int N, bsmm_dtype t, cudaStream_t s)
{
    return fb_tc<false>(h, x, w, y, N, t, s);
}

bsmm_status tc_bprop(bsmm_ctx *h, const void *dy, const void *w, void *dx, int N, bsmm_dtype t, cudaStream_t s)
{
    return fb_tc<true>(h, dy, w, dx, N, t, s);
}

bsmm_status tc_updat(bsmm_ctx *h, const GroupPtrs &g, void *dw, int N, bsmm_dtype t, bsmm_dtype dw_t,
                     int accumulate, cudaStream_t s)
{
    TcState *st = state(h);
    const bool bf = t == BSMM_BF16;
    // Dense 128 x 256 tiles when bs = 32, at least a quarter of the layout is present and
    // the minibatch spans two or more 64-row stages (BSMM_TC_UPDAT=stack / dense overrides).
    const double density = (double)h->nnz / ((double)h->R * h->S);
    bool dense = h->bs == 32 && density >= 0.25 && N * g.G > 64 && h->nnz < (1 << 24);
    bool pair = true;                                // CTA-pair tiles unless the table does not fit
    if (const char *e = getenv("BSMM_TC_UPDAT")) {
        if (!strcmp(e, "stack")) dense = false;
        if (!strcmp(e, "dense")) dense = h->bs == 32 && h->nnz < (1 << 24);
        if (!strcmp(e, "dense1")) dense = h->bs == 32 && h->nnz < (1 << 24), pair = false;
    }
    if (dense && pair) {
        {
            std::lock_guard<std::mutex> lk(st->mu);
            if (!st->upp) st->upp = new UpPairSched();
            if (!st->upp->built && !st->upp->too_big && !build_up_pair(h, *st->upp)) return BSMM_ERR_OOM;
        }
        if (st->upp->built) {
            if (st->upp->ctas == 0) return BSMM_OK;
            if (h->fa) return bf ? launch_up_pair<1, true>(h, *st->upp, g, dw, N, t, accumulate, s, dw_t)
                                 : launch_up_pair<1, false>(h, *st->upp, g, dw, N, t, accumulate, s, dw_t);
            return bf ? launch_up_pair<0, true>(h, *st->upp, g, dw, N, t, accumulate, s, dw_t)
                      : launch_up_pair<0, false>(h, *st->upp, g, dw, N, t, accumulate, s, dw_t);
        }
    }
    if (dense) {
        {
            std::lock_guard<std::mutex> lk(st->mu);
            if (!st->upd) st->upd = new UpDenseSched();
            if (!st->upd->built && !build_up_dense(h, *st->upd)) return BSMM_ERR_OOM;
        }
        if (st->upd->ctas == 0) return BSMM_OK;
        if (h->fa) return bf ? launch_up_dense<1, true>(h, *st->upd, g, dw, N, t, accumulate, s, dw_t)
                             : launch_up_dense<1, false>(h, *st->upd, g, dw, N, t, accumulate, s, dw_t);
        return bf ? launch_up_dense<0, true>(h, *st->upd, g, dw, N, t, accumulate, s, dw_t)
                  : launch_up_dense<0, false>(h, *st->upd, g, dw, N, t, accumulate, s, dw_t);
    }
    {
        std::lock_guard<std::mutex> lk(st->mu);
        if (!st->up.built && !build_up(h, st->up)) return BSMM_ERR_OOM;
    }
    if (st->up.ctas == 0) return BSMM_OK;
#define UP_CASE(BS_, FA_)                                                                         \
    if (h->bs == BS_ && h->fa == FA_)                                                             \
        return bf ? launch_up<BS_, FA_, true>(h, st->up, g, dw, N, t, accumulate, s, dw_t)       \
                  : launch_up<BS_, FA_, false>(h, st->up, g, dw, N, t, accumulate, s, dw_t);
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
    for (auto &kv : st->fb) {
        FbSched &f = kv.second;
        cudaFree(f.d_stream);
        cudaFree(f.d_win_desc);
        cudaFree(f.d_win_out);
    }
    cudaFree(st->up.d_table);
    if (st->upd) {
        cudaFree(st->upd->d_table);
        delete st->upd;
    }
    if (st->upp) {
        cudaFree(st->upp->d_table);
        delete st->upp;
    }
    for (auto *f : st->fbd)
        if (f) {
            cudaFree(f->d_stream);
            cudaFree(f->d_off);
            cudaFree(f->d_len);
            delete f;
        }
    cudaFree(st->d_zero);
    delete st;
    h->tc = nullptr;
}

// ---------------------------------------------------------------------------------------
// Allocation-free weight gradient
// ---------------------------------------------------------------------------------------
// Some callers cannot call cudaMalloc: code that runs under a framework's memory budget or
// caching allocator (where a raw driver allocation would bypass it, fragment it or fail at
// the memory limit), and latency-critical loops where an allocation's cost or failure is
// not acceptable.  bsmm_updat_noalloc serves them: it runs the stacked weight-gradient
// kernel with its unit table in the fixed device array below instead of a table the
// handle would allocate.  The array is a module global: every GPU that loads this library
// holds its 4 MB until the process exits.

namespace {

constexpr int kNoAllocTableWords = 1 << 20;          // 4 MB: at most this many table words
__device__ __align__(256) int32_t g_noalloc_table[kNoAllocTableWords];

int32_t g_noalloc_host[kNoAllocTableWords];          // host staging copy (static, not allocated)
std::mutex g_noalloc_mu;
int32_t *g_noalloc_dev_ptr[64] = {nullptr};          // device address of the array, per device

// Builds the stacked-updat unit tables into g_noalloc_host (same layout as build_up).
// Returns the number of CTAs, 0 for an empty layout, or -1 if the tables do not fit.
int noalloc_build(const bsmm_ctx *h)
{
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;
    const int Rc = (h->R + f - 1) / f, Sc = (h->S + f - 1) / f;
    const int MS = coarse ? 8 : 128 / h->bs;
    BidLookup bid{h};
    // count units first
    int64_t nunits = 0;
    for (int kc = 0; kc < Sc; ++kc) {
        int n = 0;
        for (int cc = 0; cc < Rc; ++cc) {
            bool any = false;
            for (int cs = 0; cs < f; ++cs)
                for (int ks = 0; ks < f; ++ks) any |= bid(cc * f + cs, kc * f + ks) >= 0;
            n += any;
        }
        nunits += (n + MS - 1) / MS;
    }
    if (nunits == 0) return 0;
    int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(nunits, 2 * std::max(1, h->sm_count)));
    ctas = std::max<int64_t>(ctas, (nunits + kUnitsPerCta - 1) / kUnitsPerCta);
    if (ctas * kTableWords > kNoAllocTableWords) return -1;
    std::fill(g_noalloc_host, g_noalloc_host + ctas * kTableWords, 0);
    int64_t u = 0;
    for (int kc = 0; kc < Sc; ++kc) {
        int32_t *cur = nullptr;
        int m = 0;
        for (int cc = 0; cc < Rc; ++cc) {
            int32_t ids[4];
            bool any = false;
            for (int cs = 0; cs < f; ++cs)
                for (int ks = 0; ks < f; ++ks) {
                    ids[cs * 2 + ks] = bid(cc * f + cs, kc * f + ks);
                    any |= ids[cs * 2 + ks] >= 0;
                }
            if (!any) continue;
            if (!cur || m == MS) {                    // start a new unit in CTA u % ctas
                int32_t *t = g_noalloc_host + (u % ctas) * kTableWords;
                const int i = (int)(u / ctas);
                t[0] = i + 1;
                cur = t + 4 + i * kUnitWords;
                cur[0] = kc;
                m = 0;
                ++u;
            }
            int32_t *r = cur + 2 + 5 * m;
            r[0] = cc;
            for (int q = 0; q < 4; ++q) r[1 + q] = ids[q];
            cur[1] = ++m;
        }
    }
    return (int)ctas;
}

} // namespace

extern "C" bsmm_status bsmm_updat_noalloc(bsmm_t h, const void *x, const void *dy, float *dw, int N, bsmm_dtype t,
                                          int accumulate, void *stream)
{
    if (!h || N < 0) return BSMM_ERR_INVALID;
    if (t != BSMM_F16 && t != BSMM_BF16) return BSMM_ERR_UNSUPPORTED;
    if (h->fa == 0 && ((int64_t)N * 2) % 16 != 0) return BSMM_ERR_ALIGN;
    if (h->nnz == 0) return BSMM_OK;
    if (!x || !dy || !dw) return BSMM_ERR_INVALID;
    if (((uintptr_t)x | (uintptr_t)dy | (uintptr_t)dw) & 15u) return BSMM_ERR_ALIGN;
    if (h->device < 0 || h->device >= 64) return BSMM_ERR_UNSUPPORTED;
    if (cudaSetDevice(h->device) != cudaSuccess) return BSMM_ERR_CUDA;
    if (!tc_supported(h, t)) return BSMM_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    // The table reaches the device by a copy from one shared host buffer that the next call
    // overwrites; a graph captured around this call would replay that copy later and read
    // another call's table.  Refuse before anything is enqueued.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return BSMM_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return BSMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_dev_ptr[h->device]) {
        // One-time set-up on this device: the array's device address (a host-side symbol
        // is not a device pointer).
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_table) != cudaSuccess || !ptr) return BSMM_ERR_CUDA;
        g_noalloc_dev_ptr[h->device] = static_cast<int32_t *>(ptr);
    }
    int32_t *table = g_noalloc_dev_ptr[h->device];
    if (N == 0) {
        if (accumulate) return BSMM_OK;
        return cudaMemsetAsync(dw, 0, (size_t)h->nnz * h->bs * h->bs * sizeof(float), s) == cudaSuccess
                   ? BSMM_OK
                   : BSMM_ERR_CUDA;
    }
    const int ctas = noalloc_build(h);
    if (ctas < 0) return BSMM_ERR_UNSUPPORTED;       // layout needs more than the fixed 4 MB table
    if (ctas == 0) return BSMM_OK;
    // Pageable copy: returns once the host buffer has been staged, ordered before the kernel,
    // which is launched without programmatic dependent launch (nothing to overlap with a copy).
    if (cudaMemcpyAsync(table, g_noalloc_host, (size_t)ctas * kTableWords * sizeof(int32_t), cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
        return BSMM_ERR_CUDA;
    UpSched us;
    us.ctas = ctas;
    us.d_table = table;
    us.built = true;
    GroupPtrs g{};
    g.x[0] = x;
    g.dy[0] = dy;
    g.G = 1;
    const bool bf = t == BSMM_BF16;
    const int acc = accumulate ? 1 : 0;
    bsmm_status st = BSMM_ERR_UNSUPPORTED;
#define NA_CASE(BS_, FA_)                                                                      \
    if (h->bs == BS_ && h->fa == FA_)                                                          \
        st = bf ? launch_up<BS_, FA_, true>(h, us, g, dw, N, t, acc, s, BSMM_F32, false)       \
                : launch_up<BS_, FA_, false>(h, us, g, dw, N, t, acc, s, BSMM_F32, false);
    NA_CASE(32, 1)
    NA_CASE(32, 0)
    NA_CASE(16, 1)
    NA_CASE(16, 0)
    NA_CASE(8, 1)
    NA_CASE(8, 0)
#undef NA_CASE
    us.d_table = nullptr;                            // the array is not the handle's to free
    return st;
}
