// Sparse-window fprop / bprop (k_tc_sp): a CTA accumulates a window of output blocks in tensor
// memory and gathers exactly the weight blocks and activation panels the window needs.
//
// The passes are those of BlocksparseMatMul in the blocksparse README ("API Documentation:
// blocksparse.matmul"): fprop y = x.W (__call__) and bprop dx = dy.W^T, for block sizes 32,
// 16 and 8 and both activation layouts (feature_axis 1: (N, F), 0: (F, N)).
//
// A CTA owns a window of W output blocks for a tile of 128 minibatch rows and accumulates
// D[128 rows][W * BSE] in tensor memory.  It walks the sources (input block rows for fprop,
// output block columns for bprop) with a block in the window, in increasing order; per source the
// activation panel (128 rows x BSE features) is staged once in shared memory and each present
// block of the source issues D[:, slot] += panel . block (M = 128, N = BSE, K = BSE in steps of
// 16).  Absent blocks cost nothing.
//
// Block size 8 runs on 16 x 16 coarse blocks: two adjacent source block rows are concatenated
// along the reduction axis into one K = 16 step (their 8-feature panels form one 16-feature panel,
// shared by every output block of the window), and two adjacent output blocks form N = 16; absent
// 8 x 8 sub-blocks are zero-filled in shared memory.
//
// Issue rate.  On GB300 one issuing thread sustains roughly one instruction per 3 to 10 clocks,
// so the per-MMA instruction count decides the rate as much as the MMA itself (39 clocks for
// M128 x N16 x K16 with both operands in shared memory).  Four MMA warps therefore issue in
// parallel: warp q owns the output slots s with s % 4 == q, so every accumulator still receives
// its MMAs from one thread in schedule order (deterministic sums).  Per chunk each MMA warp reads
// a ready-made list of at most 8 words (accumulator column, panel, block, accumulate flag) with
// two vector loads and issues from registers, predicated, without branches.  The loaders
// likewise read a chunk's schedule words into registers before issuing its copies; two loader
// warps share each chunk (panels 0-3 and blocks 0-15, panels 4-7 and blocks 16-31), which halves
// the time to issue a stage's copies, the limit on how fast stages refill.
//
// Loads.  Weight blocks are gathered with cp.async, 16 bytes per lane, straight into the canonical
// no-swizzle operand layout: one warp instruction moves one 512-byte block, about 50 bytes per
// clock per SM for 512-byte blocks on GB300, where TMA boxes of the same size reach 8.  (N, F)
// activation panels are gathered the same way from their rows; (F, N) activations are first
// rearranged by k_sp_panelize into contiguous panels of the operand layout (a transpose).  Every
// stage's copies complete on one mbarrier.
//
// Split over sources.  A window may be split between the two CTAs of a cluster (each takes a
// contiguous half of the window's sources); their fp32 partial tiles are summed in distributed
// shared memory in a fixed order, so results do not depend on the split.
//
// Checks.  Block ids and sources read from the schedule are checked against the layout before
// any global access (a failed check records BSMM_ERR_BOUNDS and the copy is zero-filled);
// accumulator columns are masked to the allocation.  Every wait is bounded (BSMM_ERR_TIMEOUT).
#include "bsmm_internal.cuh"
#include "tc_common.cuh"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

using namespace tc;

namespace {

constexpr int kSpProducers = 4;                 // chunk c is loaded by producer slot c % 4 ...
constexpr int kSpLoaders = 2 * kSpProducers;    // ... whose two warps s and s + 4 (warps 0-7) split it
constexpr int kSpMmaWarps = 4;                  // warps 8-11 issue MMAs (warp 8 allocates tensor memory)
constexpr int kSpThreads = 32 * (kSpLoaders + kSpMmaWarps);     // all twelve store the outputs
constexpr int kSpEpiGroups = kSpThreads / 128;  // warp groups sharing the epilogue
constexpr int kSpMaxStages = 16;
constexpr int kSpSchedWords = 6144;             // per-unit schedule budget (24 KB)
constexpr int kSpSmemBudget = 226 * 1024;       // dynamic shared memory limit of one CTA
constexpr int kSpHead = 4;                      // stream header words
constexpr int kSpList = 8;                      // MMA list words per MMA warp per chunk
constexpr int kSpChunkHead = 4 + kSpMmaWarps * kSpList;   // chunk prefix words
constexpr uint32_t kIdMask = (1u << 27) - 1;    // record: (slot << 27) | block id

// Runtime stage geometry of a launch (host-chosen; the kernel checks it).
struct SpGeo {
    int W;          // output slots per window
    int split;      // CTAs per window (1 or 2, a cluster)
    int E, R;       // entries (sources) and records (blocks) per chunk at most
    int stages;     // a multiple of kSpProducers
    int stage_bytes, b_off;
};

struct SpParams {
    const void *act;            // x (fprop) / dy (bprop); for feature_axis 0 the panelised copy
    const void *w;
    void *out;
    const uint32_t *stream;
    const int4 *desc;           // per (launch position, part): window, stream offset, length
    int32_t *status;
    int N, Fin, Fout, Fsrc, Fslots, ntiles;
    int64_t nnz;
    int bf16;
    SpGeo g;
};

__device__ __forceinline__ uint16_t sp_cvt(float a, int bf16)
{
    if (bf16) {
        __nv_bfloat16 v = __float2bfloat16_rn(a);
        return *reinterpret_cast<uint16_t *>(&v);
    }
    __half v = __float2half_rn(a);
    return *reinterpret_cast<uint16_t *>(&v);
}

__device__ __forceinline__ uint32_t sp_pack(float a, float b, int bf16)
{
    return (uint32_t)sp_cvt(a, bf16) | ((uint32_t)sp_cvt(b, bf16) << 16);
}

__device__ __forceinline__ void sp_flag(int32_t *status, int32_t code) { atomicExch(status, code); }

// D[tmem] (+)= A[smem] . B[smem] issued when `issue` is set; the descriptors are given as their
// low words (start address and leading byte offset) and a common high word.
__device__ __forceinline__ void sp_mma(uint32_t issue, uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, q;\n\t.reg .b64 da, db;\n\t"
                 "setp.ne.b32 p, %5, 0;\n\tsetp.ne.b32 q, %6, 0;\n\t"
                 "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
                 "@q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d),
                 "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

// fprop (BWD = false) / bprop (BWD = true).  BS = block size; bs 8 runs on 16 x 16 coarse blocks.
template <int BS, int FA, bool BWD>
__global__ void __launch_bounds__(kSpThreads, 1) k_tc_sp(const SpParams p)
{
    constexpr int BSE = BS == 8 ? 16 : BS;          // (coarse) block edge
    constexpr bool COARSE = BS == 8;
    constexpr int RW = COARSE ? 4 : 1;              // schedule words per record
    constexpr int PANEL = 128 * BSE * 2;            // activation panel: 128 rows x BSE features
    constexpr int BSLOT = BSE * BSE * 2;            // one (coarse) weight block
    constexpr uint32_t SBO = BSE * 16;              // 8-row (M or N) group stride of the operands
    constexpr uint32_t LBO = 128;                   // K-direction core-matrix stride
    constexpr int KSTEPS = BSE / 16;
    constexpr int CPR = BSE / 8;                    // 16-byte chunks per panel row
    constexpr int WCH = COARSE ? 1 : BS * BS / 256; // 16-byte chunks of a block per lane
    const uint32_t idesc = idesc_f16(128, BSE, p.bf16 != 0, false, !BWD);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SpGeo g = p.g;
    uint32_t *sched = reinterpret_cast<uint32_t *>(smem + g.stages * g.stage_bytes);
    __shared__ __align__(8) uint64_t full[kSpMaxStages], empty[kSpMaxStages], acc_full, sched_full;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int aborted;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int split = g.split;
    const int part = split > 1 ? (int)cluster_ctarank() : 0;
    const int unit = blockIdx.x / split;
    const int4 desc = __ldg(p.desc + (unit / p.ntiles) * split + part);
    const int win = desc.x;
    const int tile = unit % p.ntiles;
    const int n0 = tile * 128;

    if (g.stages < kSpProducers || g.stages > kSpMaxStages || g.stages % kSpProducers != 0 || g.W < 1 ||
        g.W > 32 || g.W * BSE > 512 || g.E < 1 || g.E > 8 || g.R < 1 || g.R > 32) {
        // the host guarantees the geometry; every CTA of a cluster takes this branch alike
        if (threadIdx.x == 0) sp_flag(p.status, BSMM_ERR_INVALID);
        return;
    }

    if (threadIdx.x == 0) {
        aborted = 0;
        for (int i = 0; i < g.stages; ++i) {
            mbar_init(&full[i], 1 + 64);        // the first loading warp's lane 0 + 2 x 32 cp.async arrivals
            mbar_init(&empty[i], kSpMmaWarps);  // one commit per MMA warp
        }
        mbar_init(&acc_full, kSpMmaWarps);
        mbar_init(&sched_full, 1);
        fence_barrier_init();
    }
    if (warp == kSpLoaders) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // Every CTA holds its tensor memory before a dependent kernel may start, so a dependent CTA
    // that waits for it in tcgen05.alloc waits only on CTAs that will finish.
    pdl_launch_dependents();
    if (warp == 0 && lane == 0) {
        const int len = desc.z;
        mbar_arrive_expect_tx(&sched_full, (uint32_t)len * 4u);
        bulk_load(sched, p.stream + desc.y, (uint32_t)len * 4u, &sched_full, policy_evict_last());
    }
    pdl_wait();
    const bool sched_ok = mbar_wait_warp(&sched_full, 0, p.status, 64);
    if (!sched_ok && lane == 0) aborted = 1;
    __syncwarp();

    const uint16_t *act = static_cast<const uint16_t *>(p.act);
    const uint16_t *wts = static_cast<const uint16_t *>(p.w);

    if (warp < kSpLoaders) {
        // ---------------- loads: warps s and s + 4 fill chunks s, s+4, ...; chunk c uses stage
        // c % stages; warp s loads panels 0-3 and blocks 0-15 of the chunk, warp s + 4 the rest ----
        const int slot = warp % kSpProducers, sub = warp / kSpProducers;
        // Lane-constant offsets of this lane's 16-byte chunks of a weight block: fprop B[K = i][N = j]
        // (MN-major), bprop B[K = j][N = i] (K-major); for bs 8 the lane's 8 x 8 sub-block row.
        uint32_t w_dst[WCH], w_src[WCH];
        if (!COARSE) {
#pragma unroll
            for (int q = 0; q < WCH; ++q) {
                const int ci = q * 32 + lane, i = ci / (BS / 8), h = ci % (BS / 8);
                w_dst[q] = BWD ? (i >> 3) * SBO + h * LBO + (i & 7) * 16 : (i >> 3) * LBO + h * SBO + (i & 7) * 16;
                w_src[q] = i * BS + h * 8;
            }
        } else {
            const int sub = lane >> 3, i = lane & 7, cs = sub >> 1, ks = sub & 1;
            w_dst[0] = BWD ? cs * SBO + ks * LBO + i * 16 : cs * LBO + ks * SBO + i * 16;
            w_src[0] = i * 8;
        }
        const uint32_t nnz32 = (uint32_t)p.nnz;
        int chunk = 0;
        for (int pos = kSpHead; !aborted; ++chunk) {
            const uint32_t hdr = sched[pos];
            if (hdr == 0) break;
            const int ne = (int)(hdr >> 16), nr = (int)(hdr & 0xFFFFu);
            const int next = (pos + kSpChunkHead + ne + nr * RW + 3) & ~3;
            if (chunk % kSpProducers != slot) {
                pos = next;
                continue;
            }
            const int st = chunk % g.stages;
            if (lane == 0) {
                if (chunk >= g.stages && !mbar_wait(&empty[st], ((chunk / g.stages) - 1) & 1, p.status))
                    aborted = 1;
                else if (sub == 0)
                    mbar_arrive(&full[st]);
            }
            __syncwarp();
            if (aborted) break;
            uint8_t *stage = smem + st * g.stage_bytes;
            // the chunk's schedule words into registers first, so no copy waits on a load
            const uint32_t *ent = sched + pos + kSpChunkHead;
            const uint32_t *rec = ent + ne;
            const int e0 = sub * 4, r0 = sub * 16;                  // this warp's panels and blocks
            uint32_t srcw[4], rw[16];
#pragma unroll
            for (int e = 0; e < 4; ++e) srcw[e] = e0 + e < ne ? ent[e0 + e] : 0u;
#pragma unroll
            for (int r = 0; r < 16; ++r) rw[r] = r0 + r < nr ? rec[COARSE ? (r0 + r) * 4 + (lane >> 3) : r0 + r] : 0u;
            bool bad = false;
            // activation panels: entry e into panel slot e
#pragma unroll
            for (int ee = 0; ee < 4; ++ee) {
                const int e = e0 + ee;
                const uint32_t on = e < ne ? 1u : 0u;
                uint32_t src = srcw[ee] >> 8;
                const bool sbad = on && src >= (uint32_t)p.Fsrc;
                bad |= sbad;
                src = sbad ? 0u : src;
                if (!FA) {
                    // the panel is contiguous and already in the operand layout
                    const uint16_t *pan = act + ((size_t)tile * p.Fsrc + src) * (PANEL / 2);
#pragma unroll
                    for (int q = 0; q < PANEL / 512; ++q) {
                        const int ci = q * 32 + lane;
                        cp_async16_if(on, stage + e * PANEL + ci * 16, pan + ci * 8, sbad ? 0u : 16u);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4 * CPR; ++q) {
                        const int ci = q * 32 + lane;           // chunk (row r, 8 features h)
                        const int r = ci / CPR, h = ci % CPR;
                        const int n = n0 + r, f = (int)src * BSE + h * 8;
                        const bool ok = !sbad && n < p.N && f < p.Fin;
                        cp_async16_if(on, stage + e * PANEL + (r >> 3) * SBO + h * LBO + (r & 7) * 16,
                                      ok ? act + (size_t)n * p.Fin + f : act, ok ? 16u : 0u);
                    }
                }
            }
            // weight blocks into record slots, rearranged into the operand layout
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = r0 + rr;
                const uint32_t on = r < nr ? 1u : 0u;
                uint8_t *dst = stage + g.b_off + r * BSLOT;
                const uint32_t v = rw[rr] & kIdMask;
                if (!COARSE) {
                    const bool ok = v < nnz32;
                    bad |= on && !ok;
#pragma unroll
                    for (int q = 0; q < WCH; ++q)
                        cp_async16_if(on, dst + w_dst[q], wts + (size_t)(ok ? v : 0u) * (BS * BS) + w_src[q],
                                      ok ? 16u : 0u);
                } else {
                    // (block id + 1) of the lane's 8 x 8 sub-block, 0 when absent
                    const bool ok = v != 0 && v <= nnz32;
                    bad |= on && v > nnz32;
                    cp_async16_if(on, dst + w_dst[0], wts + (size_t)(ok ? v - 1 : 0u) * 64 + w_src[0], ok ? 16u : 0u);
                }
            }
            cp_async_mbar_arrive(&full[st]);
            if (__any_sync(0xffffffffu, bad) && lane == 0) sp_flag(p.status, BSMM_ERR_BOUNDS);
            pos = next;
        }
        cp_async_wait_all();                                    // no copy outlives the CTA
        __syncwarp();
    } else {
        // ---------------- MMA warps: warp 8 + q issues the MMAs of the slots s with s % 4 == q --------
        // List word: accumulate flag << 31 | block (record) index << 16 | panel (entry) << 12 |
        // accumulator column.
        const int q = warp - kSpLoaders;
        const uint32_t leader = lane == 0 ? 1u : 0u;
        const uint64_t desc0 = sdesc(smem_u32(smem), LBO, SBO, SW_NONE);
        const uint32_t dlo = (uint32_t)desc0, dhi = (uint32_t)(desc0 >> 32);
        int chunk = 0;
        for (int pos = kSpHead; !aborted; ++chunk) {
            const uint4 h0 = *reinterpret_cast<const uint4 *>(sched + pos);
            if (h0.x == 0) break;
            const uint4 l0 = *reinterpret_cast<const uint4 *>(sched + pos + 4 + q * kSpList);
            const uint4 l1 = *reinterpret_cast<const uint4 *>(sched + pos + 8 + q * kSpList);
            const uint32_t lw[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
            const uint32_t cnt = (h0.y >> (q * 8)) & 0xFFu;
            const int ne = (int)(h0.x >> 16), nr = (int)(h0.x & 0xFFFFu);
            const int st = chunk % g.stages;
            uint32_t got = 1;
            if (leader) got = mbar_wait(&full[st], (chunk / g.stages) & 1, p.status) ? 1u : 0u;
            if (__shfl_sync(0xffffffffu, got, 0) == 0) {
                if (leader) aborted = 1;
                break;
            }
            tc_fence_after();
            fence_proxy_async_smem();                           // cp.async (generic proxy) writes -> MMA reads
            const uint32_t slo = dlo + ((uint32_t)(st * g.stage_bytes) >> 4);
            const uint32_t blo = slo + ((uint32_t)g.b_off >> 4);
#pragma unroll
            for (int j = 0; j < kSpList; ++j) {
                const uint32_t w = lw[j];
                const uint32_t go = leader & ((uint32_t)j < cnt ? 1u : 0u);
                const uint32_t d = tmem + (w & 0x1FFu);
                const uint32_t a_lo = slo + ((w >> 12) & 7u) * (uint32_t)(PANEL >> 4);
                const uint32_t b_lo = blo + ((w >> 16) & 31u) * (uint32_t)(BSLOT >> 4);
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks)
                    sp_mma(go, d, a_lo + ks * (2 * LBO >> 4), b_lo + ks * (2 * LBO >> 4), dhi, idesc,
                           ks > 0 ? 1u : (w >> 31));
            }
            mma_commit_if(leader, &empty[st]);
            pos = (pos + kSpChunkHead + ne + nr * RW + 3) & ~3;
        }
        mma_commit_if(leader, &acc_full);
        __syncwarp();
    }

    // ---------------- epilogue: all eight warps, two per tensor-memory lane quarter ----------------
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int n = n0 + row;
    const int grp = warp >> 2;                                  // epilogue warp group, 0 .. kSpEpiGroups - 1
    const bool ok = mbar_wait_warp(&acc_full, 0, p.status, 256) && sched_ok;
    tc_fence_after();
    const uint32_t mask_own = sched[0], mask_other = sched[1];
    uint16_t *out = static_cast<uint16_t *>(p.out);
    const int Wh = (g.W + 1) / 2;                               // slots owned by part 0 (split 2)

    // reads the BSE accumulator columns of `slot` (zeros when the slot received no MMA)
    auto load_slot = [&](int slot, bool present, float (&v)[BSE]) {
        if (ok && present) {
#pragma unroll
            for (int c0 = 0; c0 < BSE; c0 += 16) {
                uint32_t rr[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + slot * BSE + c0, rr);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(rr[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < BSE; ++j) v[j] = 0.f;
        }
    };
    // (F, N) outputs go through a [BSE][128] tile per epilogue group in the idle stage memory
    // (after the split reduction buffer), so that the group's 128 threads store whole 16-byte
    // pieces of feature rows; without room for the tiles every thread stores its own 2-byte values.
    const size_t red_bytes = split == 2 ? (size_t)((g.W + 1) / 2) * BSE * 128 * 4 : 0;
    const bool staged = !FA && red_bytes + (size_t)kSpEpiGroups * BSE * 256 <= (size_t)g.stages * g.stage_bytes;
    uint16_t *tile_s = reinterpret_cast<uint16_t *>(smem + red_bytes) + grp * (BSE * 128);
    auto store_slot = [&](int slot, const float (&v)[BSE]) {
        const int o = win * g.W + slot;
        const int f0 = o * BSE;
        if (staged) {
            // every thread of the group takes part (named barrier 1 + grp over its 128 threads)
#pragma unroll
            for (int j = 0; j < BSE; ++j) tile_s[j * 128 + row] = sp_cvt(v[j], p.bf16);
            named_sync(1 + grp, 128);
            const int t = (warp & 3) * 32 + lane;
#pragma unroll
            for (int c = t; c < BSE * 16; c += 128) {
                const int fr = c >> 4, nn = n0 + (c & 15) * 8;
                if (o < p.Fslots && f0 + fr < p.Fout && nn < p.N)
                    *reinterpret_cast<uint4 *>(out + (size_t)(f0 + fr) * p.N + nn) =
                        *reinterpret_cast<const uint4 *>(tile_s + fr * 128 + (c & 15) * 8);
            }
            named_sync(1 + grp, 128);                           // the tile may be written again
            return;
        }
        if (n >= p.N || o >= p.Fslots) return;
        if (FA) {
            uint16_t *dst = out + (size_t)n * p.Fout + f0;
            if (f0 + BSE <= p.Fout) {
#pragma unroll
                for (int j = 0; j < BSE; j += 8) {
                    uint4 pk;
                    pk.x = sp_pack(v[j], v[j + 1], p.bf16);
                    pk.y = sp_pack(v[j + 2], v[j + 3], p.bf16);
                    pk.z = sp_pack(v[j + 4], v[j + 5], p.bf16);
                    pk.w = sp_pack(v[j + 6], v[j + 7], p.bf16);
                    *reinterpret_cast<uint4 *>(dst + j) = pk;
                }
            } else {
#pragma unroll
                for (int j = 0; j < BSE; ++j)
                    if (f0 + j < p.Fout) dst[j] = sp_cvt(v[j], p.bf16);
            }
        } else {
#pragma unroll
            for (int j = 0; j < BSE; ++j)
                if (f0 + j < p.Fout) out[(size_t)(f0 + j) * p.N + n] = sp_cvt(v[j], p.bf16);
        }
    };

    if (split == 1) {
        for (int s = grp; s < g.W; s += kSpEpiGroups) {
            float v[BSE];
            load_slot(s, ((mask_own >> s) & 1u) != 0, v);
            store_slot(s, v);
        }
    } else {
        // Partial tiles of the two CTAs: part 0 owns slots [0, Wh), part 1 the rest.  Each CTA
        // sends its partial of the slots the other owns into the owner's (idle) stage memory:
        // red[local slot][column / 4][row][4] floats.
        float *red = reinterpret_cast<float *>(smem);
        cluster_sync();                                         // both CTAs' MMAs are done
        {
            const int peer = part ^ 1;
            const int lo = peer == 0 ? 0 : Wh, hi = peer == 0 ? Wh : g.W;
            for (int s = lo + grp; s < hi; s += kSpEpiGroups) {
                if (!((mask_own >> s) & 1u)) continue;          // the owner reads zeros for it
                float v[BSE];
                load_slot(s, true, v);
                const int ls = s - lo;
                const uint32_t base = map_to_rank(smem_u32(red + ((size_t)ls * (BSE / 4) * 128 + row) * 4), peer);
#pragma unroll
                for (int c4 = 0; c4 < BSE / 4; ++c4)
                    st_cluster_v4(base + c4 * 128 * 16, v[c4 * 4], v[c4 * 4 + 1], v[c4 * 4 + 2], v[c4 * 4 + 3]);
            }
        }
        cluster_sync();                                         // every partial has landed
        {
            const int lo = part == 0 ? 0 : Wh, hi = part == 0 ? Wh : g.W;
            for (int s = lo + grp; s < hi; s += kSpEpiGroups) {
                float v[BSE], pv[BSE];
                load_slot(s, ((mask_own >> s) & 1u) != 0, v);
                const bool peer_has = ((mask_other >> s) & 1u) != 0;
                const int ls = s - lo;
#pragma unroll
                for (int c4 = 0; c4 < BSE / 4; ++c4) {
                    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (peer_has)
                        t = *reinterpret_cast<const float4 *>(red + (((size_t)ls * (BSE / 4) + c4) * 128 + row) * 4);
                    pv[c4 * 4] = t.x;
                    pv[c4 * 4 + 1] = t.y;
                    pv[c4 * 4 + 2] = t.z;
                    pv[c4 * 4 + 3] = t.w;
                }
                // part 0's sources precede part 1's: add in that order on both CTAs
#pragma unroll
                for (int j = 0; j < BSE; ++j) v[j] = part == 0 ? v[j] + pv[j] : pv[j] + v[j];
                store_slot(s, v);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kSpLoaders) tmem_dealloc(tmem, 512);
}

// (F, N) activations -> contiguous panels: pan[tile][source][panel], each panel 128 rows x BSE
// features in the K-major operand layout, chunk (row r, 8 features h) at
// (r / 8) * BSE * 16 + h * 128 + (r % 8) * 16 bytes.  Rows >= N and features >= Fin are zero.
// A CTA transposes 64 features x 128 rows through shared memory, holding each pair of feature
// rows interleaved as 32-bit words t[pair][sample] (padded rows), so that an output chunk -- 8
// features of one sample -- is four 32-bit reads without bank conflicts.
template <int BSE>
__global__ void __launch_bounds__(256) k_sp_panelize(const uint16_t *act, uint16_t *pan, int N, int Fin, int Fsrc)
{
    constexpr int LD = 128 + 4;                        // words per padded row of t
    __shared__ __align__(16) uint32_t t[32][LD];       // t[p][n]: features f0 + 2p, f0 + 2p + 1 of sample n0 + n
    const int tile = blockIdx.x, f0 = blockIdx.y * 64, n0 = tile * 128;
    pdl_launch_dependents();
    pdl_wait();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int c = k * 256 + threadIdx.x;           // feature pair p, 8 samples from 8 cc
        const int p = c >> 4, cc = c & 15;
        const int f = f0 + 2 * p, nn = n0 + cc * 8;
        uint4 va = make_uint4(0, 0, 0, 0), vb = va;
        if (nn < N) {
            if (f < Fin) va = *reinterpret_cast<const uint4 *>(act + (size_t)f * N + nn);
            if (f + 1 < Fin) vb = *reinterpret_cast<const uint4 *>(act + (size_t)(f + 1) * N + nn);
        }
        const uint32_t a4[4] = {va.x, va.y, va.z, va.w}, b4[4] = {vb.x, vb.y, vb.z, vb.w};
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {                  // samples 2j, 2j + 1: low halves of a, b, then high
            w[2 * j] = (a4[j] & 0xFFFFu) | (b4[j] << 16);
            w[2 * j + 1] = (a4[j] >> 16) | (b4[j] & 0xFFFF0000u);
        }
        *reinterpret_cast<uint4 *>(&t[p][cc * 8]) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(&t[p][cc * 8 + 4]) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    __syncthreads();
    constexpr int CPR = BSE / 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = k * 256 + threadIdx.x;           // output chunk, in panel byte order
        const int r8 = c & 7, h = (c >> 3) % CPR, rg = (c / (8 * CPR)) & 15, pi = c / (128 * CPR);
        const int r = rg * 8 + r8;
        const int s = f0 / BSE + pi;
        if (s >= Fsrc) continue;
        const int p0 = (pi * BSE + h * 8) / 2;         // pairs p0 .. p0 + 3: features h*8 .. h*8 + 7
        uint16_t *dst = pan + ((size_t)tile * Fsrc + s) * (128 * BSE) + rg * (BSE * 8) + h * 64 + r8 * 8;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(t[p0][r], t[p0 + 1][r], t[p0 + 2][r], t[p0 + 3][r]);
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------

struct SpSched {
    int W = 0, split = 1, E = 0, R = 0, nwin = 0;
    uint32_t *d_stream = nullptr;
    int4 *d_desc = nullptr;     // per (launch position, part): window, stream offset, length, 0
    int max_words = 0;
    bool built = false;
};

struct SpScratch {
    void *ptr = nullptr;
    size_t bytes = 0;
};

struct SpState {
    std::map<uint64_t, SpSched> plans;           // key: pass, tiles
    std::map<cudaStream_t, SpScratch> scratch;   // (F, N) panels, one buffer per stream
    std::mutex mu;
};

template <typename T> bool sp_upload(T **d, const std::vector<T> &h)
{
    size_t n = std::max<size_t>(h.size(), 1);
    if (cudaMalloc(d, n * sizeof(T)) != cudaSuccess) return false;
    if (!h.empty() && cudaMemcpy(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
        return false;
    return true;
}

// (coarse) block edge, output slots and sources of a pass
void sp_shape(const bsmm_ctx *h, bool bwd, int &bse, int &Fslots, int &Fsrc)
{
    const int f = h->bs == 8 ? 2 : 1;
    const int Rc = (h->R + f - 1) / f, Sc = (h->S + f - 1) / f;
    bse = h->bs == 8 ? 16 : h->bs;
    Fslots = bwd ? Rc : Sc;
    Fsrc = bwd ? Sc : Rc;
}

// One window's entries: (source, records), sources increasing; records are the present
// (coarse) blocks of the source among the window's slots, slots increasing.
struct SpEnt {
    int src;
    std::vector<uint32_t> recs;
};

void sp_window(const bsmm_ctx *h, bool bwd, int W, int w, std::vector<SpEnt> &ents)
{
    const bool coarse = h->bs == 8;
    const int f = coarse ? 2 : 1;
    int bse, Fslots, Fsrc;
    sp_shape(h, bwd, bse, Fslots, Fsrc);
    std::vector<std::vector<uint32_t>> per(Fsrc);
    // walk the (coarse) layout rows/columns of the window's slots
    auto bid = [&](int c, int k) -> int32_t {
        if (c < 0 || c >= h->R || k < 0 || k >= h->S) return -1;
        const int32_t *b = h->h_row_ent.data() + h->h_row_ptr[c];
        const int32_t *e = h->h_row_ent.data() + h->h_row_ptr[c + 1];
        const int32_t *q = std::lower_bound(b, e, k);
        return (q != e && *q == k) ? h->h_row_ptr[c] + (int32_t)(q - b) : -1;
    };
    for (int sl = 0; sl < W; ++sl) {
        const int o = w * W + sl;
        if (o >= Fslots) break;
        if (!coarse) {
            if (!bwd) {
                // fprop: output column o, sources = rows with a block in column o
                for (int e = h->h_col_ptr[o]; e < h->h_col_ptr[o + 1]; ++e) {
                    const int id = h->h_col_ent[2 * e], c = h->h_col_ent[2 * e + 1];
                    per[c].push_back(((uint32_t)sl << 27) | (uint32_t)id);
                }
            } else {
                for (int e = h->h_row_ptr[o]; e < h->h_row_ptr[o + 1]; ++e)
                    per[h->h_row_ent[e]].push_back(((uint32_t)sl << 27) | (uint32_t)e);
            }
        } else {
            for (int s = 0; s < Fsrc; ++s) {
                const int cc = bwd ? o : s, kc = bwd ? s : o;   // coarse (c', k')
                int32_t ids[4];
                bool any = false;
                for (int cs = 0; cs < 2; ++cs)
                    for (int ks = 0; ks < 2; ++ks) {
                        ids[cs * 2 + ks] = bid(cc * 2 + cs, kc * 2 + ks);
                        any |= ids[cs * 2 + ks] >= 0;
                    }
                if (!any) continue;
                per[s].push_back(((uint32_t)sl << 27) | (uint32_t)(ids[0] + 1));
                for (int qq = 1; qq < 4; ++qq) per[s].push_back((uint32_t)(ids[qq] + 1));
            }
        }
    }
    (void)f;
    ents.clear();
    for (int s = 0; s < Fsrc; ++s)
        if (!per[s].empty()) ents.push_back(SpEnt{s, std::move(per[s])});
}

// Builds the schedule for windows of W slots, each split into `split` parts, chunks of at most
// E entries and R records.  Per window part a word stream:
//   [0] slots that receive a block in this part, [1] slots that do in the other part, [2..3] 0,
//   chunks: a 36-word prefix -- header (ne << 16) | nr, the MMA list lengths (byte q: MMA warp q),
//     2 spare words, and per MMA warp q 8 list words (accumulate flag << 31 | record << 16 |
//     entry << 12 | accumulator column) for the records whose slot % 4 == q -- then ne entries
//     (source << 8) | nrec and nr records (bs 32/16: (slot << 27) | id; bs 8: (slot << 27) |
//     (id00 + 1), id01 + 1, id10 + 1, id11 + 1, 0 = absent), padded to 4 words;
//   0 ends the stream; streams are padded to 4 words.  The accumulate flag is clear on the first
//   record of each slot in the part.  Returns false on an allocation failure; leaves built =
//   false when a stream exceeds kSpSchedWords.
bool sp_build(const bsmm_ctx *h, bool bwd, int W, int split, int E, int R, SpSched &sc)
{
    const int rw = h->bs == 8 ? 4 : 1;
    int bse, Fslots, Fsrc;
    sp_shape(h, bwd, bse, Fslots, Fsrc);
    const int nwin = (Fslots + W - 1) / W;
    const int panel = 128 * bse * 2, bslot = bse * bse * 2;
    std::vector<uint32_t> stream;
    std::vector<int32_t> off(nwin * split), len(nwin * split), order(nwin);
    std::vector<double> work(nwin, 0.0);
    std::vector<SpEnt> ents;
    int longest = 0;
    for (int w = 0; w < nwin; ++w) {
        sp_window(h, bwd, W, w, ents);
        // entries longer than R records are cut into several entries of the same source
        std::vector<SpEnt> cut;
        for (SpEnt &e : ents) {
            const int nrec = (int)e.recs.size() / rw;
            for (int r0 = 0; r0 < nrec; r0 += R)
                cut.push_back(SpEnt{e.src, std::vector<uint32_t>(e.recs.begin() + r0 * rw,
                                                                e.recs.begin() + std::min(nrec, r0 + R) * rw)});
        }
        double total = 0;
        for (const SpEnt &e : cut) total += panel + (double)e.recs.size() / rw * bslot;
        work[w] = total;
        // part boundaries by load bytes
        std::vector<size_t> bound(split + 1, cut.size());
        bound[0] = 0;
        if (split == 2) {
            double acc = 0;
            size_t i = 0;
            for (; i < cut.size(); ++i) {
                acc += panel + (double)cut[i].recs.size() / rw * bslot;
                if (acc >= total / 2) { ++i; break; }
            }
            bound[1] = std::min(i, cut.size());
        }
        std::vector<uint32_t> masks(split, 0);
        for (int pt = 0; pt < split; ++pt)
            for (size_t i = bound[pt]; i < bound[pt + 1]; ++i)
                for (size_t r = 0; r < cut[i].recs.size(); r += rw) masks[pt] |= 1u << (cut[i].recs[r] >> 27);
        for (int pt = 0; pt < split; ++pt) {
            const size_t start = stream.size();
            off[w * split + pt] = (int32_t)start;
            stream.push_back(masks[pt]);
            stream.push_back(split == 2 ? masks[pt ^ 1] : 0u);
            stream.push_back(0);
            stream.push_back(0);
            uint32_t seen = 0;                                  // slots that received an MMA so far
            size_t i = bound[pt];
            while (i < bound[pt + 1]) {
                // greedy: entries while at most E entries, R records, and 8 records per MMA warp
                int ne = 0, nr = 0, cnt[kSpMmaWarps] = {0, 0, 0, 0};
                size_t j = i;
                while (j < bound[pt + 1] && ne < E) {
                    const int er = (int)cut[j].recs.size() / rw;
                    int c2[kSpMmaWarps] = {cnt[0], cnt[1], cnt[2], cnt[3]};
                    bool fits = ne == 0 || nr + er <= R;
                    for (size_t q = 0; q < cut[j].recs.size(); q += rw) {
                        const int mw = (int)((cut[j].recs[q] >> 27) % kSpMmaWarps);
                        if (++c2[mw] > kSpList) fits = false;
                    }
                    if (!fits) break;
                    for (int q = 0; q < kSpMmaWarps; ++q) cnt[q] = c2[q];
                    ++ne;
                    nr += er;
                    ++j;
                }
                uint32_t lists[kSpMmaWarps][kSpList] = {};
                int lc[kSpMmaWarps] = {0, 0, 0, 0}, rr = 0;
                for (size_t k = i; k < j; ++k)
                    for (size_t q = 0; q < cut[k].recs.size(); q += rw, ++rr) {
                        const uint32_t sl = cut[k].recs[q] >> 27;
                        const int mw = (int)(sl % kSpMmaWarps);
                        const uint32_t acc = (seen >> sl) & 1u;
                        seen |= 1u << sl;
                        lists[mw][lc[mw]++] =
                            (acc << 31) | ((uint32_t)rr << 16) | ((uint32_t)(k - i) << 12) | (sl * (uint32_t)bse);
                    }
                stream.push_back(((uint32_t)ne << 16) | (uint32_t)nr);
                stream.push_back((uint32_t)lc[0] | ((uint32_t)lc[1] << 8) | ((uint32_t)lc[2] << 16) |
                                 ((uint32_t)lc[3] << 24));
                stream.push_back(0);
                stream.push_back(0);
                for (int q = 0; q < kSpMmaWarps; ++q) stream.insert(stream.end(), lists[q], lists[q] + kSpList);
                for (size_t k = i; k < j; ++k)
                    stream.push_back(((uint32_t)cut[k].src << 8) | (uint32_t)(cut[k].recs.size() / rw));
                for (size_t k = i; k < j; ++k) stream.insert(stream.end(), cut[k].recs.begin(), cut[k].recs.end());
                while (stream.size() % 4) stream.push_back(0);
                i = j;
            }
            stream.push_back(0);
            while (stream.size() % 4) stream.push_back(0);
            len[w * split + pt] = (int32_t)(stream.size() - start);
            longest = std::max(longest, len[w * split + pt]);
        }
    }
    if (longest > kSpSchedWords) return true;                  // built stays false
    // BSMM_SP_TEST_BAD_ID (tests only): the first record of the first window names block nnz + 5,
    // which the kernel must refuse (zero-filled, BSMM_ERR_BOUNDS) without touching memory past w
    if (getenv("BSMM_SP_TEST_BAD_ID") && stream.size() > (size_t)kSpHead + 1 && stream[kSpHead] != 0) {
        const uint32_t hdr = stream[kSpHead];
        const size_t r0 = kSpHead + kSpChunkHead + (hdr >> 16);
        if ((hdr & 0xFFFFu) > 0 && r0 < stream.size())
            stream[r0] = (stream[r0] & ~kIdMask) | (uint32_t)((h->nnz + 5) & kIdMask);
    }
    for (int w = 0; w < nwin; ++w) order[w] = w;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return work[a] > work[b]; });
    sc.W = W;
    sc.split = split;
    sc.E = E;
    sc.R = R;
    sc.nwin = nwin;
    sc.max_words = longest;
    std::vector<int4> desc((size_t)nwin * split);
    for (int j = 0; j < nwin; ++j)
        for (int pt = 0; pt < split; ++pt) {
            const int w = order[j];
            desc[(size_t)j * split + pt] = make_int4(w, off[w * split + pt], len[w * split + pt], 0);
        }
    if (!sp_upload(&sc.d_stream, stream) || !sp_upload(&sc.d_desc, desc))
        return false;
    sc.built = true;
    return true;
}

// Stage geometry for a plan: E panels and R blocks per stage, as many stages (a multiple of the
// producer count) as fit next to the schedule.
bool sp_geometry(const bsmm_ctx *h, const SpSched &sc, SpGeo &g, int &smem)
{
    const int bse = h->bs == 8 ? 16 : h->bs;
    const int panel = 128 * bse * 2, bslot = bse * bse * 2;
    g.W = sc.W;
    g.split = sc.split;
    g.E = sc.E;
    g.R = sc.R;
    g.b_off = sc.E * panel;
    g.stage_bytes = (g.b_off + sc.R * bslot + 1023) & ~1023;
    if (sc.W * bse > 512) return false;
    const int avail = kSpSmemBudget - 1024 - sc.max_words * 4;
    g.stages = std::min(kSpMaxStages, avail / g.stage_bytes) / kSpProducers * kSpProducers;
    if (g.stages < kSpProducers) return false;
    // the split reduction buffer lives in the stage memory
    if (sc.split == 2 && (size_t)((sc.W + 1) / 2) * bse * 128 * 4 > (size_t)g.stages * g.stage_bytes) return false;
    // more than half of an SM's shared memory: two CTAs never share an SM, so the two CTAs of a
    // cluster never wait on each other for the SM's 512 tensor-memory columns
    smem = std::max(g.stages * g.stage_bytes + sc.max_words * 4 + 1024, 120 * 1024);
    return true;
}

// Chooses window size and split for a pass and minibatch by an estimate of the slowest CTA:
// max(bytes loaded / 64 B per clk, MMA clocks) per window part plus per-chunk and fixed costs,
// times the number of waves over the SMs; MMA cost M128 x N16 x K16 39 clk, N32 40 clk per K step
// (both operands in shared memory, measured on GB300).  Then builds the schedule.
bool sp_plan(const bsmm_ctx *h, bool bwd, int ntiles, SpSched &out)
{
    int bse, Fslots, Fsrc;
    sp_shape(h, bwd, bse, Fslots, Fsrc);
    const int rw = h->bs == 8 ? 4 : 1;
    const double panel = 128.0 * bse * 2, bslot = bse * bse * 2.0;
    const int sms = std::max(1, h->sm_count);
    const double dens = std::min(1.0, (double)h->nnz / ((double)h->R * h->S) * (h->bs == 8 ? 4.0 : 1.0));
    // BSMM_SP_E / BSMM_SP_R pin the panels and blocks per stage (tuning and tests)
    const char *ee = getenv("BSMM_SP_E"), *er = getenv("BSMM_SP_R");
    const int E = ee ? std::max(1, std::min(8, atoi(ee))) : (bse == 32 ? 4 : 8);
    const int r_pin = er ? std::max(1, std::min(32, atoi(er))) : 0;
    const double mma_clk = bse == 32 ? 80.0 : 39.0;
    const int Wmax = std::min(32, 512 / bse);
    struct Cand { double t; int W, split, R; };
    std::vector<Cand> cands;
    std::vector<SpEnt> ents;
    // BSMM_SP_W / BSMM_SP_SPLIT pin the choice (tests)
    const char *ew = getenv("BSMM_SP_W"), *es = getenv("BSMM_SP_SPLIT");
    const int w_pin = ew ? std::max(1, std::min(Wmax, atoi(ew))) : 0, s_pin = es ? atoi(es) : 0;
    for (int W = Wmax; W >= 1; --W) {
        if (w_pin && W != w_pin) continue;
        // records per chunk: 1.5x the expected blocks of E sources over the window, capped so that
        // four stages fit next to the largest schedule
        const int r_fit = (int)(((kSpSmemBudget - 1024 - kSpSchedWords * 4) / kSpProducers - E * panel) / bslot);
        const int R = r_pin ? std::min(r_pin, std::max(1, r_fit))
                            : std::max(1, std::min({32, r_fit, std::max(8, (int)std::ceil(1.5 * E * W * dens) + 4)}));
        const int nwin = (Fslots + W - 1) / W;
        double worst = 0;
        for (int w = 0; w < nwin; ++w) {
            sp_window(h, bwd, W, w, ents);
            double u = 0, b = 0;
            for (const SpEnt &e : ents) {
                const int nrec = (int)e.recs.size() / rw;
                u += (nrec + R - 1) / R;
                b += nrec;
            }
            const double chunks = std::max(u / E, b / R);
            worst = std::max(worst, std::max((u * panel + b * bslot) / 64.0, b * mma_clk) + chunks * 300.0);
        }
        for (int split = 1; split <= 2; ++split) {
            if ((s_pin == 1 || s_pin == 2) && split != s_pin) continue;
            const long units = (long)nwin * ntiles * split;
            const double waves = std::ceil((double)units / sms);
            // fixed costs: launch and first loads, the split reduction, and the output stores
            const double t = waves * (worst / split + 3000.0 + (split == 2 ? 1500.0 : 0.0) + (double)W * bse * 2.0);
            cands.push_back(Cand{t, W, split, R});
        }
    }
    std::stable_sort(cands.begin(), cands.end(), [](const Cand &a, const Cand &b) { return a.t < b.t; });
    for (const Cand &c : cands) {
        SpSched sc;
        if (!sp_build(h, bwd, c.W, c.split, E, c.R, sc)) return false;
        if (!sc.built) continue;
        SpGeo g;
        int smem;
        if (!sp_geometry(h, sc, g, smem)) {
            cudaFree(sc.d_stream);
            cudaFree(sc.d_desc);
            continue;
        }
        out = sc;
        if (getenv("BSMM_SP_VERBOSE"))
            fprintf(stderr, "k_tc_sp plan: %s bs %d fa %d tiles %d: W %d split %d E %d R %d stages %d stage %d B, "
                            "grid %d, schedule %d words, estimate %.0f clk\n", bwd ? "bprop" : "fprop", h->bs, h->fa,
                    ntiles, g.W, g.split, g.E, g.R, g.stages, g.stage_bytes, sc.nwin * ntiles * sc.split,
                    sc.max_words, c.t);
        return true;
    }
    return true;                                                // nothing fits: out.built == false
}

SpState *sp_state(bsmm_ctx *h)
{
    if (!h->sp) h->sp = new SpState();
    return static_cast<SpState *>(h->sp);
}

template <typename... KArgs, typename... Args>
cudaError_t sp_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                      Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int BS, int FA, bool BWD>
bsmm_status sp_launch_kernel(bsmm_ctx *h, const SpSched &sc, const void *act, const void *w, void *out, int N,
                             bsmm_dtype t, cudaStream_t s)
{
    int bse, Fslots, Fsrc;
    sp_shape(h, BWD, bse, Fslots, Fsrc);
    SpParams p;
    p.act = act;
    p.w = w;
    p.out = out;
    p.stream = sc.d_stream;
    p.desc = sc.d_desc;
    p.status = h->d_status;
    p.N = N;
    p.Fin = (BWD ? h->S : h->R) * h->bs;
    p.Fout = (BWD ? h->R : h->S) * h->bs;
    p.Fsrc = Fsrc;
    p.Fslots = Fslots;
    p.ntiles = (N + 127) / 128;
    p.nnz = h->nnz;
    p.bf16 = t == BSMM_BF16 ? 1 : 0;
    int smem = 0;
    if (!sp_geometry(h, sc, p.g, smem)) return BSMM_ERR_UNSUPPORTED;
    auto kern = k_tc_sp<BS, FA, BWD>;
    static std::atomic<int> attr_set{-1};
    if (attr_set.load() != h->device) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpSmemBudget) != cudaSuccess)
            return BSMM_ERR_CUDA;
        attr_set.store(h->device);
    }
    const dim3 grid((unsigned)(sc.nwin * p.ntiles * sc.split));
    const cudaError_t le = sp_launch(kern, grid, dim3(kSpThreads), smem, s, sc.split, p);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

template <int BSE>
bsmm_status sp_panelize(bsmm_ctx *h, const void *act, void *pan, int N, int Fin, int Fsrc, cudaStream_t s)
{
    const dim3 grid((unsigned)((N + 127) / 128), (unsigned)((Fsrc * BSE + 63) / 64));
    const cudaError_t le =
        sp_launch(k_sp_panelize<BSE>, grid, dim3(256), 0, s, 1, static_cast<const uint16_t *>(act),
                  static_cast<uint16_t *>(pan), N, Fin, Fsrc);
    g_bsmm_launches += 1;
    return le == cudaSuccess ? BSMM_OK : BSMM_ERR_CUDA;
}

} // namespace

bool sp_supported(const bsmm_ctx *h, bsmm_dtype t)
{
    return (t == BSMM_F16 || t == BSMM_BF16) && h->nnz < (int64_t)kIdMask;
}

bsmm_status sp_fb(bsmm_ctx *h, bool bwd, const void *act, const void *w, void *out, int N, bsmm_dtype t,
                  cudaStream_t s)
{
    if (!sp_supported(h, t)) return BSMM_ERR_UNSUPPORTED;
    const int ntiles = (N + 127) / 128;
    SpState *st = sp_state(h);
    const SpSched *sc = nullptr;
    void *pan = nullptr;
    int bse, Fslots, Fsrc;
    sp_shape(h, bwd, bse, Fslots, Fsrc);
    {
        std::lock_guard<std::mutex> lk(st->mu);
        const uint64_t key = (uint64_t)bwd | ((uint64_t)ntiles << 1);
        auto it = st->plans.find(key);
        if (it == st->plans.end()) {
            SpSched plan;
            if (!sp_plan(h, bwd, ntiles, plan)) return BSMM_ERR_OOM;
            it = st->plans.emplace(key, plan).first;
        }
        if (!it->second.built) return BSMM_ERR_UNSUPPORTED;
        sc = &it->second;
        if (h->fa == 0) {
            const size_t bytes = (size_t)ntiles * Fsrc * 128 * bse * 2;
            SpScratch &sp = st->scratch[s];
            if (sp.bytes < bytes) {
                cudaFree(sp.ptr);                       // synchronises with work that may still use it
                sp.ptr = nullptr;
                sp.bytes = 0;
                if (cudaMalloc(&sp.ptr, bytes) != cudaSuccess) return BSMM_ERR_OOM;
                sp.bytes = bytes;
            }
            pan = sp.ptr;
        }
    }
    if (h->fa == 0) {
        const int Fin = (bwd ? h->S : h->R) * h->bs;
        const bsmm_status ps = bse == 32 ? sp_panelize<32>(h, act, pan, N, Fin, Fsrc, s)
                                         : sp_panelize<16>(h, act, pan, N, Fin, Fsrc, s);
        if (ps != BSMM_OK) return ps;
        act = pan;
    }
#define SP_CASE(BS_, FA_)                                                                          \
    if (h->bs == BS_ && h->fa == FA_)                                                              \
        return bwd ? sp_launch_kernel<BS_, FA_, true>(h, *sc, act, w, out, N, t, s)                \
                   : sp_launch_kernel<BS_, FA_, false>(h, *sc, act, w, out, N, t, s);
    SP_CASE(32, 1)
    SP_CASE(32, 0)
    SP_CASE(16, 1)
    SP_CASE(16, 0)
    SP_CASE(8, 1)
    SP_CASE(8, 0)
#undef SP_CASE
    return BSMM_ERR_UNSUPPORTED;
}

void sp_release(bsmm_ctx *h)
{
    if (!h->sp) return;
    SpState *st = static_cast<SpState *>(h->sp);
    for (auto &kv : st->plans) {
        cudaFree(kv.second.d_stream);
        cudaFree(kv.second.d_desc);
    }
    for (auto &kv : st->scratch) cudaFree(kv.second.ptr);
    delete st;
    h->sp = nullptr;
}
