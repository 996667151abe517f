// Flash-attention mainloop for sm_103a on the 5th-generation tensor cores:
// TMA loads Q/K/V tiles into 128-byte-swizzled shared memory, one thread
// issues tcgen05.mma into TMEM accumulators, and a warpgroup runs the online
// softmax reading S from TMEM and writing P (bf16) back into TMEM over the
// same columns, where the P.V product reads it as its A operand.  MMAs from
// one thread execute in issue order, so S of tile t+2 (same columns) is
// written only after P.V of tile t has read P.
//
// Persistent: one CTA per SM walks the work items (128-row query tile x head)
// item = blockIdx.x, blockIdx.x + gridDim.x, ...  The pipeline (K/V stages,
// S buffers, barrier phases) runs on across items, so the next item's Q/K/V
// loads and first Q.K^T overlap the current item's softmax and epilogue.
//   warps 0-7  softmax + epilogue: two warpgroups share each query row
//              (TMEM lane); warpgroup h runs an online softmax of its own over
//              key columns [64h, 64h + 64) of every tile, with its own
//              accumulator O_h; the two are merged at the end of the item
//   warp  8    TMA producer (Q per item, K/V double-buffered) + key-tile
//              group bitmaps for the masks
//   warp  9    TMEM allocator and MMA issuer: S = Q K^T, then O_h += P_h V_h
//              for each half as soon as that half's P is written
// TMEM columns: S double buffer at [0,128) and [128,256) (P_h written over
// S columns [64h, 64h + 32)), O_0 at [256, 256+D), O_1 at [384, 384+D).
//
// Modes (the decomposition of the allowed-pair set of Focus attention,
// gist.science/zh technical summary 2.1.3: within-group causal attention
// plus cross-group local attention):
//   kGroup  : query/key rows are one group's gathered members (ascending
//             token order); causal in that order; a pair whose tokens share
//             several groups is scored only in the lowest shared group.
//   kWindow : original token order; keys with i - window < j <= i that share
//             no group with the query.
//   kDense  : plain causal attention (the comparison baseline).
// kGroup and kWindow write partial results: the normalised output of every
// (row, head) in fp16, scaled by a power of two 2^-e that puts its largest
// entry in [2^14, 2^15) (11-bit precision at any magnitude, no overflow), and
// {base-2 log-sum-exp, 2^e}.  The merge kernel combines them.  kDense writes
// its final bf16 output directly.
//
// Group masks: for every key tile the producer builds colbits[g][4], the set
// of the tile's 128 key columns whose token belongs to group g.  A query row
// excludes the columns in the union of colbits over the groups that must not
// be shared (all its groups for kWindow; its groups below the tile's group
// for kGroup): k lookups of 16 bytes instead of a test per column.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "focus_ptx.cuh"
#include "focus_tmem_wide.cuh"

namespace focus {

enum AttnMode { kGroup = 0, kWindow = 1, kDense = 2 };

struct AttnArgs {
    int B, n, Hq, Hkv;
    int rows;              // rows per batch of the Q/K/V tensors (n or n*topk packed)
    int window;
    float scale_log2;      // softmax scale * log2(e)
    int K, topk;
    const int32_t *gids;   // group ids per Q/K/V row: [B, rows, topk]
    const int32_t *offsets;  // [B, K+1]
    const int32_t *pos;    // [B, n*topk] token of each group-order row
    const int2 *tiles;     // kGroup work list: (b*K + g, tile index in group)
    const int *ntiles;     // kGroup: number of valid entries in tiles
    __nv_bfloat16 *out;    // kDense: O [B, n, Hq, D]
    float *lse;            // kDense: lse [B, Hq, n], natural log (nullable)
    // partial results: O / l as fp16 scaled by 2^-e, and {lse base 2, 2^e}
    __half *part_out16;    // kGroup  [B, rows, Hq, D]
    float2 *part_meta_out; // kGroup  [B, rows, Hq]
    __half *win_out16;     // kWindow [B, n, Hq, D]
    float2 *win_meta_out;  // kWindow [B, n, Hq]
    int *status;           // device status word
    int32_t *pair_count;   // nullable: scored pairs per query (head 0)
    long long *trace;      // nullable: per-CTA wait/phase cycle counters [grid][32]
};

// Per-CTA trace slots (SM cycles): producer 0-5, MMA issuer 8-14, softmax 16-24.
enum {
    TR_P_IEMPTY = 0, TR_P_QEMPTY = 1, TR_P_KEMPTY = 2, TR_P_VEMPTY = 3, TR_P_TOTAL = 4,
    TR_P_RING = 5, TR_M_PFULL = 8, TR_M_VFULL = 9, TR_M_IFULL = 10, TR_M_QFULL = 11,
    TR_M_KFULL = 12, TR_M_SEMPTY = 13, TR_M_TOTAL = 14, TR_M_ISSUE = 15, TR_S_IFULL = 16, TR_S_META = 17,
    TR_S_SFULL = 18, TR_S_PVDONE = 19, TR_S_PVLAST = 20, TR_S_EPI = 21, TR_S_TOTAL = 22,
    TR_S_ITEMS = 23, TR_S_TILES = 24, TR_E_TMEM = 25, TR_E_SCALE = 26, TR_E_STORE = 27,
    TR_T_SLOAD = 28, TR_T_MASK = 29, TR_T_RESCALE = 30, TR_T_P = 31, kTraceSlots = 32
};

__device__ __forceinline__ void trace_flush(const long long *tr, long long *dst, int lo, int hi)
{
    for (int i = lo; i < hi; ++i) dst[i] = tr[i];
}

constexpr int kThreads = 320;   // 2 softmax warpgroups + producer + MMA warp
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSoftmaxThreads = 256;
constexpr int kSoftmaxWarps = kSoftmaxThreads / 32;
constexpr uint32_t kOStride = 128;   // TMEM columns from O_0 to O_1
constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // key rows per tile
constexpr int kMaxTopk = 8;

template <int D>
struct AttnSmem {
    static constexpr uint32_t kTile = kBM * D * 2;           // one bf16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;               // 2 stages
    static constexpr uint32_t kV = kK + 2 * kTile;           // 2 stages
    static constexpr uint32_t kP = kV + 2 * kTile;           // epilogue staging, 128 x D x 2 B
    static constexpr uint32_t kBar = kP + kBM * D * 2;       // 28 mbarriers
    static constexpr uint32_t kMisc = kBar + 28 * 8;         // tmem slot, abort flag
    static constexpr uint32_t kTrace = kMisc + 16;           // int64 [32] trace counters
    static constexpr uint32_t kXchg = kTrace + 256;          // float [1024]: softmax exchange
    static constexpr uint32_t kColbits = (kXchg + 4096 + 127) / 128 * 128;   // uint32 [2][K][4]
    // then the work-item ring: 2 slots of ring_slot_bytes()
    __host__ __device__ static constexpr uint32_t colbits_bytes(int K)
    {
        return 2u * 16u * (uint32_t)K;
    }
    __host__ __device__ static constexpr uint32_t ring_slot_bytes(int mode, int topk)
    {
        return (32u + 128u * 4u * (uint32_t)topk + 127u) / 128u * 128u;
    }
    // dynamic shared memory of a launch (K groups and topk are 0 for kDense)
    __host__ __device__ static constexpr uint32_t bytes(int mode, int K, int topk)
    {
        return kColbits + colbits_bytes(K) + 2u * ring_slot_bytes(mode, topk) + 1024u;
    }
};

// mbarrier slots
// (B_PFULL and B_PVD: [half h][tile parity], index 2h + (tile & 1))
enum {
    B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_VFULL = 4, B_KEMPTY = 6, B_VEMPTY = 8,
    B_SFULL = 10, B_SEMPTY = 12, B_PFULL = 14, B_PVD = 18, B_META = 22, B_IFULL = 24,
    B_IEMPTY = 26, kNumBars = 28
};

// Work-item ring slot: the decoded item (8 ints) followed by the group ids of
// its 128 query rows, [128][topk].
struct RingSlot {
    int *item;
    int *gid;
};

template <int D>
__device__ __forceinline__ RingSlot ring_slot(uint8_t *sm, int mode, int K, int topk, int slot)
{
    using L = AttnSmem<D>;
    uint8_t *base = sm + L::kColbits + L::colbits_bytes(K) + slot * L::ring_slot_bytes(mode, topk);
    RingSlot r;
    r.item = reinterpret_cast<int *>(base);
    r.gid = r.item + 8;
    return r;
}

// Bit mask of columns c in [lo, hi] within the 32-column word starting at c0.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int c0)
{
    int a = lo - c0, b = hi - c0;
    if (a < 0) a = 0;
    if (b > 31) b = 31;
    if (a > b) return 0u;
    const uint32_t upto_b = (b == 31) ? 0xffffffffu : ((2u << b) - 1u);
    const uint32_t below_a = (1u << a) - 1u;
    return upto_b & ~below_a;
}

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct WorkItem {
    int b, h, q0, qend, kv_lo, nkv, g, gend;
};

// O *= f for this thread's TMEM lane (D columns), 32 columns at a time.
// Rarely taken (the row max has to grow by more than 2^8); it runs after the
// tile's scores are dead, so its registers do not add to the softmax loop's.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float f)
{
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(taddr + c * 32, o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] *= f;
        tmem_st32(taddr + c * 32, o);
    }
    tmem_st_wait();
}

template <int MODE>
__device__ __forceinline__ int total_items(const AttnArgs &a)
{
    if (MODE == kGroup) return (*a.ntiles) * a.Hq;
    return a.B * ((a.n + kBM - 1) / kBM) * a.Hq;
}

// The k-th item of CTA c among G persistent CTAs: rounds of G items, walked
// forwards in even rounds and backwards in odd ones, so that on a list sorted
// by decreasing cost every CTA gets a similar total.
__device__ __forceinline__ int item_of(int k, int c, int G)
{
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Work item -> query tile.  Heads vary fastest, so the heads that share a key
// tile run side by side; items come heaviest first (kGroup: the tile list is
// ordered by decreasing cost; kDense: the last query tiles first).
template <int MODE>
__device__ __forceinline__ WorkItem decode_item(const AttnArgs &a, int item)
{
    WorkItem w;
    w.g = 0;
    w.gend = 0;
    if (MODE == kGroup) {
        const int tr = item / a.Hq;
        w.h = item - tr * a.Hq;
        const int2 tl = a.tiles[tr];
        w.b = tl.x / a.K;
        w.g = tl.x - w.b * a.K;
        const int gs = a.offsets[w.b * (a.K + 1) + w.g];
        w.gend = a.offsets[w.b * (a.K + 1) + w.g + 1];
        w.q0 = gs + kBM * tl.y;
        w.qend = min(w.q0 + kBM, w.gend);
        w.kv_lo = gs;
        w.nkv = tl.y + 1;
    } else {
        const int nqt = (a.n + kBM - 1) / kBM;
        w.h = item % a.Hq;
        const int rest = item / a.Hq;
        int qt = rest % nqt;
        w.b = rest / nqt;
        if (MODE == kDense) qt = nqt - 1 - qt;
        w.q0 = kBM * qt;
        w.qend = min(w.q0 + kBM, a.n);
        if (MODE == kDense) {
            w.kv_lo = 0;
            w.nkv = qt + 1;
        } else {
            w.kv_lo = max(0, w.q0 - a.window + 1);
            w.nkv = a.window > 0 ? (w.qend - w.kv_lo + kBN - 1) / kBN : 0;
        }
    }
    return w;
}

template <int MODE, int D>
__global__ void __launch_bounds__(kThreads, 1)
    focus_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnArgs a)
{
    using L = AttnSmem<D>;
    constexpr int kChunks = D / 64;   // 64-column (128-byte) chunks per row

    const int nitems = total_items<MODE>(a);
    if ((int)blockIdx.x >= nitems) return;       // whole CTA leaves before any set-up
    const int kv_per_q = a.Hq / a.Hkv;

    // ------------------------------------------------------------ set-up
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sQ = sm + L::kQ;
    uint8_t *sK = sm + L::kK;
    uint8_t *sV = sm + L::kV;
    uint8_t *sStage = sm + L::kP;       // epilogue staging: one output row per thread
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kMisc + 4);
    uint32_t *colbits = reinterpret_cast<uint32_t *>(sm + L::kColbits);   // [2][K][4]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_QEMPTY], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_KFULL + s], 1);
            mbar_init(&bars[B_VFULL + s], 1);
            mbar_init(&bars[B_KEMPTY + s], 1);
            mbar_init(&bars[B_VEMPTY + s], 1);
            mbar_init(&bars[B_SFULL + s], 1);
            mbar_init(&bars[B_SEMPTY + s], kSoftmaxWarps);   // one lane per warp
            mbar_init(&bars[B_META + s], 32);
        }
        for (int s = 0; s < 4; ++s) {
            mbar_init(&bars[B_PFULL + s], kSoftmaxWarps / 2);   // one lane per warp of a half
            mbar_init(&bars[B_PVD + s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_IFULL + s], 32);           // the producer warp's lanes
            mbar_init(&bars[B_IEMPTY + s], kSoftmaxWarps + 1);   // softmax warps + MMA thread
        }
        long long *trz = reinterpret_cast<long long *>(sm + L::kTrace);
        for (int i = 0; i < kTraceSlots; ++i) trz[i] = 0;
        *abort_flag = 0;
        mbar_fence_init();
    }
    const int rtopk = (MODE == kDense) ? 0 : a.topk;    // per-row ring data width
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 256;     // O_0; O_1 at tmem_o + kOStride

    long long *tr = reinterpret_cast<long long *>(sm + L::kTrace);   // zeroed at set-up
    const long long t_start = clock64();

    if (warp == kProducerWarp) {
        // ------------------------------------------------- TMA producer
        const bool trc = a.trace != nullptr && lane == 0;
        int T = 0, iq = 0;            // key tiles and query tiles issued so far
        bool ok = true;
        for (int k = 0, item = blockIdx.x; ok && item < nitems;
             item = item_of(++k, blockIdx.x, gridDim.x)) {
            // ---- publish the decoded item and its rows' metadata (ring slot k & 1,
            // free once item k - 2 is fully consumed)
            if (k >= 2 && lane == 0)
                ok = mbar_wait_t(&bars[B_IEMPTY + (k & 1)], ((k >> 1) - 1) & 1, abort_flag,
                                 a.status, trc, tr[0]);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                ok = false;
                break;
            }
            const long long t_ring = trc ? clock64() : 0;
            const WorkItem w = decode_item<MODE>(a, item);
            {
                const RingSlot rs = ring_slot<D>(sm, MODE, a.K, rtopk, k & 1);
                if (lane == 0) {
                    rs.item[0] = w.b;
                    rs.item[1] = w.h;
                    rs.item[2] = w.q0;
                    rs.item[3] = w.qend;
                    rs.item[4] = w.kv_lo;
                    rs.item[5] = w.nkv;
                    rs.item[6] = w.g;
                    rs.item[7] = w.gend;
                }
                if (MODE != kDense) {
                    // the 128 query rows' group ids, [128][topk], coalesced
                    const int32_t *src = a.gids + ((int64_t)w.b * a.rows + w.q0) * a.topk;
                    const int nval = (w.qend - w.q0) * a.topk;
                    for (int i = lane; i < kBM * a.topk; i += 32)
                        rs.gid[i] = i < nval ? src[i] : -1;
                }
                __syncwarp();
                mbar_arrive(&bars[B_IFULL + (k & 1)]);
                if (trc) tr[TR_P_RING] += clock64() - t_ring;
            }
            if (w.nkv == 0) continue;
            const int kvh = w.h / kv_per_q;
            const int kv_end = (MODE == kGroup) ? w.gend : a.n;
            // Q buffer free once the last Q.K^T of the previous item is done
            if (iq >= 1 && lane == 0)
                ok = mbar_wait_t(&bars[B_QEMPTY], (iq - 1) & 1, abort_flag, a.status, trc, tr[1]);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_QFULL], L::kTile);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_4d(sQ + c * 16384, &tmQ, &bars[B_QFULL], c * 64, w.h, w.q0, w.b);
            }
            ++iq;
            for (int u = 0; u < w.nkv; ++u, ++T) {
                const int st = T & 1;
                const int r0 = w.kv_lo + kBN * u;
                // Group ids of this tile's key rows (lane: rows lane + 32 j),
                // loaded now so that the waits below hide their latency.
                int kg[4][kMaxTopk];
                if (MODE != kDense) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = r0 + lane + 32 * j;
                        const int32_t *gp = a.gids + ((int64_t)w.b * a.rows + row) * a.topk;
#pragma unroll
                        for (int s = 0; s < kMaxTopk; ++s)
                            kg[j][s] = (row < kv_end && s < a.topk) ? gp[s] : -1;
                    }
                }
                if (T >= 2 && lane == 0)
                    ok = mbar_wait_t(&bars[B_KEMPTY + st], ((T >> 1) - 1) & 1, abort_flag,
                                     a.status, trc, tr[2]);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[B_KFULL + st], L::kTile);
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_4d(sK + st * L::kTile + c * 16384, &tmK, &bars[B_KFULL + st],
                                    c * 64, kvh, r0, w.b);
                }
                // V and the masks of stage st are free once P.V of tile T-2 is
                // done (its softmax finished reading colbits[st] before P).
                if (T >= 2 && lane == 0)
                    ok = mbar_wait_t(&bars[B_VEMPTY + st], ((T >> 1) - 1) & 1, abort_flag,
                                     a.status, trc, tr[3]);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[B_VFULL + st], L::kTile);
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_4d(sV + st * L::kTile + c * 16384, &tmV, &bars[B_VFULL + st],
                                    c * 64, kvh, r0, w.b);
                }
                if (MODE != kDense) {
                    // colbits[st][g][q] bit c: key column 32q + c belongs to group g
                    uint32_t *cb = colbits + (size_t)st * a.K * 4;
                    for (int i = lane; i < a.K * 4; i += 32) cb[i] = 0u;
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int s = 0; s < kMaxTopk; ++s) {
                            const int gi = kg[j][s];
                            if ((unsigned)gi < (unsigned)a.K)
                                atomicOr(&cb[gi * 4 + j], 1u << lane);
                        }
                    }
                    mbar_arrive(&bars[B_META + st]);
                }
                __syncwarp();
            }
        }
        if (trc) {
            tr[TR_P_TOTAL] = clock64() - t_start;
            trace_flush(tr, a.trace + (int64_t)blockIdx.x * kTraceSlots, 0, 8);
        }
        // If the CTA gave up early, let the copies already issued land before
        // shared memory is released.
        if (*abort_flag && lane == 0) {
            const uint64_t t0 = global_timer_ns();
            while (iq > 0 && !mbar_try_wait(&bars[B_QFULL], (iq - 1) & 1) &&
                   global_timer_ns() - t0 < 100000000ull) {
            }
            for (int t = max(0, T - 2); t < T + 1; ++t) {
                const int st = t & 1;
                while (!mbar_try_wait(&bars[B_KFULL + st], (t >> 1) & 1) &&
                       global_timer_ns() - t0 < 200000000ull) {
                }
                while (!mbar_try_wait(&bars[B_VFULL + st], (t >> 1) & 1) &&
                       global_timer_ns() - t0 < 300000000ull) {
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0) {
            const bool trc = a.trace != nullptr;
            constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
            const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK);
            const uint32_t v_base = smem_u32(sV);

            // O_h += P_h(t) V_h(t) for both halves h of the tile's keys, each
            // as soon as its P is written; `first` starts the item's accumulators.
            auto issue_pv = [&](int t, bool first) -> bool {
                const int st = t & 1;
                if (!mbar_wait_t(&bars[B_VFULL + st], (t >> 1) & 1, abort_flag, a.status, trc,
                                 tr[9]))
                    return false;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait_t(&bars[B_PFULL + 2 * h + (t & 1)], (t >> 1) & 1, abort_flag,
                                     a.status, trc, tr[8]))
                        return false;
                    tc_fence_after();
                    const long long ti = trc ? clock64() : 0;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // A = P_h in TMEM over the half's S columns: 16 keys = 8 columns.
                        const uint32_t at = tmem + st * kBN + 64 * h + kk * 8;
                        // B = V (MN-major): 16 key rows of 128 bytes; the second
                        // 64-column half of D lies 16 KB further (LBO).
                        const uint64_t bd = sdesc_sw128(
                            v_base + st * L::kTile + (4 * h + kk) * 2048, 16384, 1024);
                        tc_mma_bf16_ts(tmem_o + h * kOStride, at, bd, kIdescPV,
                                       (!first || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&bars[B_PVD + 2 * h + (t & 1)]);
                    if (trc) tr[TR_M_ISSUE] += clock64() - ti;
                }
                tc_commit(&bars[B_VEMPTY + st]);
                return true;
            };

            int T = 0, iq = 0;
            bool ok = true;
            for (int k = 0, item = blockIdx.x; ok && item < nitems;
             item = item_of(++k, blockIdx.x, gridDim.x)) {
                ok = mbar_wait_t(&bars[B_IFULL + (k & 1)], (k >> 1) & 1, abort_flag, a.status, trc,
                                 tr[10]);
                if (!ok) break;
                const int *wi = ring_slot<D>(sm, MODE, a.K, rtopk, k & 1).item;
                WorkItem w;
                w.nkv = wi[5];
                mbar_arrive(&bars[B_IEMPTY + (k & 1)]);
                if (w.nkv == 0) continue;
                ok = mbar_wait_t(&bars[B_QFULL], iq & 1, abort_flag, a.status, trc, tr[11]);
                for (int u = 0; ok && u < w.nkv; ++u, ++T) {
                    const int st = T & 1;
                    ok = mbar_wait_t(&bars[B_KFULL + st], (T >> 1) & 1, abort_flag, a.status, trc,
                                     tr[12]);
                    if (!ok) break;
                    if (T >= 2) {
                        ok = mbar_wait_t(&bars[B_SEMPTY + st], ((T >> 1) - 1) & 1, abort_flag,
                                         a.status, trc, tr[13]);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const long long ti = trc ? clock64() : 0;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint64_t ad = sdesc_sw128(q_base + off, 16, 1024);
                        const uint64_t bd = sdesc_sw128(k_base + st * L::kTile + off, 16, 1024);
                        tc_mma_bf16(tmem + st * kBN, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&bars[B_SFULL + st]);
                    tc_commit(&bars[B_KEMPTY + st]);
                    if (u == w.nkv - 1) tc_commit(&bars[B_QEMPTY]);
                    if (trc) tr[TR_M_ISSUE] += clock64() - ti;
                    if (u >= 1) ok = issue_pv(T - 1, u == 1);
                }
                if (ok) ok = issue_pv(T - 1, w.nkv == 1);
                ++iq;
            }
            if (trc) {
                tr[TR_M_TOTAL] = clock64() - t_start;
                trace_flush(tr, a.trace + (int64_t)blockIdx.x * kTraceSlots, 8, 16);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------- softmax: two independent warpgroups
        // Thread t: query row r = t mod 128 (its TMEM lane).  Warpgroup wg =
        // t / 128 owns key columns [64 wg, 64 wg + 64) of every S tile and runs
        // its own online softmax over them (reference max, row sum, and the
        // accumulator O_wg = sum of P V over its keys).  The warpgroups meet
        // only at the start and the end of an item, where the two partial
        // softmaxes of each row are merged exactly.
        constexpr int kDH = D / 2;                       // output columns per warpgroup
        constexpr int kCh = D / 8;                       // 16-byte chunks per output row
        const int wg = warp >> 2;
        const int r = threadIdx.x & 127;                 // row in tile, TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int cb0 = wg * 64;                         // first key column of this half
        const uint32_t o_own = tmem_o + lane_off + wg * kOStride;   // O_wg, this lane
        float *xm = reinterpret_cast<float *>(sm + L::kXchg);   // [2 wg][128] reference max
        float *xl = xm + 256;                                    // [2 wg][128] row sum
        float *xa = xl + 256;                                    // [2 wg][128] max |O|
        int *xc = reinterpret_cast<int *>(xa + 256);             // [2 wg][128] pair count
        const bool trc = a.trace != nullptr && threadIdx.x == 0;
        int T = 0;
        bool ok = true;
        for (int k = 0, item = blockIdx.x; ok && item < nitems;
             item = item_of(++k, blockIdx.x, gridDim.x)) {
            // the item and this row's metadata, published by the producer
            // A failed wait is carried in okl to the next 256-thread barrier,
            // which ends the loops in both warpgroups together.
            const int slot = k & 1;
            bool okl = mbar_wait_t(&bars[B_IFULL + slot], (k >> 1) & 1, abort_flag, a.status, trc,
                                   tr[16]);
            if (!named_bar_and(1, kSoftmaxThreads, okl)) {
                ok = false;
                break;
            }
            const RingSlot rs = ring_slot<D>(sm, MODE, a.K, rtopk, slot);
            WorkItem w;
            w.b = rs.item[0];
            w.h = rs.item[1];
            w.q0 = rs.item[2];
            w.qend = rs.item[3];
            w.kv_lo = rs.item[4];
            w.nkv = rs.item[5];
            w.g = rs.item[6];
            w.gend = rs.item[7];
            const int prow = w.q0 + r;                   // row in the Q tensor
            const bool qvalid = prow < w.qend;
            int qi = prow;                               // token index of the row
            // Groups whose columns this row must not score: every group of the
            // row (kWindow), or the row's groups below the tile's group (kGroup).
            int qg[kMaxTopk];          // -1 = unused slot
#pragma unroll
            for (int s = 0; s < kMaxTopk; ++s) {
                qg[s] = -1;
                if (MODE != kDense && qvalid && s < a.topk) {
                    const int gi = rs.gid[r * a.topk + s];
                    if ((MODE == kWindow || gi < w.g) && (unsigned)gi < (unsigned)a.K)
                        qg[s] = gi;
                }
            }
            if (MODE == kGroup && qvalid && a.pair_count)
                qi = a.pos[(int64_t)w.b * a.rows + prow];

            float m_ref = -CUDART_INF_F;   // reference max (base 2) applied to O_wg and l
            float l = 0.f;                 // row sum over this half's keys
            int cnt = 0;

            for (int u = 0; u < w.nkv; ++u, ++T) {
                const int st = T & 1;
                const int kvb = w.kv_lo + kBN * u;       // first key row of the tile
                if (MODE != kDense)
                    okl = mbar_wait_t(&bars[B_META + st], (T >> 1) & 1, abort_flag, a.status, trc,
                                      tr[17]);
                okl = okl && mbar_wait_t(&bars[B_SFULL + st], (T >> 1) & 1, abort_flag, a.status,
                                         trc, tr[18]);
                if (!okl) break;                         // on to the end-of-item barrier
                tc_fence_after();
                long long tt = trc ? clock64() : 0;
                float s[64];
                tmem_ld32(tmem + lane_off + st * kBN + cb0, s);
                tmem_ld32(tmem + lane_off + st * kBN + cb0 + 32, s + 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_SEMPTY + st]);
                // Keep this half's P.V barriers at most one phase behind: S of
                // tile T complete means P.V of tile T - 2 complete (the tensor
                // pipe runs in issue order), so this wait returns at once.
                if (T >= 2)
                    okl = mbar_wait_t(&bars[B_PVD + 2 * wg + (T & 1)], ((T - 2) >> 1) & 1,
                                      abort_flag, a.status, trc, tr[19]);
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_SLOAD] += t2 - tt;
                    tt = t2;
                }

                // ---- which of this half's 64 keys the row may score
                uint32_t ex0 = 0u, ex1 = 0u;
                if (MODE != kDense) {
                    const uint4 *cb =
                        reinterpret_cast<const uint4 *>(colbits + (size_t)st * a.K * 4);
#pragma unroll
                    for (int x = 0; x < kMaxTopk; ++x) {
                        if (qg[x] >= 0) {
                            const uint4 v = cb[qg[x]];
                            ex0 |= wg ? v.z : v.x;
                            ex1 |= wg ? v.w : v.y;
                        }
                    }
                }
                uint32_t okb[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c0 = cb0 + 32 * j;
                    uint32_t bits;
                    if (!qvalid)
                        bits = 0u;
                    else if (MODE == kGroup)
                        bits = range_bits(0, prow - kvb, c0);          // causal, group order
                    else if (MODE == kWindow)
                        bits = range_bits(qi - a.window + 1 - kvb, qi - kvb, c0);
                    else
                        bits = range_bits(0, qi - kvb, c0);
                    okb[j] = bits & ~(j ? ex1 : ex0);
                }
                if (a.pair_count) cnt += __popc(okb[0]) + __popc(okb[1]);

                // masked raw scores; the half-row max over 8 independent chains
                // (no selects where every key of the warp's rows is allowed)
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = -CUDART_INF_F;
                if (!__all_sync(0xffffffffu, (okb[0] & okb[1]) == 0xffffffffu)) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const bool on = (okb[c >> 5] >> (c & 31)) & 1u;
                        s[c] = on ? s[c] : -CUDART_INF_F;
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7])) *
                                 a.scale_log2;   // scale > 0, so max(s) * scale = max(s * scale)
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_MASK] += t2 - tt;
                    tt = t2;
                }

                // Lazy rescaling: keep the reference max unless the half-row
                // max grows by more than 2^8.  Only a rescale touches O_wg, so
                // only a rescale waits for the previous tile's P.V (after P is
                // written, so that the wait overlaps the exponentials).
                const float m_new = fmaxf(m_ref, mx);
                const bool grow = (m_ref == -CUDART_INF_F) || (m_new > m_ref + 8.f);
                const bool resc = grow && m_ref != -CUDART_INF_F;
                const float new_ref = grow ? m_new : m_ref;
                const float f = resc ? exp2f(m_ref - new_ref) : 1.f;
                const bool any_resc = __any_sync(0xffffffffu, resc);
                m_ref = new_ref;
                const float ref = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;

                // ---- P = 2^(s * scale - ref) in bf16 into TMEM over this half's
                // own S columns (key c in column 64 wg + c / 2): the A operand of
                // this half's P.V
                const float nref = -ref, sc2 = a.scale_log2;
                float rs8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p0 = exp2f(fmaf(s[2 * j], sc2, nref));
                    const float p1 = exp2f(fmaf(s[2 * j + 1], sc2, nref));
                    rs8[j & 7] += p0 + p1;
                    pk[j] = pack_bf16x2(p0, p1);
                }
                tmem_st32u(tmem + lane_off + st * kBN + cb0, pk);
                tmem_st_wait();
                l = fmaf(l, f, ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                                   ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7])));
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_P] += t2 - tt;
                    tt = t2;
                }
                if (any_resc) {
                    okl = okl && mbar_wait_t(&bars[B_PVD + 2 * wg + ((T - 1) & 1)],
                                             ((T - 1) >> 1) & 1, abort_flag, a.status, trc,
                                             tr[19]);
                    tc_fence_after();
                    rescale_o<D>(o_own, f);   // warp-wide
                    if (trc) tr[TR_T_RESCALE] += clock64() - tt;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFULL + 2 * wg + (T & 1)]);
                if (!okl) break;
            }

            // ---- epilogue: merge the two halves of each row
            const long long t_epi = trc ? clock64() : 0;
            if (w.nkv > 0) {
                // both halves' last two P.V (this thread reads both accumulators),
                // in phase order
                const int last = T - 1;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (last >= 1)
                        okl = okl && mbar_wait_t(&bars[B_PVD + 2 * h + ((last - 1) & 1)],
                                                 ((last - 1) >> 1) & 1, abort_flag, a.status, trc,
                                                 tr[20]);
                    okl = okl && mbar_wait_t(&bars[B_PVD + 2 * h + (last & 1)], (last >> 1) & 1,
                                             abort_flag, a.status, trc, tr[20]);
                }
                tc_fence_after();
            }
            xm[wg * 128 + r] = m_ref;
            xl[wg * 128 + r] = l;
            xc[wg * 128 + r] = cnt;
            if (!named_bar_and(1, kSoftmaxThreads, okl)) {
                ok = false;
                break;
            }
            long long te = trc ? clock64() : 0;
            const float m0 = xm[r], m1 = xm[128 + r];
            const float mrow = fmaxf(m0, m1);
            const float f0 = (m0 == -CUDART_INF_F) ? 0.f : exp2f(m0 - mrow);
            const float f1 = (m1 == -CUDART_INF_F) ? 0.f : exp2f(m1 - mrow);
            const float lt = f0 * xl[r] + f1 * xl[128 + r];
            const bool has = lt > 0.f;
            const float lse2 = has ? mrow + log2f(lt) : -CUDART_INF_F;   // base 2
            const float inv_l = has ? 1.f / lt : 0.f;
            const float g0 = f0 * inv_l, g1 = f1 * inv_l;   // weights of O_0 and O_1
            // this warpgroup's output columns [kDH wg, kDH wg + kDH) of both accumulators
            const uint32_t oa = tmem_o + lane_off + wg * kDH;
            // Pass 1: the largest |O| entry of this half row (partials only),
            // then of the whole row through shared memory.
            float amax_h = 0.f;
            if (MODE != kDense && w.nkv > 0) {
                float am8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) am8[i] = 0.f;
#pragma unroll 1
                for (int c = 0; c < kDH / 16; ++c) {
                    float o0[16], o1[16];
                    tmem_ld16(oa + c * 16, o0);
                    tmem_ld16(oa + kOStride + c * 16, o1);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        am8[e & 7] = fmaxf(am8[e & 7], fabsf(fmaf(o0[e], g0, o1[e] * g1)));
                }
                amax_h = fmaxf(fmaxf(fmaxf(am8[0], am8[1]), fmaxf(am8[2], am8[3])),
                               fmaxf(fmaxf(am8[4], am8[5]), fmaxf(am8[6], am8[7])));
            }
            xa[wg * 128 + r] = amax_h;
            named_bar_sync(1, kSoftmaxThreads);
            const float amax = fmaxf(xa[r], xa[128 + r]);
            const int cnt_row = xc[r] + xc[128 + r];
            int64_t orow = 0;
            if (MODE == kGroup)
                orow = ((int64_t)w.b * a.rows + prow) * a.Hq + w.h;
            else
                orow = ((int64_t)w.b * a.n + qi) * a.Hq + w.h;
            if (trc) {
                const long long t2 = clock64();
                tr[TR_E_TMEM] += t2 - te;
                te = t2;
            }
            // Partials: O in fp16 scaled by a power of two so that the largest
            // entry lies in [2^14, 2^15) (11-bit precision at any magnitude, no
            // overflow), plus {lse (base 2), 2^e}.  Dense: O in bf16.
            int ex = 0;
            if (amax > 0.f && amax < CUDART_INF_F) frexpf(amax, &ex);   // amax < 2^ex
            const float mul = (MODE == kDense) ? 1.f : __int_as_float((127 + 15 - ex) << 23);
            const float up = __int_as_float((127 - 15 + ex) << 23);     // 2^(ex - 15)
            const float w0 = g0 * mul, w1 = g1 * mul;
            // Pass 2: combine, scale, pack and stage this half row, 16 columns at
            // a time (16-byte chunk q at slot q ^ (r mod D/8): conflict-free).
            const uint32_t srow = smem_u32(sStage) + r * (D * 2);
#pragma unroll 1
            for (int c = 0; c < kDH / 16; ++c) {
                float o[16];
                if (w.nkv > 0) {
                    float o1[16];
                    tmem_ld16(oa + c * 16, o);
                    tmem_ld16(oa + kOStride + c * 16, o1);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = fmaf(o[e], w0, o1[e] * w1);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = 0.f;
                }
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int q = wg * (kCh / 2) + c * 2 + qq;
                    const float *v = o + qq * 8;
                    if (MODE == kDense)
                        st_shared_v4(srow + ((q ^ (r & (kCh - 1))) << 4),
                                     pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                     pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                    else
                        st_shared_v4(srow + ((q ^ (r & (kCh - 1))) << 4),
                                     pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]),
                                     pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
                }
            }
            if (qvalid && wg == 0) {
                if (MODE == kDense) {
                    if (a.lse)
                        a.lse[((int64_t)w.b * a.Hq + w.h) * a.n + qi] =
                            lse2 * 0.69314718055994531f;
                } else {
                    (MODE == kGroup ? a.part_meta_out : a.win_meta_out)[orow] =
                        make_float2(lse2, up);
                }
            }
            if (trc) {
                const long long t2 = clock64();
                tr[TR_E_SCALE] += t2 - te;
                te = t2;
            }
            named_bar_sync(1, kSoftmaxThreads);          // whole rows staged
            {
                // warps q and q + 4 copy out the first and second 16 rows of
                // quadrant q with whole-row, coalesced 16-byte stores
                constexpr int kRowsPer = 32 / kCh;            // rows per warp instruction
                const int sub = lane / kCh, q = lane % kCh;
                uint16_t *obase = (MODE == kDense) ? reinterpret_cast<uint16_t *>(a.out)
                                  : (MODE == kGroup) ? reinterpret_cast<uint16_t *>(a.part_out16)
                                                     : reinterpret_cast<uint16_t *>(a.win_out16);
                const int64_t rstride = (MODE == kGroup) ? (int64_t)a.rows : (int64_t)a.n;
#pragma unroll
                for (int it = 0; it < 16 / kRowsPer; ++it) {
                    const int j = (warp & 3) * 32 + wg * 16 + it * kRowsPer + sub;   // tile row
                    const int row = w.q0 + j;
                    uint4 v;
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                 : "r"(smem_u32(sStage) + j * (D * 2) + ((q ^ (j & (kCh - 1))) << 4)));
                    if (row < w.qend) {
                        const int64_t orr = ((int64_t)w.b * rstride + row) * a.Hq + w.h;
                        reinterpret_cast<uint4 *>(obase + orr * D)[q] = v;
                    }
                }
            }
            named_bar_sync(1, kSoftmaxThreads);          // staging free for the next item
            if (trc) tr[TR_E_STORE] += clock64() - te;
            if (qvalid && a.pair_count && w.h == 0 && wg == 0)
                atomicAdd(&a.pair_count[(int64_t)w.b * a.n + qi], cnt_row);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_IEMPTY + slot]);     // ring slot no longer read
            if (trc) {
                tr[TR_S_EPI] += clock64() - t_epi;
                tr[TR_S_ITEMS] += 1;
                tr[TR_S_TILES] += w.nkv;
            }
        }
        if (trc) {
            tr[TR_S_TOTAL] = clock64() - t_start;
            trace_flush(tr, a.trace + (int64_t)blockIdx.x * kTraceSlots, 16, 32);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace focus
