// Flash-attention mainloop for sm_103a on the 5th-generation tensor cores.
//
// One CTA takes two 128-row query tiles, its two "halves" h = 0, 1, against
// one stream of 128-row key/value tiles, so that every K/V tile that TMA
// brings into shared memory feeds twice the tensor work: either the same
// query rows for two heads that share a key/value head (GQA with an even
// ratio), or two consecutive query tiles of one head.  One thread issues
// tcgen05.mma into TMEM accumulators,
//   S_h = Q_h K^T   (both operands in 128-byte-swizzled shared memory)
//   O_h += P_h V    (P_h in TMEM, V in shared memory)
// in the order  S_0(j), O_1 += P_1(j-1) V(j-1), S_1(j), O_0 += P_0(j) V(j),
// so that while one warpgroup turns S_h into P_h the tensor core runs the
// other half's two products: each half has a full tile of tensor time for
// its softmax.  The tensor pipe executes in issue order, hence when S_h(j) is
// complete, O_h += P_h(j-1) V(j-1) is complete as well: the softmax may
// rescale O_h without a wait, and S_h(j+1), written over the same TMEM
// columns, comes only after P_h(j) was read.
//
// Roles (384 threads, three warpgroups):
//   warps 0-3  softmax and epilogue of half 0 (thread r: query row r = TMEM lane r)
//   warps 4-7  softmax and epilogue of half 1
//   warp  8    producer: publishes each work item, loads Q of each half by TMA,
//              streams K/V (double-buffered) and each key tile's group bitmaps
//   warp  9    TMEM allocator and MMA issuer
//   warps 10-11 kGroup: copy the query rows of half 0 / 1 from the original Q
//              (through pos); otherwise idle
// The third warpgroup hands registers to the softmax warpgroups (setmaxnreg),
// which keep a whole 128-column row of S in registers.
// TMEM columns: S_0 [0,128), S_1 [128,256) (P_h over the first 64 columns of
// S_h, two bf16 keys per column), O_0 [256, 256+D), O_1 [384, 384+D).
//
// Persistent: one CTA per SM runs work items one after another.  Its
// producer takes the next item from a counter (group and window kernels: the
// list is ordered by decreasing cost, so a CTA that is ahead takes more of the
// cheap items at its end) or from a fixed share of the list (dense kernel),
// and publishes it in a two-slot ring that the other roles read, an end mark
// after the last.  The pipeline (K/V stages, barrier phases) runs on across
// items, so the next item's loads and first Q.K^T overlap the current item's
// softmax and epilogue.
//
// Modes (the decomposition of the allowed-pair set of Focus attention,
// gist.science/zh technical summary 2.1.3: within-group causal attention
// plus cross-group local attention):
//   kGroup  : query/key rows are one group's gathered members (ascending
//             token order); causal in that order and outside the window
//             (i - j >= window); a pair whose tokens share several groups is
//             scored only in the lowest shared group.
//   kWindow : original token order; every key with i - window < j <= i.
// The two modes split the allowed set without overlap: the window pairs all
// go to kWindow, which then needs no group masks, and kGroup leaves them out
// with one bound per row (the window holds few of a group's members, so that
// bound cuts into one or two key tiles of an item).
//   kDense  : plain causal attention (the comparison baseline).
// kGroup and kWindow write partial results: the normalised output of every
// (row, head) in fp16, scaled by a power of two 2^-e that puts its largest
// entry in [2^14, 2^15) (11-bit precision at any magnitude, no overflow), and
// {base-2 log-sum-exp, 2^e}.  The merge kernel combines them.  kDense writes
// its final bf16 output directly.
//
// Group masks (kGroup): for every key tile a bulk copy brings colbits[g][4],
// the set of the tile's 128 key columns whose token belongs to group g, from a
// table that the mask-table kernel writes before the attention kernels run.  A
// query row excludes the columns in the union of colbits over its groups below
// the tile's group: k lookups of 16 bytes instead of a test per column.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "focus_ptx.cuh"
#include "focus_tmem_wide.cuh"
#include "focus_internal.h"

namespace focus {

enum AttnMode { kGroup = 0, kWindow = 1, kDense = 2 };

struct AttnArgs {
    int B, n, Hq, Hkv;
    int rows;              // rows per batch of the Q/K/V tensors (n or n*topk packed)
    int window;
    float scale_log2;      // softmax scale * log2(e)
    int K, topk;
    int pair_heads;        // 1: halves are heads 2s, 2s+1 of one query tile; 0: query
                           // tiles 2p, 2p+1 of one head
    const int32_t *gids;   // group ids per Q/K/V row: [B, rows, topk]
    const int32_t *offsets;  // [B, K+1]
    const int32_t *pos;    // [B, n*topk] token of each group-order row
    const int2 *tiles;     // kGroup work list: (b*K + g, tile or tile-pair index in group)
    const int *ntiles;     // kGroup: number of valid entries in tiles
    const __nv_bfloat16 *q;  // kGroup: the original Q [B, n, Hq, D]; its rows are
                             // copied into the query tiles through pos
    const uint4 *masks;    // kGroup: group bitmaps of the key tiles: [B][mask_tiles][K],
                           // word j bit c = key 32 j + c of the tile is in the group
    int64_t mask_tiles;    // slots per batch (group tile u of g: off[g] / 128 + g + u)
    const int32_t *wlo;    // kGroup: [B, rows] the first row of each row's group
                           // inside its window; keys from there on are kWindow's
    __nv_bfloat16 *out;    // kDense: O [B, n, Hq, D]
    float *lse;            // kDense: lse [B, Hq, n], natural log (nullable)
    // partial results: O / l as fp16 scaled by 2^-e, and {lse base 2, 2^e}
    __half *part_out16;    // kGroup  [B, rows, Hq, D]
    float2 *part_meta_out; // kGroup  [B, rows, Hq]
    __half *win_out16;     // kWindow [B, n, Hq, D]
    float2 *win_meta_out;  // kWindow [B, n, Hq]
    int *work;             // nullable: work-item counter, zero before the launch; the
                           // producers take items from it in list order (null: CTA c
                           // takes items c, 2G - 1 - c, 2G + c, ... of G CTAs)
    int *status;           // device status word
    int32_t *pair_count;   // nullable: scored pairs per query (head 0)
    long long *trace;      // nullable: per-CTA wait/phase cycle counters [grid][32]
};

// Per-CTA trace slots (SM cycles): producer 0-5, MMA issuer 8-15, softmax of
// half 0 (its first thread) 16-31.
enum {
    TR_P_IEMPTY = 0, TR_P_QEMPTY = 1, TR_P_KEMPTY = 2, TR_P_VEMPTY = 3, TR_P_TOTAL = 4,
    TR_P_RING = 5, TR_M_PFULL = 8, TR_M_LOADS = 9, TR_M_IFULL = 10, TR_M_TOTAL = 14,
    TR_M_ISSUE = 15, TR_S_IFULL = 16, TR_S_META = 17,
    TR_S_SFULL = 18, TR_S_ODONE = 20, TR_S_EPI = 21, TR_S_TOTAL = 22, TR_S_ITEMS = 23,
    TR_S_TILES = 24, TR_E_TMEM = 25, TR_E_SCALE = 26, TR_E_STORE = 27, TR_T_SLOAD = 28,
    TR_T_MASK = 29, TR_T_RESCALE = 30, TR_T_P = 31, kTraceSlots = 32
};

__device__ __forceinline__ void trace_flush(const long long *tr, long long *dst, int lo, int hi)
{
    for (int i = lo; i < hi; ++i) dst[i] = tr[i];
}

constexpr int kThreads = 384;   // 2 softmax warpgroups + producer, MMA and 2 idle warps
// Registers per thread after the split: softmax warpgroups / the third one.
// 256 * kRegsSoftmax + 128 * kRegsOther must not exceed the launch's
// kThreads * (registers per thread at launch), which the launcher checks.
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 104;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // key rows per tile
constexpr int kMaxTopk = 8;
constexpr uint32_t kOStride = 128;        // TMEM columns from O_0 to O_1

// mbarrier slots ([half] or [stage] pairs)
enum {
    B_QFULL = 0, B_QEMPTY = 2, B_KFULL = 4, B_VFULL = 6, B_KEMPTY = 8, B_VEMPTY = 10,
    B_SFULL = 12, B_PFULL = 14, B_ODONE = 16, B_META = 18, B_IFULL = 20, B_IEMPTY = 22,
    B_DRAIN = 24, kNumBars = 25
};

template <int D>
struct AttnSmem {
    static constexpr uint32_t kTile = kBM * D * 2;           // one bf16 tile
    static constexpr uint32_t kQ = 0;                        // Q_0, Q_1
    static constexpr uint32_t kK = kQ + 2 * kTile;           // 2 stages
    static constexpr uint32_t kV = kK + 2 * kTile;           // 2 stages
    static constexpr uint32_t kBar = kV + 2 * kTile;
    static constexpr uint32_t kMisc = kBar + kNumBars * 8;   // tmem slot, abort flag
    static constexpr uint32_t kTrace = kMisc + 16;           // int64 [32] trace counters
    static constexpr uint32_t kColbits = (kTrace + 256 + 127) / 128 * 128;   // uint32 [2][K][4]
    // then the work-item ring: 2 slots of kRingSlot bytes
    static constexpr uint32_t kRingSlot = 128;               // an Item (16 ints)
    __host__ __device__ static constexpr uint32_t colbits_bytes(int K)
    {
        return 2u * 16u * (uint32_t)K;
    }
    // dynamic shared memory of a launch (K groups; 0 for kDense)
    __host__ __device__ static constexpr uint32_t bytes(int K)
    {
        return kColbits + colbits_bytes(K) + 2u * kRingSlot + 1024u;
    }
};

// A work item: two halves over one key/value row range.  Half h has query
// rows [q0[h], qend[h]) of head hd[h] and scores key tiles [ulo[h], uhi[h])
// of the item's nkv tiles (none when ulo == uhi).
struct Item {
    int b, g, gend, kv_lo, nkv;
    int hd[2], q0[2], qend[2], ulo[2], uhi[2];
};

// Work-item ring slot: the fields of one Item as put_item lays them out.
template <int D>
__device__ __forceinline__ int *ring_slot(uint8_t *sm, int K, int slot)
{
    using L = AttnSmem<D>;
    return reinterpret_cast<int *>(sm + L::kColbits + L::colbits_bytes(K) + slot * L::kRingSlot);
}

// p[15]: the item's index, or -1 for "no more items" (the other fields unset).
__device__ __forceinline__ void put_item(int *p, const Item &w, int item)
{
    p[15] = item;
    if (item < 0) return;
    p[0] = w.b;
    p[1] = w.g;
    p[2] = w.gend;
    p[3] = w.kv_lo;
    p[4] = w.nkv;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        p[5 + h] = w.hd[h];
        p[7 + h] = w.q0[h];
        p[9 + h] = w.qend[h];
        p[11 + h] = w.ulo[h];
        p[13 + h] = w.uhi[h];
    }
}

__device__ __forceinline__ Item get_item(const int *p)
{
    Item w;
    w.b = p[0];
    w.g = p[1];
    w.gend = p[2];
    w.kv_lo = p[3];
    w.nkv = p[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        w.hd[h] = p[5 + h];
        w.q0[h] = p[7 + h];
        w.qend[h] = p[9 + h];
        w.ulo[h] = p[11 + h];
        w.uhi[h] = p[13 + h];
    }
    return w;
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

// Head slots per query tile: heads pair up when they share a key/value head.
__device__ __forceinline__ int head_slots(const AttnArgs &a)
{
    return a.pair_heads ? a.Hq / 2 : a.Hq;
}

template <int MODE>
__device__ __forceinline__ int total_items(const AttnArgs &a)
{
    if (MODE == kGroup) return (*a.ntiles) * head_slots(a);
    const int nqt = (a.n + kBM - 1) / kBM;
    const int nq = a.pair_heads ? nqt : (nqt + 1) / 2;
    return a.B * nq * head_slots(a);
}

// The k-th item of CTA c among G persistent CTAs: rounds of G items, walked
// forwards in even rounds and backwards in odd ones, so that on a list sorted
// by decreasing cost every CTA gets a similar total.
__device__ __forceinline__ int item_of(int k, int c, int G)
{
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Work item -> two query tiles and their key tiles.  Head slots vary
// fastest, so items that share key tiles run side by side; items come
// heaviest first (kGroup: the tile list is ordered by decreasing cost;
// kDense: the last query tiles first).
template <int MODE>
__device__ __forceinline__ Item decode_item(const AttnArgs &a, int item)
{
    Item w;
    const int hsl = head_slots(a);
    const int hs = item % hsl;
    const int rest = item / hsl;
    w.hd[0] = a.pair_heads ? 2 * hs : hs;
    w.hd[1] = a.pair_heads ? 2 * hs + 1 : hs;
    w.g = 0;
    w.gend = 0;
    int t0, base, end;     // first half's query tile; the row range tiles index into
    if (MODE == kGroup) {
        const int2 tl = a.tiles[rest];
        w.b = tl.x / a.K;
        w.g = tl.x - w.b * a.K;
        base = a.offsets[w.b * (a.K + 1) + w.g];
        end = a.offsets[w.b * (a.K + 1) + w.g + 1];
        w.gend = end;
        t0 = a.pair_heads ? tl.y : 2 * tl.y;
    } else {
        const int nqt = (a.n + kBM - 1) / kBM;
        const int nq = a.pair_heads ? nqt : (nqt + 1) / 2;
        int qp = rest % nq;
        w.b = rest / nq;
        if (MODE == kDense) qp = nq - 1 - qp;
        base = 0;
        end = a.n;
        t0 = a.pair_heads ? qp : 2 * qp;
    }
    int lo[2], hi[2];      // key rows of each half: [lo, hi)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int t = (a.pair_heads || h == 0) ? t0 : t0 + 1;
        w.q0[h] = base + kBM * t;
        w.qend[h] = min(w.q0[h] + kBM, end);
        if (w.qend[h] < w.q0[h]) w.qend[h] = w.q0[h];
        if (MODE == kWindow) {
            // key tiles on multiples of 128 rows (the same tile count as
            // starting at the band's first key), so that each has a mask slot
            lo[h] = max(0, w.q0[h] - a.window + 1) / kBN * kBN;
            hi[h] = a.window > 0 ? w.qend[h] : lo[h];
        } else {
            lo[h] = base;
            hi[h] = w.qend[h];
        }
    }
    w.kv_lo = lo[0];
    const int kv_hi = max(hi[0], hi[1]);
    w.nkv = kv_hi > w.kv_lo ? (kv_hi - w.kv_lo + kBN - 1) / kBN : 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (hi[h] > lo[h]) {
            w.ulo[h] = (lo[h] - w.kv_lo) / kBN;
            w.uhi[h] = (hi[h] - w.kv_lo + kBN - 1) / kBN;
        } else {
            w.ulo[h] = 0;
            w.uhi[h] = 0;
        }
    }
    return w;
}

// (x0, x1) * s + c on two fp32 lanes in one instruction.
__device__ __forceinline__ void fma2(float &d0, float &d1, float x0, float x1, float s, float c)
{
    asm("{\n\t.reg .b64 rx, rs, rc, rd;\n\t"
        "mov.b64 rx, {%2, %3};\n\t"
        "mov.b64 rs, {%4, %4};\n\t"
        "mov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, rx, rs, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(x0), "f"(x1), "f"(s), "f"(c));
}

// (a0, a1) += (b0, b1) on two fp32 lanes in one instruction.
__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

template <int MODE, int D>
__global__ void __launch_bounds__(kThreads, 1)
    focus_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnArgs a)
{
    using L = AttnSmem<D>;
    constexpr int kChunks = D / 64;   // 64-column (128-byte) chunks per row

    // kGroup's work-list length is written by an earlier kernel on the stream
    if (MODE == kGroup) grid_dep_sync();
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
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kMisc + 4);
    uint32_t *colbits = reinterpret_cast<uint32_t *>(sm + L::kColbits);   // [2][K][4]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_QFULL + s], MODE == kGroup ? 32 : 1);   // Q-loader lanes
            mbar_init(&bars[B_QEMPTY + s], 1);
            mbar_init(&bars[B_KFULL + s], 1);
            mbar_init(&bars[B_VFULL + s], 1);
            mbar_init(&bars[B_KEMPTY + s], 1);
            mbar_init(&bars[B_VEMPTY + s], 1);
            mbar_init(&bars[B_SFULL + s], 1);
            mbar_init(&bars[B_PFULL + s], 4);            // one lane per warp of the half
            mbar_init(&bars[B_ODONE + s], 1);
            mbar_init(&bars[B_META + s], 1);             // + the mask copy's bytes
            mbar_init(&bars[B_IFULL + s], 32);
            // 8 softmax warps + MMA thread (+ the two Q-loader warps of kGroup)
            mbar_init(&bars[B_IEMPTY + s], MODE == kGroup ? 11 : 9);
        }
        mbar_init(&bars[B_DRAIN], 1);
        long long *trz = reinterpret_cast<long long *>(sm + L::kTrace);
        for (int i = 0; i < kTraceSlots; ++i) trz[i] = 0;
        *abort_flag = 0;
        mbar_fence_init();
    }
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
    // (set-up above touches no global memory; launched with launch_pdl)
    grid_dep_sync();

    long long *tr = reinterpret_cast<long long *>(sm + L::kTrace);   // zeroed at set-up
    const long long t_start = clock64();

    if (warp >= 8) {
        // third warpgroup: gives registers back, then producer and MMA issuer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
        if (warp == kProducerWarp) {
            // ------------------------------------------------- TMA producer
            const bool trc = a.trace != nullptr && lane == 0;
            int T = 0;                    // key tiles issued so far
            int iq[2] = {0, 0};           // query tiles loaded per half
            bool ok = true;
            for (int k = 0; ok; ++k) {
                // ---- take the next item and publish it decoded (ring slot k & 1,
                // free once item k - 2 is fully consumed); past the list's end,
                // an end mark that stops the other roles
                if (k >= 2 && lane == 0)
                    ok = mbar_wait_t(&bars[B_IEMPTY + (k & 1)], ((k >> 1) - 1) & 1, abort_flag,
                                     a.status, trc, tr[TR_P_IEMPTY]);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                const long long t_ring = trc ? clock64() : 0;
                int item = 0;
                if (lane == 0)
                    item = a.work ? atomicAdd(a.work, 1) : item_of(k, blockIdx.x, gridDim.x);
                item = __shfl_sync(0xffffffffu, item, 0);
                const bool more = item < nitems;
                Item w;
                w.nkv = 0;
                if (more) w = decode_item<MODE>(a, item);
                {
                    if (lane == 0) put_item(ring_slot<D>(sm, a.K, k & 1), w, more ? item : -1);
                    __syncwarp();
                    mbar_arrive(&bars[B_IFULL + (k & 1)]);
                    if (trc) tr[TR_P_RING] += clock64() - t_ring;
                }
                if (!more) break;
                if (w.nkv == 0) continue;
                const int kvh = w.hd[0] / kv_per_q;
                // Q_h: its buffer is free once the last Q_h.K^T of its previous
                // item is done.  (kGroup: the Q-loader warps copy the rows.)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (MODE == kGroup || w.uhi[h] <= w.ulo[h]) continue;
                    if (iq[h] >= 1 && lane == 0)
                        ok = mbar_wait_t(&bars[B_QEMPTY + h], (iq[h] - 1) & 1, abort_flag, a.status,
                                         trc, tr[TR_P_QEMPTY]);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[B_QFULL + h], L::kTile);
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_4d(sQ + h * L::kTile + c * 16384, &tmQ, &bars[B_QFULL + h],
                                        c * 64, w.hd[h], w.q0[h], w.b);
                    }
                    ++iq[h];
                }
                if (!ok) break;
                // mask slot of tile 0 (see AttnArgs::masks)
                const int64_t mslot =
                    (int64_t)w.b * a.mask_tiles + w.kv_lo / kBN + (MODE == kGroup ? w.g : 0);
                for (int u = 0; u < w.nkv; ++u, ++T) {
                    const int st = T & 1;
                    const int r0 = w.kv_lo + kBN * u;
                    if (T >= 2 && lane == 0)
                        ok = mbar_wait_t(&bars[B_KEMPTY + st], ((T >> 1) - 1) & 1, abort_flag,
                                         a.status, trc, tr[TR_P_KEMPTY]);
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
                    // V and the masks of stage st are free once every P.V of tile
                    // T-2 is done (its softmaxes read colbits[st] before writing P).
                    if (T >= 2 && lane == 0)
                        ok = mbar_wait_t(&bars[B_VEMPTY + st], ((T >> 1) - 1) & 1, abort_flag,
                                         a.status, trc, tr[TR_P_VEMPTY]);
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
                    if (MODE == kGroup && lane == 0) {
                        // colbits[st] <- the tile's group bitmaps
                        mbar_arrive_expect_tx(&bars[B_META + st], 16u * (uint32_t)a.K);
                        bulk_load(colbits + (size_t)st * a.K * 4, a.masks + (mslot + u) * a.K,
                                  16u * (uint32_t)a.K, &bars[B_META + st]);
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
                for (int h = 0; h < 2; ++h)
                    while (iq[h] > 0 && !mbar_try_wait(&bars[B_QFULL + h], (iq[h] - 1) & 1) &&
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
                    while (MODE == kGroup && !mbar_try_wait(&bars[B_META + st], (t >> 1) & 1) &&
                           global_timer_ns() - t0 < 400000000ull) {
                    }
                }
            }
        } else if (warp == kMmaWarp) {
            // -------------------------------------------------- MMA issuer
            if (lane == 0) {
                const bool trc = a.trace != nullptr;
                // trace: waits for the ring, for loads (K, V, Q), for P; time in issue
                long long c_if = 0, c_ld = 0, c_p = 0, c_is = 0;
                constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false, false);
                constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
                // Low descriptor words of the first Q, K and V tiles.  The start
                // address is the low field (address / 16), so any other tile or
                // step inside a tile is one add of a constant.
                constexpr uint32_t kHiKM = sdesc_hi(1024);     // Q, K: K-major rows
                constexpr uint32_t kHiMN = sdesc_hi(1024);     // V: MN-major
                const uint32_t dq0 = sdesc_lo(smem_u32(sQ), 16);
                const uint32_t dk0 = sdesc_lo(smem_u32(sK), 16);
                const uint32_t dv0 = sdesc_lo(smem_u32(sV), 16384);
                constexpr uint32_t kTileD = L::kTile >> 4;
                int T = 0;                     // key tiles of earlier items
                int iq[2] = {0, 0};            // Q loads consumed per half
                int np[2] = {0, 0};            // P.V products issued per half
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    ok = mbar_wait_t(&bars[B_IFULL + (k & 1)], (k >> 1) & 1, abort_flag, a.status,
                                     trc, c_if);
                    if (!ok) break;
                    const int *wi = ring_slot<D>(sm, a.K, k & 1);   // Item fields
                    if (wi[15] < 0) break;                           // no more items
                    const int nkv = wi[4];
                    const int ulo[2] = {wi[11], wi[12]}, uhi[2] = {wi[13], wi[14]};
                    mbar_arrive(&bars[B_IEMPTY + (k & 1)]);
                    if (nkv == 0) continue;
                    bool qready[2] = {false, false}, first[2] = {true, true};
                    int kready = -1, vready = -1;   // last tile whose K / V load was waited
                    // Q_h.K^T of tile u into S_h
                    auto issue_qk = [&](int h, int u) -> bool {
                        const int t = T + u, st = t & 1;
                        if (kready < u) {
                            if (!mbar_wait_t(&bars[B_KFULL + st], (t >> 1) & 1, abort_flag, a.status,
                                             trc, c_ld))
                                return false;
                            kready = u;
                        }
                        if (!qready[h]) {
                            if (!mbar_wait_t(&bars[B_QFULL + h], iq[h] & 1, abort_flag, a.status, trc,
                                             c_ld))
                                return false;
                            qready[h] = true;
                        }
                        tc_fence_after();
                        const long long ti = trc ? clock64() : 0;
                        const uint32_t qd = dq0 + h * kTileD, kd = dk0 + st * kTileD;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // 16 columns = 32 bytes; 64 columns = one 16 KB swizzle block
                            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                            tc_mma_bf16_lo<kHiKM, kHiKM>(tmem + h * kBN, qd + off, kd + off,
                                                         kIdescQK, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(&bars[B_SFULL + h]);
                        if (u == uhi[h] - 1) tc_commit(&bars[B_QEMPTY + h]);
                        if (trc) c_is += clock64() - ti;
                        return true;
                    };
                    // O_h += P_h(u) V(u)
                    auto issue_pv = [&](int h, int u) -> bool {
                        const int t = T + u, st = t & 1;
                        if (vready < u) {
                            if (!mbar_wait_t(&bars[B_VFULL + st], (t >> 1) & 1, abort_flag, a.status,
                                             trc, c_ld))
                                return false;
                            vready = u;
                        }
                        if (!mbar_wait_t(&bars[B_PFULL + h], np[h] & 1, abort_flag, a.status, trc,
                                         c_p))
                            return false;
                        tc_fence_after();
                        const long long ti = trc ? clock64() : 0;
                        const uint32_t vd = dv0 + st * kTileD;
                        const uint32_t acc0 = first[h] ? 0u : 1u;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            // A = P_h in TMEM: 16 keys = 8 columns.  B = V (MN-major):
                            // 16 key rows of 128 bytes (2 KB); the second 64-column half
                            // of D lies 16 KB further (LBO).
                            tc_mma_bf16_ts_lo<kHiMN>(tmem_o + h * kOStride, tmem + h * kBN + kk * 8,
                                                     vd + ((kk * 2048) >> 4), kIdescPV,
                                                     kk > 0 ? 1u : acc0);
                        }
                        first[h] = false;
                        ++np[h];
                        if (u == uhi[h] - 1) tc_commit(&bars[B_ODONE + h]);
                        if (trc) c_is += clock64() - ti;
                        return true;
                    };
                    auto in = [&](int h, int u) { return u >= ulo[h] && u < uhi[h]; };
                    for (int u = 0; ok && u <= nkv; ++u) {
                        if (u < nkv && in(0, u)) ok = issue_qk(0, u);
                        if (ok && u >= 1) {
                            if (in(1, u - 1)) ok = issue_pv(1, u - 1);
                            if (ok) tc_commit(&bars[B_VEMPTY + ((T + u - 1) & 1)]);   // V(u-1) read
                        }
                        if (ok && u < nkv) {
                            if (in(1, u)) ok = issue_qk(1, u);
                            if (ok) tc_commit(&bars[B_KEMPTY + ((T + u) & 1)]);       // K(u) read
                        }
                        if (ok && u < nkv && in(0, u)) ok = issue_pv(0, u);
                    }
                    T += nkv;
#pragma unroll
                    for (int h = 0; h < 2; ++h) iq[h] += (uhi[h] > ulo[h]) ? 1 : 0;
                }
                if (trc) {
                    tr[TR_M_IFULL] = c_if;
                    tr[TR_M_LOADS] = c_ld;
                    tr[TR_M_PFULL] = c_p;
                    tr[TR_M_ISSUE] = c_is;
                    tr[TR_M_TOTAL] = clock64() - t_start;
                    trace_flush(tr, a.trace + (int64_t)blockIdx.x * kTraceSlots, 8, 16);
                }
                // Every MMA this thread issued completes before TMEM is released
                // (already so on the normal path; needed when a wait gave up).
                tc_commit(&bars[B_DRAIN]);
                mbar_wait_until(&bars[B_DRAIN], 0, global_timer_ns() + 500000000ull);
            }
            __syncwarp();
        } else if (MODE == kGroup) {
            // --------------------------- Q loaders: warp 10 + h fills Q_h
            // The group's query rows are gathered from the original Q through
            // pos with 16-byte asynchronous copies (lane: rows lane + 32 i),
            // laid out as the 128-byte-swizzled K-major tile that a TMA load
            // would write: 16-byte unit u of row r at (u / 8) * 16 KB + 128 r
            // + 16 ((u mod 8) xor (r mod 8)).
            const int h = warp - 10;
            int iq = 0;    // query tiles loaded
            bool ok = true;
            for (int k = 0; ok; ++k) {
                if (lane == 0)
                    ok = mbar_wait(&bars[B_IFULL + (k & 1)], (k >> 1) & 1, abort_flag, a.status);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                const int *wi = ring_slot<D>(sm, a.K, k & 1);   // Item fields
                if (wi[15] < 0) break;                           // no more items
                const int wb = wi[0], nkv = wi[4], hd = wi[5 + h], q0 = wi[7 + h];
                const int qend = wi[9 + h], ulo = wi[11 + h], uhi = wi[13 + h];
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_IEMPTY + (k & 1)]);
                if (nkv == 0 || uhi <= ulo) continue;
                int tok[4];    // token of row lane + 32 i, -1 past the group
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = q0 + lane + 32 * i;
                    tok[i] = row < qend ? a.pos[(int64_t)wb * a.rows + row] : -1;
                    if ((unsigned)tok[i] >= (unsigned)a.n) tok[i] = -1;   // never read past Q
                }
                if (iq >= 1 && lane == 0)
                    ok = mbar_wait(&bars[B_QEMPTY + h], (iq - 1) & 1, abort_flag, a.status);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                uint8_t *dq = sQ + h * L::kTile;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i;
                    const uint8_t *src = reinterpret_cast<const uint8_t *>(
                        a.q + (((int64_t)wb * a.n + max(tok[i], 0)) * a.Hq + hd) * D);
                    const uint32_t nb = tok[i] >= 0 ? 16u : 0u;
#pragma unroll
                    for (int u = 0; u < D / 8; ++u)
                        cp_async16(dq + (u >> 3) * 16384 + r * 128 + (((u & 7) ^ (r & 7)) << 4),
                                   src + u * 16, nb);
                }
                cp_async_wait_all();
                fence_proxy_async_smem();     // the MMAs read Q_h through the async proxy
                mbar_arrive(&bars[B_QFULL + h]);
                ++iq;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ---------------------------------------- softmax of half hh = warp / 4
        // Thread t: query row r = t mod 128 of the half (TMEM lane r).
        const int hh = warp >> 2;
        const int r = threadIdx.x & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_off + hh * kBN;        // S_h / P_h of this lane
        const uint32_t o_col = tmem_o + lane_off + hh * kOStride; // O_h of this lane
        const bool trc = a.trace != nullptr && threadIdx.x == 0;
        int T = 0;          // key tiles of earlier items
        int ns = 0;         // S_h tiles consumed
        int nod = 0;        // items of this half with tiles (O_h completions)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            ok = mbar_wait_t(&bars[B_IFULL + slot], (k >> 1) & 1, abort_flag, a.status, trc,
                             tr[TR_S_IFULL]);
            // a warp leaves together: its lanes meet warp-collective instructions
            // (tcgen05.ld/st, votes) next, so one lane's timeout ends them all
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int *wi = ring_slot<D>(sm, a.K, slot);   // the fields of Item
            if (wi[15] < 0) break;                         // no more items
            const int wb = wi[0], wg = wi[1], kv_lo = wi[3], nkv = wi[4];
            const int hd = wi[5 + hh], q0 = wi[7 + hh], qend = wi[9 + hh];
            const int ulo = wi[11 + hh], uhi = wi[13 + hh];
            const int prow = q0 + r;                     // row in the Q tensor
            const bool qvalid = prow < qend;
            int qi = prow;                               // token index of the row
            // kGroup: the groups whose columns this row must not score (the
            // row's groups below the tile's group), and its last key row
            // outside the window.
            int qg[kMaxTopk];          // -1 = unused slot
#pragma unroll
            for (int s = 0; s < kMaxTopk; ++s) {
                qg[s] = -1;
                if (MODE == kGroup && qvalid && s < a.topk) {
                    const int gi = a.gids[((int64_t)wb * a.rows + prow) * a.topk + s];
                    if (gi < wg && (unsigned)gi < (unsigned)a.K)
                        qg[s] = gi;
                }
            }
            const int hib = (MODE == kGroup && qvalid)
                                ? min(prow, a.wlo[(int64_t)wb * a.rows + prow] - 1)
                                : prow;
            if (MODE == kGroup && qvalid && a.pair_count)
                qi = a.pos[(int64_t)wb * a.rows + prow];
            const bool count_ok = (unsigned)qi < (unsigned)a.n;

            float m_ref = -CUDART_INF_F;   // reference max (base 2) applied to O_h and l
            float l = 0.f;                 // row sum
            int cnt = 0;

            for (int u = ulo; u < uhi; ++u) {
                const int t = T + u, st = t & 1;
                const int kvb = kv_lo + kBN * u;         // first key row of the tile
                // ---- the keys of the tile that share an excluded group with the
                // row: the union of the masks of the row's excluded groups
                uint32_t ex[4] = {0u, 0u, 0u, 0u};
                auto fetch_ex = [&]() -> bool {
                    if (!mbar_wait_t(&bars[B_META + st], (t >> 1) & 1, abort_flag, a.status, trc,
                                     tr[TR_S_META]))
                        return false;
                    const uint4 *cb =
                        reinterpret_cast<const uint4 *>(colbits + (size_t)st * a.K * 4);
#pragma unroll
                    for (int x = 0; x < kMaxTopk; ++x) {
                        if (qg[x] >= 0) {
                            const uint4 v = cb[qg[x]];
                            ex[0] |= v.x;
                            ex[1] |= v.y;
                            ex[2] |= v.z;
                            ex[3] |= v.w;
                        }
                    }
                    return true;
                };
                // Once this half has scored tiles t-2 and t-1 of the item, the
                // masks of t-2 have landed (it waited for them), so the phase of
                // t is at most one ahead: fetch the masks before S_h, their
                // latency hidden behind the wait.  For the first two tiles S_h of
                // tile t gives that order instead: the MMA thread issues both
                // P.V of t-2 before either Q.K^T of t, so a softmax has finished
                // t-2 by the time S_h(t) is complete.
                const bool early = MODE == kGroup && u >= ulo + 2;
                ok = !early || fetch_ex();
                if (ok)
                    ok = mbar_wait_t(&bars[B_SFULL + hh], ns & 1, abort_flag, a.status, trc,
                                     tr[TR_S_SFULL]);
                ++ns;
                if (ok && MODE == kGroup && !early) ok = fetch_ex();
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                long long tt = trc ? clock64() : 0;
                float s[128];
                tmem_ld128(s_col, s);
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_SLOAD] += t2 - tt;
                    tt = t2;
                }

                uint32_t okb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t bits;
                    if (!qvalid)
                        bits = 0u;
                    else if (MODE == kGroup)
                        bits = range_bits(0, hib - kvb, 32 * j);   // causal, outside the window
                    else if (MODE == kWindow)
                        bits = range_bits(qi - a.window + 1 - kvb, qi - kvb, 32 * j);
                    else
                        bits = range_bits(0, qi - kvb, 32 * j);
                    okb[j] = bits & ~ex[j];
                }
                if (a.pair_count)
                    cnt += __popc(okb[0]) + __popc(okb[1]) + __popc(okb[2]) + __popc(okb[3]);

                // masked raw scores (no selects where every key of the warp's
                // rows is allowed); the row max over 8 independent chains
                if (!__all_sync(0xffffffffu, (okb[0] & okb[1] & okb[2] & okb[3]) == 0xffffffffu)) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const bool on = (okb[c >> 5] >> (c & 31)) & 1u;
                        s[c] = on ? s[c] : -CUDART_INF_F;
                    }
                }
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
                for (int c = 24; c < 120; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[120 + i]);
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7])) *
                                 a.scale_log2;   // scale > 0, so max(s) * scale = max(s * scale)
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_MASK] += t2 - tt;
                    tt = t2;
                }

                // Lazy rescaling: keep the reference max unless the row max
                // grows by more than 2^8.
                const float m_new = fmaxf(m_ref, mx);
                const bool grow = (m_ref == -CUDART_INF_F) || (m_new > m_ref + 8.f);
                const bool resc = grow && m_ref != -CUDART_INF_F;
                const float new_ref = grow ? m_new : m_ref;
                const float f = resc ? exp2f(m_ref - new_ref) : 1.f;
                const bool any_resc = __any_sync(0xffffffffu, resc);
                m_ref = new_ref;
                const float nref = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;

                // ---- P = 2^(s * scale - ref) in bf16 into TMEM over the first 64
                // columns of S_h (keys 2c, 2c+1 in column c): the A operand of P.V
                const float sc2 = a.scale_log2;
                float rs8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int c = half * 64 + 2 * j;
                        float x0, x1;
                        fma2(x0, x1, s[c], s[c + 1], sc2, nref);
                        const float p0 = exp2f(x0), p1 = exp2f(x1);
                        add2(rs8[2 * (j & 3)], rs8[2 * (j & 3) + 1], p0, p1);
                        pk[j] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32u(s_col + half * 32, pk);
                }
                tmem_st_wait();
                l = fmaf(l, f, ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                                   ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7])));
                if (trc) {
                    const long long t2 = clock64();
                    tr[TR_T_P] += t2 - tt;
                    tt = t2;
                }
                // O_h += P_h(t-1) V(t-1) is complete (it precedes S_h(t) on the
                // tensor pipe), so a rescale needs no wait.
                if (any_resc) {
                    rescale_o<D>(o_col, f);   // warp-wide
                    if (trc) tr[TR_T_RESCALE] += clock64() - tt;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFULL + hh]);
            }
            if (!ok) break;
            T += nkv;

            // ---- epilogue: this half's rows
            const long long t_epi = trc ? clock64() : 0;
            const bool has_tiles = uhi > ulo;
            if (has_tiles) {
                ok = mbar_wait_t(&bars[B_ODONE + hh], nod & 1, abort_flag, a.status, trc,
                                 tr[TR_S_ODONE]);
                ++nod;
                tc_fence_after();
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            long long te = trc ? clock64() : 0;
            const bool has = l > 0.f;
            const float lse2 = has ? m_ref + log2f(l) : -CUDART_INF_F;   // base 2
            const float inv_l = has ? 1.f / l : 0.f;
            // O_h of this row, all D columns in one TMEM load (the tile's score
            // registers are dead here), then its largest |entry| (partials).
            float o[D];
            if (has_tiles) {
                if constexpr (D == 128) {
                    tmem_ld128(o_col, o);
                } else {
                    tmem_ld32(o_col, o);
                    tmem_ld32(o_col + 32, o + 32);
                }
            } else {
#pragma unroll
                for (int e = 0; e < D; ++e) o[e] = 0.f;
            }
            float amax = 0.f;
            if (MODE != kDense) {
                float am8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) am8[i] = 0.f;
#pragma unroll
                for (int e = 0; e < D; ++e) am8[e & 7] = fmaxf(am8[e & 7], fabsf(o[e]));
                amax = fmaxf(fmaxf(fmaxf(am8[0], am8[1]), fmaxf(am8[2], am8[3])),
                             fmaxf(fmaxf(am8[4], am8[5]), fmaxf(am8[6], am8[7]))) *
                       inv_l;
            }
            int64_t orow = 0;
            if (MODE == kGroup)
                orow = ((int64_t)wb * a.rows + prow) * a.Hq + hd;
            else
                orow = ((int64_t)wb * a.n + qi) * a.Hq + hd;
            if (trc) {
                const long long t2 = clock64();
                tr[TR_E_TMEM] += t2 - te;
                te = t2;
            }
            // Partials: O / l in fp16 scaled by a power of two so that the largest
            // entry lies in [2^14, 2^15) (11-bit precision at any magnitude, no
            // overflow), plus {lse (base 2), 2^e}.  Dense: O / l in bf16.
            int ex2 = 0;
            if (amax > 0.f && amax < CUDART_INF_F) frexpf(amax, &ex2);   // amax < 2^ex2
            const float mul = (MODE == kDense) ? inv_l
                                               : inv_l * __int_as_float((127 + 15 - ex2) << 23);
            const float up = __int_as_float((127 - 15 + ex2) << 23);     // 2^(ex2 - 15)
            if (qvalid) {
                if (MODE == kDense) {
                    if (a.lse)
                        a.lse[((int64_t)wb * a.Hq + hd) * a.n + qi] = lse2 * 0.69314718055994531f;
                } else {
                    (MODE == kGroup ? a.part_meta_out : a.win_meta_out)[orow] =
                        make_float2(lse2, up);
                }
            }
            // The row straight from registers, 32 columns at a time; each lane
            // writes its own row.  Partials (workspace rows, 32-byte aligned)
            // go out as 32-byte stores, whole sectors; the dense output as
            // 16-byte stores.
            uint16_t *obase = (MODE == kDense) ? reinterpret_cast<uint16_t *>(a.out)
                              : (MODE == kGroup) ? reinterpret_cast<uint16_t *>(a.part_out16)
                                                 : reinterpret_cast<uint16_t *>(a.win_out16);
            uint16_t *orow_p = obase + orow * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float x0 = o[32 * c + 2 * q] * mul, x1 = o[32 * c + 2 * q + 1] * mul;
                    pk[q] = (MODE == kDense) ? pack_bf16x2(x0, x1) : pack_f16x2(x0, x1);
                }
                if (qvalid) {
                    if (MODE == kDense) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow_p + c * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                                                pk[4 * q + 3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            st_global_v8(orow_p + c * 32 + q * 16, pk + 8 * q);
                    }
                }
            }
            if (trc) tr[TR_E_STORE] += clock64() - te;
            if (qvalid && a.pair_count && hd == 0 && count_ok)
                atomicAdd(&a.pair_count[(int64_t)wb * a.n + qi], cnt);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_IEMPTY + slot]);     // ring slot no longer read
            if (trc) {
                tr[TR_S_EPI] += clock64() - t_epi;
                tr[TR_S_ITEMS] += 1;
                tr[TR_S_TILES] += uhi - ulo;
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
