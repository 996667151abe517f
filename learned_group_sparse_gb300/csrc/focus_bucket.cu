// Group bucketing and the data movement around the group attention kernel.
//
// Bucketing turns the hard top-k memberships (gist.science/zh technical
// summary 2.1.3) into per-group member lists so that "within-group causal
// attention" can run over each group as one dense problem:
//   1. bucket_count    per chunk of 4096 (token, slot) entries, a histogram
//                      of group ids in shared memory;
//   2. bucket_scan     per group, an exclusive scan of the chunk counts;
//   3. bucket_scatter  per chunk, a stable scatter: the block scans the
//                      group sizes into offsets (chunk 0 stores them), then
//                      each warp walks its slice of the chunk in order and
//                      ranks equal ids inside a 32-entry step with
//                      __match_any_sync.
// The plan kernel orders the group kernel's tiles by decreasing cost, the
// gather kernel copies K/V rows into group order (the group kernel copies its
// Q rows itself), and the mask-table kernel writes every key tile's group
// bitmaps.
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "focus_internal.h"

namespace focus {

namespace {

constexpr int kScatterWarps = 8;
constexpr int kWarpSlice = kBucketChunk / kScatterWarps;   // 512 entries per warp

__global__ void bucket_count(const int32_t *__restrict__ ids, int64_t nk, int K, int nchunks,
                             int32_t *__restrict__ counts)
{
    grid_dep_sync();
    extern __shared__ int hist[];
    const int chunk = blockIdx.x, b = blockIdx.y;
    for (int g = threadIdx.x; g < K; g += blockDim.x) hist[g] = 0;
    __syncthreads();
    const int64_t e0 = (int64_t)chunk * kBucketChunk;
    const int64_t e1 = min(e0 + kBucketChunk, nk);
    for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
        const int g = ids[(int64_t)b * nk + e];
        if ((unsigned)g < (unsigned)K) atomicAdd(&hist[g], 1);   // out-of-range ids are dropped
    }
    __syncthreads();
    int32_t *out = counts + ((int64_t)b * nchunks + chunk) * K;
    for (int g = threadIdx.x; g < K; g += blockDim.x) out[g] = hist[g];
}

// blockDim (32, 32): x = group within a tile of 32 groups, y = slice of chunks.
__global__ void bucket_scan(int32_t *__restrict__ counts, int K, int nchunks,
                            int32_t *__restrict__ totals)
{
    grid_dep_sync();
    __shared__ int part[32][33];
    const int tx = threadIdx.x, ty = threadIdx.y, b = blockIdx.y;
    const int g = blockIdx.x * 32 + tx;
    const int per = (nchunks + 31) / 32;
    const int c0 = min(ty * per, nchunks), c1 = min(c0 + per, nchunks);
    int32_t *col = counts + (int64_t)b * nchunks * K + g;
    int sum = 0;
    if (g < K)
        for (int c = c0; c < c1; ++c) sum += col[(int64_t)c * K];
    part[ty][tx] = sum;
    __syncthreads();
    int run = 0;
    for (int y = 0; y < ty; ++y) run += part[y][tx];
    if (g < K) {
        for (int c = c0; c < c1; ++c) {
            const int v = col[(int64_t)c * K];
            col[(int64_t)c * K] = run;
            run += v;
        }
        if (ty == 31) totals[(int64_t)b * K + g] = run;
    }
}

// Exclusive scan of the K <= 1024 group sizes of one batch into soff[0..K]
// (soff[K] = total), by a block of 256 threads: four sizes per thread.
__device__ __forceinline__ void scan_sizes(const int32_t *__restrict__ totals, int K, int *soff)
{
    __shared__ int warp_sum[8];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    int v[4], local = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int g = 4 * t + q;
        v[q] = g < K ? totals[g] : 0;
        local += v[q];
    }
    int x = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sum[w] = x;
    __syncthreads();
    int before = x - local, total = 0;
    for (int i = 0; i < 8; ++i) {
        if (i < w) before += warp_sum[i];
        total += warp_sum[i];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int g = 4 * t + q;
        if (g < K) soff[g] = before;
        before += v[q];
    }
    if (t == 0) soff[K] = total;
    __syncthreads();
}

__global__ void __launch_bounds__(256) bucket_scatter(const int32_t *__restrict__ ids,
                                                      int64_t nk, int K, int topk, int nchunks,
                                                      const int32_t *__restrict__ chunk_base,
                                                      const int32_t *__restrict__ totals,
                                                      int32_t *__restrict__ offsets,
                                                      int32_t *__restrict__ pos,
                                                      int32_t *__restrict__ inv)
{
    grid_dep_sync();
    extern __shared__ int hist[];   // [kScatterWarps][K], then the offsets [K + 1]
    int *soff = hist + kScatterWarps * K;
    const int chunk = blockIdx.x, b = blockIdx.y;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kScatterWarps * K; i += blockDim.x) hist[i] = 0;
    // group offsets of this batch (every block scans the sizes; chunk 0
    // publishes them)
    scan_sizes(totals + (int64_t)b * K, K, soff);
    if (chunk == 0)
        for (int g = threadIdx.x; g <= K; g += blockDim.x)
            offsets[(int64_t)b * (K + 1) + g] = soff[g];
    const int64_t e0 = (int64_t)chunk * kBucketChunk;
    const int64_t s0 = min(e0 + (int64_t)w * kWarpSlice, nk);
    const int64_t s1 = min(s0 + kWarpSlice, nk);
    const int32_t *idb = ids + (int64_t)b * nk;
    for (int64_t e = s0 + lane; e < s1; e += 32) {
        const int g = idb[e];
        if ((unsigned)g < (unsigned)K) atomicAdd(&hist[w * K + g], 1);
    }
    __syncthreads();
    const int32_t *cb = chunk_base + ((int64_t)b * nchunks + chunk) * K;
    for (int g = threadIdx.x; g < K; g += blockDim.x) {
        int run = soff[g] + cb[g];
        for (int x = 0; x < kScatterWarps; ++x) {
            const int t = hist[x * K + g];
            hist[x * K + g] = run;
            run += t;
        }
    }
    __syncthreads();
    int32_t *pb = pos + (int64_t)b * nk;
    int32_t *ib = inv + (int64_t)b * nk;
    const uint32_t lt = (1u << lane) - 1u;
    for (int64_t base = s0; base < s1; base += 32) {
        const int64_t e = base + lane;
        int g = e < s1 ? idb[e] : -1;
        const bool active = (unsigned)g < (unsigned)K;
        if (!active) {
            g = -1 - lane;            // unique, matches no other lane
            if (e < s1) ib[e] = -1;   // an out-of-range id gets no list entry
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, g);
        const int rank = __popc(peers & lt);
        if (active) {
            const int r = hist[w * K + g] + rank;
            pb[r] = (int32_t)(e / topk);
            ib[e] = r;
        }
        __syncwarp();
        if (active && lane == __ffs(peers) - 1) hist[w * K + g] += __popc(peers);
        __syncwarp();
    }
}

// ------------------------------------------------------------------ plan
// Entries of group g: its T_g = ceil(size_g / 128) query tiles, or with
// pair_tiles the ceil(T_g / 2) pairs of consecutive tiles; entry t of a group
// costs t + 1 (tiles) or 2t + 2 (pairs) key tiles.  Emits every (group, t)
// ordered by decreasing t, groups sorted by decreasing entry count inside a
// layer.  One block of 1024 threads; B*K <= 4096.
constexpr int kPlanMax = 4096;

__device__ __forceinline__ int layer_count(const int *keyT, int G, int t)
{
    // number of sorted (descending) entries with T > t
    int lo = 0, hi = G;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (keyT[mid] > t) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ offsets, int B,
                                                    int K, int pair_tiles,
                                                    int2 *__restrict__ tiles,
                                                    int *__restrict__ ntiles)
{
    grid_dep_sync();
    __shared__ int keyT[kPlanMax];
    __shared__ int keyG[kPlanMax];
    __shared__ long long pref[kPlanMax + 1];
    __shared__ long long wsum[32];
    const int G = B * K;
    int Gp = 1;
    while (Gp < G) Gp <<= 1;
    const int tid = threadIdx.x;
    for (int i = tid; i < Gp; i += 1024) {
        if (i < G) {
            const int b = i / K, g = i - b * K;
            const int size = offsets[b * (K + 1) + g + 1] - offsets[b * (K + 1) + g];
            const int qt = (size + 127) / 128;             // query tiles of the group
            keyT[i] = pair_tiles ? (qt + 1) / 2 : qt;      // work entries of the group
            keyG[i] = i;
        } else {
            keyT[i] = -1;
            keyG[i] = 0x7fffffff;
        }
    }
    __syncthreads();
    // bitonic sort: T descending, group index ascending
    for (int k = 2; k <= Gp; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < Gp; i += 1024) {
                const int p = i ^ j;
                if (p > i) {
                    const bool desc_block = (i & k) == 0;
                    const int ti = keyT[i], tp = keyT[p], gi = keyG[i], gp = keyG[p];
                    // "first" = should come earlier in the final order
                    const bool p_first = tp > ti || (tp == ti && gp < gi);
                    if (p_first == desc_block) {
                        keyT[i] = tp;
                        keyT[p] = ti;
                        keyG[i] = gp;
                        keyG[p] = gi;
                    }
                }
            }
            __syncthreads();
        }
    }
    // inclusive prefix sums of T over the sorted order (4 entries per thread)
    long long local[4];
    long long run = 0;
    for (int q = 0; q < 4; ++q) {
        const int i = tid * 4 + q;
        run += (i < G && keyT[i] > 0) ? keyT[i] : 0;
        local[q] = run;
    }
    long long x = run;
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        long long s = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        wsum[lane] = s;
    }
    __syncthreads();
    const long long before = x - run + (w > 0 ? wsum[w - 1] : 0);
    for (int q = 0; q < 4; ++q) {
        const int i = tid * 4 + q;
        if (i < kPlanMax) pref[i + 1] = before + local[q];
    }
    if (tid == 0) pref[0] = 0;
    __syncthreads();
    const long long total = pref[G];
    const int Tmax = G > 0 ? max(keyT[0], 0) : 0;
    if (tid == 0) {
        ntiles[0] = (int)total;
        ntiles[1] = 0;   // work counters of the group and window kernels
        ntiles[2] = 0;
    }
    // S(t) = tiles in layers above t = pref[c(t)] - c(t) * (t + 1)
    for (long long p = tid; p < total; p += 1024) {
        int lo = 0, hi = Tmax - 1;   // smallest t with S(t) <= p
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const int c = layer_count(keyT, G, mid);
            const long long S = pref[c] - (long long)c * (mid + 1);
            if (S <= p) hi = mid;
            else lo = mid + 1;
        }
        const int c = layer_count(keyT, G, lo);
        const long long S = pref[c] - (long long)c * (lo + 1);
        const int rank = (int)(p - S);
        tiles[p] = make_int2(keyG[rank], lo);
    }
}

// ---------------------------------------------------------------- gather
__global__ void __launch_bounds__(256) gather_kernel(
    const uint4 *__restrict__ K, const uint4 *__restrict__ V, const int32_t *__restrict__ pos,
    const int32_t *__restrict__ ids, int B, int n, int64_t nk, int topk, int kvunits,
    uint4 *__restrict__ Kp, uint4 *__restrict__ Vp, int32_t *__restrict__ gidp)
{
    grid_dep_sync();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t total = (int64_t)B * nk;
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < total;
         row += warps) {
        const int64_t b = row / nk;
        const int p = pos[row];
        uint4 *kd = Kp + row * kvunits;
        uint4 *vd = Vp + row * kvunits;
        if ((unsigned)p >= (unsigned)n) {
            // not a token (ids outside [0, K) leave list entries unwritten):
            // an empty row that no group reads, never an out-of-range load
            if (lane < topk) gidp[row * topk + lane] = -1;
            for (int u = lane; u < kvunits; u += 32) kd[u] = vd[u] = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const int64_t src = b * n + p;
        if (lane < topk) gidp[row * topk + lane] = ids[src * topk + lane];
        const uint4 *k = K + src * kvunits;
        const uint4 *v = V + src * kvunits;
        for (int u = lane; u < kvunits; u += 32) {
            kd[u] = k[u];
            vd[u] = v[u];
        }
    }
}

// ---------------------------------------------------------------- mask tables
// Group bitmaps of the group kernel's key tiles, one [K] uint4 entry per
// tile: word j of entry g has bit c set when key row 32 j + c of the tile
// belongs to group g.  The softmax excludes a key by OR-ing the entries of
// the query's groups below the tile's group, so that a pair sharing several
// groups is scored in the lowest of them (the allowed set of the technical
// summary's section 2.1.2 with each shared pair scored once).
//
// Group tiles: 128 consecutive group-order rows from the start of group g,
// tile u at slot floor(off[g] / 128) + g + u.  That slot map needs no scan and
// never overlaps the next group: floor(a + s) - floor(a) + 1 >= ceil(s) for
// a = off[g] / 128, s = size_g / 128.  Slots past a group's last tile are
// never read and are left unwritten.
//
// Window bounds: the window kernel takes every pair with i - j < w, so the
// group kernel takes, of the keys sharing a group with query i, only those
// with i - j >= w.  A group's members are in ascending token order, so for the
// group-order row r of (i, g) those keys are the rows [off[g], wlo[r]), where
// wlo[r] is the first row of the group whose token lies inside i's window
// (r + 1 at w = 0).  Found by a backward galloping search from r: the
// window holds few of a group's members.
__global__ void __launch_bounds__(128) mask_table_kernel(
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ gidp,
    const int32_t *__restrict__ ids, const int32_t *__restrict__ pos,
    const int32_t *__restrict__ inv, int n, int64_t nk, int K, int topk, int window,
    int64_t ntg, int64_t nblk_g, uint4 *__restrict__ tab_g, int32_t *__restrict__ wlo)
{
    grid_dep_sync();
    const int tid = threadIdx.x;
    const int64_t blk = blockIdx.x;
    if (blk >= nblk_g) {
        // window bounds of the rows of tokens [128 t, 128 t + 128)
        const int64_t wb = blk - nblk_g;
        const int64_t ntw = ((int64_t)n + 127) / 128;
        const int64_t b = wb / ntw;
        const int i = (int)(128 * (wb - b * ntw)) + tid;
        if (i >= n) return;
        const int32_t *off = offsets + b * (K + 1);
        const int32_t *pb = pos + b * nk;
        for (int s = 0; s < topk; ++s) {
            const int64_t q = (b * n + i) * topk + s;
            const int g = ids[q];
            const int r = inv[q];
            if ((unsigned)g >= (unsigned)K || (int64_t)(unsigned)r >= nk) continue;
            int t = r + 1;
            if (window > 0) {
                // pb[r] = i > i - w: find the first row m in [off[g], r] with
                // pb[m] > i - w, i.e. lo < m <= hi with pb[lo] <= i - w
                const int thr = i - window, seg = off[g];
                int hi = r, lo = seg - 1;
                for (int64_t step = 1; (int64_t)hi - step >= seg; step <<= 1) {
                    const int m = (int)(hi - step);
                    if (pb[m] <= thr) {
                        lo = m;
                        break;
                    }
                    hi = m;
                }
                while (hi - lo > 1) {
                    const int m = lo + (hi - lo) / 2;
                    if (pb[m] > thr)
                        hi = m;
                    else
                        lo = m;
                }
                t = hi;
            }
            wlo[b * nk + r] = t;
        }
        return;
    }
    extern __shared__ uint32_t bm[];   // [K][4]
    __shared__ int cnt;
    const int64_t b = blk / ntg, slot = blk - b * ntg;
    const int32_t *off = offsets + b * (K + 1);
    // g = the last group whose first slot is <= slot (slots rise with g)
    if (tid == 0) cnt = 0;
    __syncthreads();
    int c = 0;
    for (int g = tid; g < K; g += 128) c += ((int64_t)(off[g] >> 7) + g <= slot) ? 1 : 0;
    if (c) atomicAdd(&cnt, c);
    __syncthreads();
    const int g = cnt - 1;
    const int64_t r0 = off[g] + 128 * (slot - ((off[g] >> 7) + g));
    const int64_t rend = off[g + 1];
    if (r0 >= rend) return;   // not a tile of group g (uniform over the block)
    const int32_t *src = gidp + b * nk * topk;
    uint4 *dst = tab_g + (b * ntg + slot) * K;
    for (int i = tid; i < 4 * K; i += 128) bm[i] = 0u;
    __syncthreads();
    const int64_t row = r0 + tid;
    if (row < rend) {
        for (int s = 0; s < topk; ++s) {
            const int gg = src[row * topk + s];
            if ((unsigned)gg < (unsigned)K) atomicOr(&bm[gg * 4 + (tid >> 5)], 1u << (tid & 31));
        }
    }
    __syncthreads();
    const uint4 *bm4 = reinterpret_cast<const uint4 *>(bm);
    for (int i = tid; i < K; i += 128) dst[i] = bm4[i];
}

}  // namespace

int64_t mask_tiles_group(int n, int K, int topk)
{
    return ((int64_t)n * topk + 127) / 128 + K;
}

cudaError_t launch_mask_tables(const int32_t *offsets, const int32_t *gidp, const int32_t *ids,
                               const int32_t *pos, const int32_t *inv, int B, int n, int K,
                               int topk, int window, uint4 *tab_g, int32_t *wlo, cudaStream_t s,
                               int *launches)
{
    const int64_t nk = (int64_t)n * topk;
    const int64_t ntg = mask_tiles_group(n, K, topk), ntw = ((int64_t)n + 127) / 128;
    const int64_t blocks = (int64_t)B * (ntg + ntw);
    if (n == 0 || blocks <= 0) return cudaSuccess;
    prof_begin("mask_table", s);
    const cudaError_t e = launch_pdl(mask_table_kernel, dim3((unsigned)blocks), dim3(128),
                                     (size_t)K * 16, s, offsets, gidp, ids, pos, inv, n, nk, K,
                                     topk, window, ntg, (int64_t)B * ntg, tab_g, wlo);
    prof_end(s);
    *launches += 1;
    return e;
}

size_t bucket_ws_bytes(int B, int n, int K, int topk)
{
    const int64_t nk = (int64_t)n * topk;
    const int64_t nchunks = (nk + kBucketChunk - 1) / kBucketChunk;
    return sizeof(int32_t) * ((size_t)B * (size_t)(nchunks > 0 ? nchunks : 1) * K + (size_t)B * K) +
           256;
}

cudaError_t launch_bucket(const int32_t *ids, int B, int n, int K, int topk, int32_t *offsets,
                          int32_t *pos, int32_t *inv, void *ws, cudaStream_t s, int *launches)
{
    const int64_t nk = (int64_t)n * topk;
    const int nchunks = (int)((nk + kBucketChunk - 1) / kBucketChunk);
    int32_t *counts = static_cast<int32_t *>(ws);
    int32_t *totals = counts + (size_t)B * (size_t)(nchunks > 0 ? nchunks : 1) * K;
    cudaError_t e;
    if (nchunks == 0)   // no entries: every group is empty
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (size_t)B * (K + 1), s);
    {
        prof_begin("bucket_count", s);
        e = launch_pdl(bucket_count, dim3(nchunks, B), dim3(256), K * sizeof(int), s, ids, nk, K,
                       nchunks, counts);
        prof_end(s);
        if (e != cudaSuccess) return e;
        prof_begin("bucket_scan", s);
        e = launch_pdl(bucket_scan, dim3((K + 31) / 32, B), dim3(32, 32), 0, s, counts, K, nchunks,
                       totals);
        prof_end(s);
        if (e != cudaSuccess) return e;
        *launches += 2;
    }
    {
        const size_t smem = sizeof(int) * ((size_t)kScatterWarps * K + K + 1);
        e = cudaFuncSetAttribute(bucket_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        prof_begin("bucket_scatter", s);
        e = launch_pdl(bucket_scatter, dim3(nchunks, B), dim3(256), smem, s, ids, nk, K, topk,
                       nchunks, counts, totals, offsets, pos, inv);
        prof_end(s);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t *offsets, int B, int K, int pair_tiles, int2 *tiles,
                        int *ntiles, cudaStream_t s, int *launches)
{
    prof_begin("plan", s);
    const cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s, offsets, B, K,
                                     pair_tiles, tiles, ntiles);
    prof_end(s);
    *launches += 1;
    return e;
}

cudaError_t launch_gather(const __nv_bfloat16 *K, const __nv_bfloat16 *V, const int32_t *pos,
                          const int32_t *ids, int B, int n, int topk, int Hkv, int d,
                          __nv_bfloat16 *Kp, __nv_bfloat16 *Vp, int32_t *gidp, cudaStream_t s,
                          int *launches)
{
    const int64_t nk = (int64_t)n * topk;
    const int64_t rows = (int64_t)B * nk;
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 32) blocks = 152 * 32;
    prof_begin("gather", s);
    const cudaError_t e =
        launch_pdl(gather_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                   reinterpret_cast<const uint4 *>(K), reinterpret_cast<const uint4 *>(V), pos, ids,
                   B, n, nk, topk, Hkv * d / 8, reinterpret_cast<uint4 *>(Kp),
                   reinterpret_cast<uint4 *>(Vp), gidp);
    prof_end(s);
    *launches += 1;
    return e;
}

}  // namespace focus

// ------------------------------------------------ allocation-free variant
// focus_bucket_static: the same bucketing for callers that cannot allocate
// device memory at all (see include/focus.h).  Its scratch (the per-chunk
// counts and the group totals) lives in the file-scope device array below
// instead of a caller workspace.  Every GPU that loads the library holds the
// array until the process exits.
namespace focus {

namespace {

constexpr size_t kStaticScratchInts = (size_t)1 << 22;   // 16 MiB of int32
__device__ __align__(256) int32_t g_bucket_scratch[kStaticScratchInts];

constexpr int kMaxDevices = 64;
int32_t *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// The array's name is only a host-side stand-in in host code: the device
// address must come from cudaGetSymbolAddress, looked up once per device
// with that device current.
cudaError_t scratch_address(int32_t **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bucket_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace focus

extern "C" int focus_bucket_static(const int32_t *ids, int B, int n, int K, int topk,
                                   int32_t *offsets, int32_t *pos, int32_t *inv, void *stream)
{
    using namespace focus;
    // the same validation and status codes as focus_bucket
    int st = check_bucket(ids, B, n, K, topk, offsets, pos, inv);
    if (st) return st;
    if (bucket_ws_bytes(B, n, K, topk) > kStaticScratchInts * sizeof(int32_t))
        return 2;   // FOCUS_ERR_UNSUPPORTED: more scratch than the fixed array holds
    int32_t *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return cuda_status(e);
    int launches = 0;
    e = launch_bucket(ids, B, n, K, topk, offsets, pos, inv, scratch,
                      static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) set_last_launches(launches);
    return cuda_status(e);
}
