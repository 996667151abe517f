// Exact count of the allowed pairs of Focus attention (the work the method
// does, for effective-FLOP accounting and the "every pair scored once"
// check).  The allowed set of query i (gist.science/zh technical summary
// 2.1.2-2.1.3) is the window keys plus the keys sharing a group with i.
#include <stdint.h>

#include "focus_internal.h"

namespace focus {

namespace {

// One warp per query token: counts, over the token's group lists, the keys
// it shares a group with (each counted in the lowest shared group) and how
// many of those lie inside the window; |A_i| = min(w, i+1) - near + share.
__global__ void __launch_bounds__(256) count_kernel(
    const int32_t *__restrict__ ids, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ pos, const int32_t *__restrict__ inv, int B, int n, int K,
    int topk, int window, int64_t *__restrict__ per_query, unsigned long long *__restrict__ totals)
{
    const int lane = threadIdx.x & 31;
    const int64_t nk = (int64_t)n * topk;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t tokrow = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         tokrow < (int64_t)B * n; tokrow += warps) {
        const int64_t b = tokrow / n;
        const int i = (int)(tokrow - b * n);
        const int32_t *gi = ids + tokrow * topk;
        long long share = 0, near = 0;
        for (int s = 0; s < topk; ++s) {
            const int g = gi[s];
            const int r = inv[tokrow * topk + s];
            if ((unsigned)g >= (unsigned)K || (unsigned)r >= (unsigned)nk) continue;
            const int gs = offsets[b * (K + 1) + g];
            for (int rr = gs + lane; rr <= r; rr += 32) {
                const int j = pos[b * nk + rr];
                if ((unsigned)j >= (unsigned)n) continue;
                const int32_t *gj = ids + (b * n + j) * topk;
                bool owned = true;
                for (int x = 0; x < topk && owned; ++x) {
                    if (gi[x] >= g) continue;
                    for (int y = 0; y < topk; ++y)
                        if (gj[y] == gi[x]) owned = false;
                }
                if (owned) {
                    share += 1;
                    if (i - j < window) near += 1;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            share += __shfl_xor_sync(0xffffffffu, share, off);
            near += __shfl_xor_sync(0xffffffffu, near, off);
        }
        if (lane == 0) {
            const long long win = window < i + 1 ? window : i + 1;
            const long long tot = win - near + share;
            if (per_query) per_query[tokrow] = tot;
            atomicAdd(&totals[0], (unsigned long long)tot);
            atomicAdd(&totals[1], (unsigned long long)share);
        }
    }
}

}  // namespace

cudaError_t launch_count_pairs(const int32_t *ids, const int32_t *offsets, const int32_t *pos,
                               const int32_t *inv, int B, int n, int K, int topk, int window,
                               int64_t *per_query, int64_t *totals, cudaStream_t s,
                               int *launches)
{
    cudaError_t e = cudaMemsetAsync(totals, 0, 2 * sizeof(int64_t), s);
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)B * n;
    if (rows == 0) return cudaSuccess;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 64) blocks = 152 * 64;
    prof_begin("count_pairs", s);
    count_kernel<<<(unsigned)blocks, 256, 0, s>>>(ids, offsets, pos, inv, B, n, K, topk, window,
                                                  per_query,
                                                  reinterpret_cast<unsigned long long *>(totals));
    prof_end(s);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace focus
