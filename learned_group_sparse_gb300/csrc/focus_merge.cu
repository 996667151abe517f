// Log-sum-exp merge of the partial attention results, and the exact count of
// allowed pairs.
//
// The allowed set of query i (gist.science/zh technical summary 2.1.2-2.1.3)
// is split without overlap into the window keys that share no group with i
// (window kernel) and the keys that share a group, each scored in the lowest
// shared group (group kernel).  An exact softmax over the union
// (gist.science/nl Kerncomponent 3) is therefore the base-2 log-sum-exp
// combination of the k + 1 normalised partials:
//   L = log2 sum_p 2^{L_p},  O = sum_p 2^{L_p - L} O_p.
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"

namespace focus {

namespace {

// One block per (b, i); the per-head weights are formed first, then every
// thread combines 8 output values at a time with 16-byte loads.
__global__ void __launch_bounds__(256) merge_kernel(
    const uint4 *__restrict__ Owin, const float *__restrict__ Lwin, const uint4 *__restrict__ Opart,
    const float *__restrict__ Lpart, const int32_t *__restrict__ inv, int n, int64_t nk,
    int topk, int Hq, int d, uint4 *__restrict__ O, float *__restrict__ lse)
{
    extern __shared__ float wts[];   // [Hq][topk + 1]
    __shared__ int rs[8];
    const int64_t tokrow = blockIdx.x;            // b * n + i
    const int64_t b = tokrow / n;
    const int i = (int)(tokrow - b * n);
    const int np = topk + 1;
    if (threadIdx.x < topk) rs[threadIdx.x] = inv[tokrow * topk + threadIdx.x];
    __syncthreads();
    for (int h = threadIdx.x; h < Hq; h += blockDim.x) {
        float l[9];
        l[0] = Lwin[tokrow * Hq + h];
        for (int s = 0; s < topk; ++s)
            l[s + 1] = ((unsigned)rs[s] < (unsigned)nk) ? Lpart[(b * nk + rs[s]) * Hq + h]
                                                        : -CUDART_INF_F;
        float m = -CUDART_INF_F;
        for (int p = 0; p < np; ++p) m = fmaxf(m, l[p]);
        float L = -CUDART_INF_F;
        if (m != -CUDART_INF_F) {
            float sum = 0.f;
            for (int p = 0; p < np; ++p) sum += exp2f(l[p] - m);
            L = m + log2f(sum);
        }
        for (int p = 0; p < np; ++p)
            wts[h * np + p] = (L == -CUDART_INF_F) ? 0.f : exp2f(l[p] - L);
        if (lse) lse[(b * Hq + h) * n + i] = L * 0.69314718055994531f;
    }
    __syncthreads();
    const int units = Hq * d / 8;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        const int h = (u * 8) / d;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int p = 0; p < np; ++p) {
            const float w = wts[h * np + p];
            if (w == 0.f) continue;
            const uint4 raw = (p == 0) ? Owin[tokrow * units + u]
                                       : Opart[(b * nk + rs[p - 1]) * units + u];
            const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] = fmaf(w, __uint_as_float(v[e] << 16), acc[2 * e]);
                acc[2 * e + 1] = fmaf(w, __uint_as_float(v[e] & 0xffff0000u), acc[2 * e + 1]);
            }
        }
        uint4 o;
        __nv_bfloat162 t;
        t = __floats2bfloat162_rn(acc[0], acc[1]);
        o.x = *reinterpret_cast<uint32_t *>(&t);
        t = __floats2bfloat162_rn(acc[2], acc[3]);
        o.y = *reinterpret_cast<uint32_t *>(&t);
        t = __floats2bfloat162_rn(acc[4], acc[5]);
        o.z = *reinterpret_cast<uint32_t *>(&t);
        t = __floats2bfloat162_rn(acc[6], acc[7]);
        o.w = *reinterpret_cast<uint32_t *>(&t);
        O[tokrow * units + u] = o;
    }
}

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
            const int gs = offsets[b * (K + 1) + g];
            for (int rr = gs + lane; rr <= r; rr += 32) {
                const int j = pos[b * nk + rr];
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

cudaError_t launch_merge(const __nv_bfloat16 *Owin, const float *Lwin,
                         const __nv_bfloat16 *Opart, const float *Lpart, const int32_t *inv,
                         int B, int n, int topk, int Hq, int d, __nv_bfloat16 *O, float *lse,
                         cudaStream_t s, int *launches)
{
    const int64_t rows = (int64_t)B * n;
    if (rows == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)Hq * (topk + 1);
    prof_begin("merge", s);
    merge_kernel<<<(unsigned)rows, 256, smem, s>>>(
        reinterpret_cast<const uint4 *>(Owin), Lwin, reinterpret_cast<const uint4 *>(Opart), Lpart,
        inv, n, (int64_t)n * topk, topk, Hq, d, reinterpret_cast<uint4 *>(O), lse);
    prof_end(s);
    *launches += 1;
    return cudaGetLastError();
}

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
