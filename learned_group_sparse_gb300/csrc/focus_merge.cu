// Log-sum-exp merge of the partial attention results.
//
// The allowed set of query i (gist.science/zh technical summary 2.1.2-2.1.3)
// is split without overlap into the window keys that share no group with i
// (window kernel) and the keys sharing a group, each scored in the lowest
// shared group (group kernel).  The exact softmax over the union
// (gist.science/nl Kerncomponent 3) is the base-2 log-sum-exp combination of
// the k + 1 normalised partials:
//   L = log2 sum_p 2^{L_p},  O = sum_p 2^{L_p - L} O_p.
// Each partial is stored as fp16 O_p 2^-e_p plus {L_p, 2^e_p}.
//
// One block per token; all heads of a token are contiguous, so every part is
// read as one contiguous run of 16-byte vectors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"

namespace focus {

namespace {

__global__ void __launch_bounds__(256) merge_kernel(
    const uint4 *__restrict__ win16, const float2 *__restrict__ win_meta,
    const uint4 *__restrict__ part16, const float2 *__restrict__ part_meta,
    const int32_t *__restrict__ inv, int n, int64_t nk, int topk, int Hq, int d,
    uint4 *__restrict__ O, float *__restrict__ lse)
{
    extern __shared__ float wts[];   // [Hq][topk + 1]
    __shared__ int64_t rows[8];
    const int64_t tokrow = blockIdx.x;            // b * n + i
    const int64_t b = tokrow / n;
    const int i = (int)(tokrow - b * n);
    const int np = topk + 1;
    if (threadIdx.x < topk) {
        const int r = inv[tokrow * topk + threadIdx.x];
        rows[threadIdx.x] = ((unsigned)r < (unsigned)nk) ? b * nk + r : -1;
    }
    __syncthreads();
    for (int h = threadIdx.x; h < Hq; h += blockDim.x) {
        float l[9], sc[9];
        const float2 mw = win_meta[tokrow * Hq + h];
        l[0] = mw.x;
        sc[0] = mw.y;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            l[s + 1] = -CUDART_INF_F;
            sc[s + 1] = 0.f;
            if (s < topk && rows[s] >= 0) {
                const float2 mp = part_meta[rows[s] * Hq + h];
                l[s + 1] = mp.x;
                sc[s + 1] = mp.y;
            }
        }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int p = 0; p < 9; ++p) m = fmaxf(m, l[p]);
        float L = -CUDART_INF_F;
        if (m != -CUDART_INF_F) {
            float sum = 0.f;
#pragma unroll
            for (int p = 0; p < 9; ++p) sum += exp2f(l[p] - m);   // absent parts add 0
            L = m + log2f(sum);
        }
#pragma unroll
        for (int p = 0; p < 9; ++p)
            if (p < np) wts[h * np + p] = (L == -CUDART_INF_F) ? 0.f : exp2f(l[p] - L) * sc[p];
        if (lse) lse[(b * Hq + h) * n + i] = L * 0.69314718055994531f;
    }
    __syncthreads();
    const int units = Hq * d / 8;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        const int h = (u * 8) / d;
        // all parts' 16-byte vectors are loaded before any is used, so that
        // the loads of a unit are in flight together
        uint4 raw[9];
        float wp[9];
#pragma unroll
        for (int p = 0; p < 9; ++p) {
            wp[p] = p < np ? wts[h * np + p] : 0.f;
            raw[p] = make_uint4(0u, 0u, 0u, 0u);
            if (wp[p] != 0.f)
                raw[p] = (p == 0) ? win16[tokrow * units + u] : part16[rows[p - 1] * units + u];
        }
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int p = 0; p < 9; ++p) {
            const __half2 *hv = reinterpret_cast<const __half2 *>(&raw[p]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(hv[e]);
                acc[2 * e] = fmaf(wp[p], f.x, acc[2 * e]);
                acc[2 * e + 1] = fmaf(wp[p], f.y, acc[2 * e + 1]);
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

}  // namespace

cudaError_t launch_merge(const __half *win16, const float2 *win_meta, const __half *part16,
                         const float2 *part_meta, const int32_t *inv, int B, int n, int topk,
                         int Hq, int d, __nv_bfloat16 *O, float *lse, cudaStream_t s,
                         int *launches)
{
    const int64_t rows = (int64_t)B * n;
    if (rows == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)Hq * (topk + 1);
    prof_begin("merge", s);
    merge_kernel<<<(unsigned)rows, 256, smem, s>>>(
        reinterpret_cast<const uint4 *>(win16), win_meta, reinterpret_cast<const uint4 *>(part16),
        part_meta, inv, n, (int64_t)n * topk, topk, Hq, d, reinterpret_cast<uint4 *>(O), lse);
    prof_end(s);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace focus
