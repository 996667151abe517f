// Log-sum-exp merge of the partial attention results.
//
// The allowed set of query i (gist.science/zh technical summary 2.1.2-2.1.3)
// is split without overlap into the window keys j > i - w (window kernel) and
// the keys sharing a group with j <= i - w, each scored in the lowest shared
// group (group kernel).  The exact softmax over the union
// (gist.science/nl Kerncomponent 3) is the base-2 log-sum-exp combination of
// the k + 1 normalised partials:
//   L = log2 sum_p 2^{L_p},  O = sum_p 2^{L_p - L} O_p.
// Each partial is stored as fp16 O_p 2^-e_p plus {L_p, 2^e_p}.
//
// All heads of a token are contiguous, so every part of a token is one
// contiguous run: merge_bulk_kernel walks the tokens with whole parts brought
// into shared memory by bulk copies, the next token's copies in flight while
// the current one is combined; merge_kernel (one block per token, 16-byte
// loads) serves shapes whose parts do not fit that double buffer.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"
#include "focus_ptx.cuh"
#include "focus_wait.cuh"

namespace focus {

namespace {

__global__ void __launch_bounds__(256) merge_kernel(
    const uint4 *__restrict__ win16, const float2 *__restrict__ win_meta,
    const uint4 *__restrict__ part16, const float2 *__restrict__ part_meta,
    const int32_t *__restrict__ inv, int n, int64_t nk, int topk, int Hq, int d,
    uint4 *__restrict__ O, float *__restrict__ lse)
{
    grid_dep_sync();
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

// Base-2 log-sum-exp weights of the np parts of one head: w_p = 2^(L_p - L) * s_p
// where {L_p, s_p} are the parts' {lse, scale}; returns L.
__device__ __forceinline__ float part_weights(const float2 *meta, int np, float *wts)
{
    float l[9], sc[9];
#pragma unroll
    for (int p = 0; p < 9; ++p) {
        l[p] = -CUDART_INF_F;
        sc[p] = 0.f;
        if (p < np) {
            l[p] = meta[p].x;
            sc[p] = meta[p].y;
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
        if (p < np) wts[p] = (L == -CUDART_INF_F) ? 0.f : exp2f(l[p] - L) * sc[p];
    return L;
}

// Shared memory of one token in merge_bulk_kernel: np fp16 part rows
// (Hq * d * 2 bytes each), then np meta rows (Hq float2 each).
__host__ __device__ inline uint32_t bulk_token_bytes(int np, int Hq, int d)
{
    return (uint32_t)np * ((uint32_t)Hq * d * 2u + (uint32_t)Hq * 8u);
}

__global__ void __launch_bounds__(256) merge_bulk_kernel(
    const uint4 *__restrict__ win16, const float2 *__restrict__ win_meta,
    const uint4 *__restrict__ part16, const float2 *__restrict__ part_meta,
    const int32_t *__restrict__ inv, int n, int64_t nk, int64_t ntok, int topk, int Hq, int d,
    uint4 *__restrict__ O, float *__restrict__ lse, const WaitCtl wc)
{
    grid_dep_sync();
    extern __shared__ __align__(16) uint8_t msm[];
    __shared__ uint64_t bar[2];
    __shared__ int present[2][9];      // part p of the token in buffer b was copied
    __shared__ volatile int abort_flag;
    float *wts = reinterpret_cast<float *>(msm);                    // [Hq][np]
    const int np = topk + 1;
    const uint32_t rowb = (uint32_t)Hq * d * 2u, metab = (uint32_t)Hq * 8u;
    uint8_t *buf0 = msm + (((uint32_t)Hq * np * 4u + 15u) & ~15u);
    const uint32_t tokb = bulk_token_bytes(np, Hq, d);
    const int units = Hq * d / 8;
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // thread 0: the copies of token tok into buffer b
    auto issue = [&](int64_t tok, int b) {
        const int64_t bb = tok / n;
        uint8_t *base = buf0 + (size_t)b * tokb;
        int64_t rows[9];
        uint32_t bytes = 0;
#pragma unroll
        for (int p = 0; p < 9; ++p) {
            rows[p] = -1;
            if (p == 0) rows[p] = tok;
            else if (p < np) {
                const int r = inv[tok * topk + (p - 1)];
                rows[p] = ((unsigned)r < (unsigned)nk) ? bb * nk + r : -1;
            }
            if (p < np) {
                present[b][p] = rows[p] >= 0;
                if (rows[p] >= 0) bytes += rowb + metab;
            }
        }
        fence_proxy_async_smem();   // earlier generic reads of the buffer come first
        mbar_arrive_expect_tx(&bar[b], bytes);
#pragma unroll
        for (int p = 0; p < 9; ++p) {
            if (p < np && rows[p] >= 0) {
                const uint8_t *src = (p == 0) ? reinterpret_cast<const uint8_t *>(win16)
                                              : reinterpret_cast<const uint8_t *>(part16);
                const uint8_t *msrc = (p == 0) ? reinterpret_cast<const uint8_t *>(win_meta)
                                               : reinterpret_cast<const uint8_t *>(part_meta);
                bulk_load(base + (size_t)p * rowb, src + (size_t)rows[p] * rowb, rowb, &bar[b]);
                bulk_load(base + (size_t)np * rowb + (size_t)p * metab,
                          msrc + (size_t)rows[p] * metab, metab, &bar[b]);
            }
        }
    };
    // thread 0: parity of the copies in flight into buffer 0 / 1 (-1: none)
    int pend0 = -1, pend1 = -1;
    int64_t tok = blockIdx.x;
    if (threadIdx.x == 0 && tok < ntok) {
        issue(tok, 0);
        pend0 = 0;
    }
    for (int k = 0; tok < ntok; ++k, tok += gridDim.x) {
        const int b = k & 1;
        const int64_t next = tok + gridDim.x;
        if (threadIdx.x == 0 && next < ntok) {
            issue(next, b ^ 1);
            (b ? pend0 : pend1) = ((k + 1) >> 1) & 1;
        }
        // every thread waits for this token's copies (bounded); the block
        // leaves together if any wait gave up
        if (!__syncthreads_and(mbar_wait(&bar[b], (k >> 1) & 1, &abort_flag, wc))) break;
        (b ? pend1 : pend0) = -1;
        const uint8_t *base = buf0 + (size_t)b * tokb;
        const float2 *meta = reinterpret_cast<const float2 *>(base + (size_t)np * rowb);
        const int64_t bb = tok / n;
        const int i = (int)(tok - bb * n);
        for (int h = threadIdx.x; h < Hq; h += blockDim.x) {
            float2 mh[9];
#pragma unroll
            for (int p = 0; p < 9; ++p)
                mh[p] = (p < np && present[b][p]) ? meta[p * Hq + h]
                                                  : make_float2(-CUDART_INF_F, 0.f);
            const float L = part_weights(mh, np, wts + h * np);
            if (lse) lse[(bb * Hq + h) * n + i] = L * 0.69314718055994531f;
        }
        __syncthreads();
        const uint4 *parts = reinterpret_cast<const uint4 *>(base);
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int h = (u * 8) / d;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
            for (int p = 0; p < 9; ++p) {
                if (p >= np) break;
                const float w = wts[h * np + p];
                if (w == 0.f) continue;
                const uint4 raw = parts[(size_t)p * units + u];
                const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(hv[e]);
                    acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
                    acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
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
            O[tok * units + u] = o;
        }
        __syncthreads();   // buffer b and the weights are free again
    }
    // A block that gave up lets its copies in flight land before it exits.
    if (abort_flag && threadIdx.x == 0) {
        const uint64_t deadline = global_timer_ns() + 100000000ull;
        if (pend0 >= 0) mbar_wait_until(&bar[0], (uint32_t)pend0, deadline);
        if (pend1 >= 0) mbar_wait_until(&bar[1], (uint32_t)pend1, deadline);
    }
}

}  // namespace

cudaError_t launch_merge(const __half *win16, const float2 *win_meta, const __half *part16,
                         const float2 *part_meta, const int32_t *inv, int B, int n, int topk,
                         int Hq, int d, __nv_bfloat16 *O, float *lse, const WaitCtl &wc,
                         cudaStream_t s, int *launches)
{
    const int64_t rows = (int64_t)B * n;
    if (rows == 0) return cudaSuccess;
    const int np = topk + 1;
    const size_t bulk_smem = (((size_t)Hq * np * 4 + 15) & ~(size_t)15) +
                             2 * (size_t)bulk_token_bytes(np, Hq, d);
    if ((Hq * 8) % 16 == 0 && bulk_smem <= 100 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(merge_bulk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bulk_smem);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        const int per_sm = (int)(220u * 1024u / (bulk_smem + 1024));
        int64_t blocks = (int64_t)sms * (per_sm < 1 ? 1 : per_sm);
        if (blocks > rows) blocks = rows;
        prof_begin("merge", s);
        e = launch_pdl(merge_bulk_kernel, dim3((unsigned)blocks), dim3(256), bulk_smem, s,
                       reinterpret_cast<const uint4 *>(win16), win_meta,
                       reinterpret_cast<const uint4 *>(part16), part_meta, inv, n,
                       (int64_t)n * topk, rows, topk, Hq, d, reinterpret_cast<uint4 *>(O), lse,
                       wc);
        prof_end(s);
        *launches += 1;
        return e;
    }
    const size_t smem = sizeof(float) * (size_t)Hq * (topk + 1);
    prof_begin("merge", s);
    const cudaError_t e = launch_pdl(
        merge_kernel, dim3((unsigned)rows), dim3(256), smem, s,
        reinterpret_cast<const uint4 *>(win16), win_meta, reinterpret_cast<const uint4 *>(part16),
        part_meta, inv, n, (int64_t)n * topk, topk, Hq, d, reinterpret_cast<uint4 *>(O), lse);
    prof_end(s);
    *launches += 1;
    return e;
}

}  // namespace focus
