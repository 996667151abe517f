// Sinkhorn normalisation of token-group affinities, the training-time
// assignment (Focus, gist.science/nl Kerncomponenten 2: group balance as a
// hard structural constraint instead of a loss; gist.science/zh technical
// summary 2.1.1: Sinkhorn in place of softmax, every group receiving an
// equal mass of tokens).
//
// For each sequence b: kernel A_ic = exp(S_ic / tau) over n tokens and K
// groups, target masses 1 per token and n / K per group.  A round is the
// Sinkhorn-Knopp row update then the column update,
//     u_i = 1 / sum_c A_ic v_c,        v_c = (n / K) / sum_i A_ic u_i,
// from v = 1; after the last round P = diag(u) A diag(v).
//
// One pass over S per round: sinkhorn_sweep_kernel gives each warp whole
// rows (coalesced, the row's K values spread over the lanes), forms
// x_ic = S_ic / tau + log v_c in base 2, the row's log-sum-exp and so log u_i,
// and adds the row-normalised entries 2^(x_ic + log u_i) (each at most 1: no
// overflow, and no second exponential) into per-lane column masses; the
// CTA's column masses go to a partial per CTA.  sinkhorn_reduce_kernel sums
// the partials per column and moves log v by log(n/K) - log(mass) (the mass
// was taken with the old v).  sinkhorn_out_kernel writes P and the
// potentials in natural log.  HBM-bound: one read of S per round, one read
// of S and one write of P at the end.
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "focus_internal.h"
#include "focus_ptx.cuh"
#include "focus_wait.cuh"

namespace focus {

namespace {

constexpr int kSkWarps = 8;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkMaxK = 1024;
constexpr int kSkBulkWarps = 16;             // warps of the bulk-copy sweep
constexpr int kSkBulkThreads = kSkBulkWarps * 32;
constexpr int kSkStages = 3;                 // stages of the bulk-copy sweep
constexpr int kSkStageBytes = 64 * 1024;     // rows of S per stage: kSkStageBytes / (4 K)
static_assert(kSkBulkWarps * kSkMaxK * 4 <= kSkStageBytes, "warp column masses fit a stage");

struct SkArgs {
    const float *S;          // [B, n, K]
    int B, n, K, ctas;       // ctas: CTAs per sequence in the sweep
    float k2;                // log2(e) / tau
    float *u2;               // [B, n]    log2 u
    float *v2;               // [B, K]    log2 v
    float *part;             // [B, ctas, K] column masses per CTA
    WaitCtl wc;              // bounded waits of the bulk-copy sweep
};

// One round's row update and column masses.  PER = columns per lane.
template <int PER>
__global__ void __launch_bounds__(kSkThreads) sinkhorn_sweep_kernel(const SkArgs a)
{
    grid_dep_sync();
    __shared__ float vs[kSkMaxK];
    __shared__ float cm[kSkWarps][kSkMaxK];
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K;
    for (int c = tid; c < K; c += kSkThreads) vs[c] = a.v2[(int64_t)b * K + c];
    __syncthreads();
    float vl[PER], col[PER];
#pragma unroll
    for (int t = 0; t < PER; ++t) {
        const int c = lane + 32 * t;
        vl[t] = c < K ? vs[c] : 0.f;
        col[t] = 0.f;
    }
    const float *Sb = a.S + (int64_t)b * a.n * K;
    const int stride = gridDim.x * kSkWarps;
    // R rows of a warp in flight at once (about 32 loads per lane)
    constexpr int R = PER >= 32 ? 1 : 32 / PER > 8 ? 8 : 32 / PER;
    for (int i0 = blockIdx.x * kSkWarps + warp; i0 < a.n; i0 += R * stride) {
        float x[R][PER];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = i0 + r * stride;
            const float *row = Sb + (int64_t)i * K;
#pragma unroll
            for (int t = 0; t < PER; ++t) {
                const int c = lane + 32 * t;
                x[r][t] = (i < a.n && c < K) ? fmaf(row[c], a.k2, vl[t]) : -CUDART_INF_F;
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = i0 + r * stride;
            if (i >= a.n) break;   // warp-uniform
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int t = 0; t < PER; ++t) mx = fmaxf(mx, x[r][t]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            float sum = 0.f;
#pragma unroll
            for (int t = 0; t < PER; ++t) {
                x[r][t] = exp2f(x[r][t] - mx);   // 0 for the lanes past K
                sum += x[r][t];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            const float inv = 1.f / sum;
            if (lane == 0) a.u2[(int64_t)b * a.n + i] = -(mx + log2f(sum));
#pragma unroll
            for (int t = 0; t < PER; ++t) col[t] = fmaf(x[r][t], inv, col[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < PER; ++t) {
        const int c = lane + 32 * t;
        if (c < K) cm[warp][c] = col[t];
    }
    __syncthreads();
    for (int c = tid; c < K; c += kSkThreads) {
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kSkWarps; ++w) m += cm[w][c];
        a.part[((int64_t)b * a.ctas + blockIdx.x) * K + c] = m;
    }
}

// The same round with S streamed through shared memory (K % 4 == 0, so that
// every row starts on a 16-byte boundary): CTA x of sequence b takes chunks
// x, x + ctas, ... of RC = kSkStageBytes / (4 K) consecutive rows, one bulk
// copy per chunk into a ring of kSkStages stages (thread 0 issues; all
// threads wait on the stage's barrier, vote at a CTA barrier on whether a wait
// ran out, and release the stage at a second CTA barrier).  LPR lanes share a
// row (32 LPR >= K), so a warp takes 32 / LPR rows at once and a row's max
// and sum need log2(LPR) shuffles for all of them together; a lane reads
// 16-byte groups 4 (j + LPR t) of its row (j its place in the row's lanes),
// eight lanes covering 128 contiguous bytes.  For K a power of two from 32
// up, a stage is exactly one row per lane group of every warp.
template <int LPR>
__global__ void __launch_bounds__(kSkBulkThreads, 1) sinkhorn_sweep_bulk_kernel(const SkArgs a)
{
    constexpr int T = 8;               // 16-byte groups per lane and row
    constexpr int RPW = 32 / LPR;      // rows per warp at once
    grid_dep_sync();
    extern __shared__ __align__(128) uint8_t skm[];   // kSkStages x kSkStageBytes
    __shared__ __align__(16) float vs[kSkMaxK];
    // after the last stage, stage 0 holds the warps' column masses
    float(*cm)[kSkMaxK] = reinterpret_cast<float(*)[kSkMaxK]>(skm);
    __shared__ __align__(8) uint64_t full[kSkStages];
    __shared__ int abort_flag;
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane / LPR, j = lane % LPR;
    const int K = a.K;
    const int RC = kSkStageBytes / (4 * K);
    const int nchunks = (a.n + RC - 1) / RC;
    const int mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / a.ctas + 1 : 0;
    const float *Sb = a.S + (int64_t)b * a.n * K;
    if (tid < kSkStages) mbar_init(&full[tid], 1);
    if (tid == 0) abort_flag = 0;
    for (int c = tid; c < kSkMaxK; c += kSkBulkThreads)
        vs[c] = c < K ? a.v2[(int64_t)b * K + c] : 0.f;
    mbar_fence_init();
    __syncthreads();
    auto arm = [&](int k) {   // chunk k of this CTA into stage k % kSkStages
        const int jc = blockIdx.x + k * a.ctas;
        const int r0 = jc * RC, cnt = min(RC, a.n - r0);
        uint64_t *bar = &full[k % kSkStages];
        mbar_arrive_expect_tx(bar, (uint32_t)(cnt * K * 4));
        bulk_load(skm + (k % kSkStages) * kSkStageBytes, Sb + (int64_t)r0 * K,
                  (uint32_t)(cnt * K * 4), bar);
    };
    if (tid == 0)
        for (int k = 0; k < kSkStages && k < mine; ++k) arm(k);
    float4 vl[T], col[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const int c0 = 4 * (j + LPR * t);
        vl[t] = c0 < K ? *reinterpret_cast<const float4 *>(vs + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
        col[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int k = 0;
    for (; k < mine; ++k) {
        const int st = k % kSkStages;
        const bool ok = mbar_wait(&full[st], (uint32_t)(k / kSkStages) & 1u, &abort_flag, a.wc);
        if (__syncthreads_or(!ok)) break;   // the whole CTA leaves together
        const int r0 = (blockIdx.x + k * a.ctas) * RC, cnt = min(RC, a.n - r0);
        const float *stage = reinterpret_cast<const float *>(skm + st * kSkStageBytes);
        for (int rr0 = warp * RPW; rr0 < cnt; rr0 += kSkBulkWarps * RPW) {
            const int rr = rr0 + grp;
            const bool live = rr < cnt;
            float4 x[T];
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const int c0 = 4 * (j + LPR * t);
                if (live && c0 < K) {
                    const float4 sv = *reinterpret_cast<const float4 *>(stage + rr * K + c0);
                    x[t].x = fmaf(sv.x, a.k2, vl[t].x);
                    x[t].y = fmaf(sv.y, a.k2, vl[t].y);
                    x[t].z = fmaf(sv.z, a.k2, vl[t].z);
                    x[t].w = fmaf(sv.w, a.k2, vl[t].w);
                } else {
                    x[t] = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
                }
                mx = fmaxf(mx, fmaxf(fmaxf(x[t].x, x[t].y), fmaxf(x[t].z, x[t].w)));
            }
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (!live) mx = 0.f;   // keeps exp2 of the -inf padding at 0, never NaN
            float sum = 0.f;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                x[t].x = exp2f(x[t].x - mx);
                x[t].y = exp2f(x[t].y - mx);
                x[t].z = exp2f(x[t].z - mx);
                x[t].w = exp2f(x[t].w - mx);
                sum += (x[t].x + x[t].y) + (x[t].z + x[t].w);
            }
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (live) {
                const float inv = 1.f / sum;
                if (j == 0) a.u2[(int64_t)b * a.n + r0 + rr] = -(mx + log2f(sum));
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    col[t].x = fmaf(x[t].x, inv, col[t].x);
                    col[t].y = fmaf(x[t].y, inv, col[t].y);
                    col[t].z = fmaf(x[t].z, inv, col[t].z);
                    col[t].w = fmaf(x[t].w, inv, col[t].w);
                }
            }
        }
        __syncthreads();   // every warp is done with the stage
        if (tid == 0 && k + kSkStages < mine) arm(k + kSkStages);
    }
    if (abort_flag) {
        // a wait ran out: let the copies in flight land, then leave (the
        // status word holds the timeout)
        if (tid == 0) {
            const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
            const int armed = min(mine, k + kSkStages);
            for (int q = k; q < armed; ++q)
                mbar_wait_until(&full[q % kSkStages], (uint32_t)(q / kSkStages) & 1u, deadline);
        }
        return;
    }
    // the warp's lanes with the same place j in their rows hold the same
    // columns: sum them, then one lane per column writes the warp's masses
#pragma unroll
    for (int t = 0; t < T; ++t) {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            col[t].x += __shfl_xor_sync(0xffffffffu, col[t].x, off);
            col[t].y += __shfl_xor_sync(0xffffffffu, col[t].y, off);
            col[t].z += __shfl_xor_sync(0xffffffffu, col[t].z, off);
            col[t].w += __shfl_xor_sync(0xffffffffu, col[t].w, off);
        }
        const int c0 = 4 * (j + LPR * t);
        if (grp == 0 && c0 < K) *reinterpret_cast<float4 *>(&cm[warp][c0]) = col[t];
    }
    __syncthreads();
    for (int c = tid; c < K; c += kSkBulkThreads) {
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kSkBulkWarps; ++w) m += cm[w][c];
        a.part[((int64_t)b * a.ctas + blockIdx.x) * K + c] = m;
    }
}

// P and log u through the same bulk-copy ring (K % 4 == 0): each lane turns
// its 16-byte groups of a row into P and stores them as 16-byte words.
template <int LPR>
__global__ void __launch_bounds__(kSkBulkThreads, 1) sinkhorn_out_bulk_kernel(
    const SkArgs a, float *__restrict__ P, float *__restrict__ log_u)
{
    constexpr int T = 8;
    constexpr int RPW = 32 / LPR;
    grid_dep_sync();
    extern __shared__ __align__(128) uint8_t skm[];
    __shared__ __align__(16) float vs[kSkMaxK];
    __shared__ __align__(8) uint64_t full[kSkStages];
    __shared__ int abort_flag;
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane / LPR, j = lane % LPR;
    const int K = a.K;
    const int RC = kSkStageBytes / (4 * K);
    const int nchunks = (a.n + RC - 1) / RC;
    const int mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / a.ctas + 1 : 0;
    const float *Sb = a.S + (int64_t)b * a.n * K;
    if (tid < kSkStages) mbar_init(&full[tid], 1);
    if (tid == 0) abort_flag = 0;
    for (int c = tid; c < kSkMaxK; c += kSkBulkThreads)
        vs[c] = c < K ? a.v2[(int64_t)b * K + c] : 0.f;
    mbar_fence_init();
    __syncthreads();
    auto arm = [&](int k) {
        const int jc = blockIdx.x + k * a.ctas;
        const int r0 = jc * RC, cnt = min(RC, a.n - r0);
        uint64_t *bar = &full[k % kSkStages];
        mbar_arrive_expect_tx(bar, (uint32_t)(cnt * K * 4));
        bulk_load(skm + (k % kSkStages) * kSkStageBytes, Sb + (int64_t)r0 * K,
                  (uint32_t)(cnt * K * 4), bar);
    };
    if (tid == 0)
        for (int k = 0; k < kSkStages && k < mine; ++k) arm(k);
    float4 vl[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const int c0 = 4 * (j + LPR * t);
        vl[t] = c0 < K ? *reinterpret_cast<const float4 *>(vs + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int k = 0;
    for (; k < mine; ++k) {
        const int st = k % kSkStages;
        const bool ok = mbar_wait(&full[st], (uint32_t)(k / kSkStages) & 1u, &abort_flag, a.wc);
        if (__syncthreads_or(!ok)) break;   // the whole CTA leaves together
        const int r0 = (blockIdx.x + k * a.ctas) * RC, cnt = min(RC, a.n - r0);
        const float *stage = reinterpret_cast<const float *>(skm + st * kSkStageBytes);
        for (int rr0 = warp * RPW; rr0 < cnt; rr0 += kSkBulkWarps * RPW) {
            const int rr = rr0 + grp;
            if (rr < cnt) {
                const int64_t row = (int64_t)b * a.n + r0 + rr;
                const float u = a.u2[row];
                if (log_u && j == 0) log_u[row] = u * 0.69314718055994531f;
                if (P) {
                    float *out = P + row * K;
#pragma unroll
                    for (int t = 0; t < T; ++t) {
                        const int c0 = 4 * (j + LPR * t);
                        if (c0 < K) {
                            const float4 sv = *reinterpret_cast<const float4 *>(stage + rr * K + c0);
                            float4 pv;
                            pv.x = exp2f(fmaf(sv.x, a.k2, u + vl[t].x));
                            pv.y = exp2f(fmaf(sv.y, a.k2, u + vl[t].y));
                            pv.z = exp2f(fmaf(sv.z, a.k2, u + vl[t].z));
                            pv.w = exp2f(fmaf(sv.w, a.k2, u + vl[t].w));
                            __stcs(reinterpret_cast<float4 *>(out + c0), pv);
                        }
                    }
                }
            }
        }
        __syncthreads();   // every warp is done with the stage
        if (tid == 0 && k + kSkStages < mine) arm(k + kSkStages);
    }
    if (abort_flag && tid == 0) {
        const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
        const int armed = min(mine, k + kSkStages);
        for (int q = k; q < armed; ++q)
            mbar_wait_until(&full[q % kSkStages], (uint32_t)(q / kSkStages) & 1u, deadline);
    }
}

// Column update: log2 v_c += log2(n / K) - log2(sum of the CTAs' masses).  A
// mass that underflows float is taken as the smallest subnormal.  Block
// (32 columns, sequence b): warp w sums the partials w, w + 8, ...
__global__ void __launch_bounds__(kSkThreads) sinkhorn_reduce_kernel(const SkArgs a,
                                                                     float *__restrict__ log_v)
{
    grid_dep_sync();
    __shared__ float red[kSkWarps][32];
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float m = 0.f;
    if (c < a.K) {
        const float *pp = a.part + (int64_t)b * a.ctas * a.K + c;
#pragma unroll 8
        for (int j = warp; j < a.ctas; j += kSkWarps) m += pp[(int64_t)j * a.K];
    }
    red[warp][lane] = m;
    __syncthreads();
    if (warp == 0 && c < a.K) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kSkWarps; ++w) tot += red[w][lane];
        const float lm = tot > 0.f ? log2f(tot) : -149.f;
        const float v = a.v2[(int64_t)b * a.K + c] + (log2f((float)a.n / (float)a.K) - lm);
        a.v2[(int64_t)b * a.K + c] = v;
        if (log_v) log_v[(int64_t)b * a.K + c] = v * 0.69314718055994531f;
    }
}

// P_ic = 2^(S_ic log2(e) / tau + log2 u_i + log2 v_c); log u in natural log.
template <int PER>
__global__ void __launch_bounds__(kSkThreads) sinkhorn_out_kernel(const SkArgs a,
                                                                  float *__restrict__ P,
                                                                  float *__restrict__ log_u)
{
    grid_dep_sync();
    __shared__ float vs[kSkMaxK];
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K;
    for (int c = tid; c < K; c += kSkThreads) vs[c] = a.v2[(int64_t)b * K + c];
    __syncthreads();
    const int stride = gridDim.x * kSkWarps;
    constexpr int R = PER >= 32 ? 1 : 32 / PER > 8 ? 8 : 32 / PER;
    for (int i0 = blockIdx.x * kSkWarps + warp; i0 < a.n; i0 += R * stride) {
        float u[R], x[R][PER];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = i0 + r * stride;
            u[r] = i < a.n ? a.u2[(int64_t)b * a.n + i] : 0.f;
            const float *row = a.S + ((int64_t)b * a.n + i) * K;
#pragma unroll
            for (int t = 0; t < PER; ++t) {
                const int c = lane + 32 * t;
                x[r][t] = (P && i < a.n && c < K) ? row[c] : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int i = i0 + r * stride;
            if (i >= a.n) break;   // warp-uniform
            if (log_u && lane == 0) log_u[(int64_t)b * a.n + i] = u[r] * 0.69314718055994531f;
            if (!P) continue;
            float *out = P + ((int64_t)b * a.n + i) * K;
#pragma unroll
            for (int t = 0; t < PER; ++t) {
                const int c = lane + 32 * t;
                if (c < K) out[c] = exp2f(fmaf(x[r][t], a.k2, u[r] + vs[c]));
            }
        }
    }
}

// lanes per row of the bulk sweep: the smallest power of two with 32 LPR >= K
inline int sinkhorn_lpr(int K)
{
    int l = 1;
    while (32 * l < K) l <<= 1;
    return l;
}

cudaError_t sinkhorn_bulk_sweep(const SkArgs &a, cudaStream_t s)
{
    const dim3 grid((unsigned)a.ctas, (unsigned)a.B);
    const size_t smem = (size_t)kSkStages * kSkStageBytes;
    switch (sinkhorn_lpr(a.K)) {
    case 1: return launch_pdl(sinkhorn_sweep_bulk_kernel<1>, grid, dim3(kSkBulkThreads), smem, s, a);
    case 2: return launch_pdl(sinkhorn_sweep_bulk_kernel<2>, grid, dim3(kSkBulkThreads), smem, s, a);
    case 4: return launch_pdl(sinkhorn_sweep_bulk_kernel<4>, grid, dim3(kSkBulkThreads), smem, s, a);
    case 8: return launch_pdl(sinkhorn_sweep_bulk_kernel<8>, grid, dim3(kSkBulkThreads), smem, s, a);
    case 16:
        return launch_pdl(sinkhorn_sweep_bulk_kernel<16>, grid, dim3(kSkBulkThreads), smem, s, a);
    default:
        return launch_pdl(sinkhorn_sweep_bulk_kernel<32>, grid, dim3(kSkBulkThreads), smem, s, a);
    }
}

cudaError_t sinkhorn_bulk_out(const SkArgs &a, float *P, float *log_u, cudaStream_t s)
{
    const dim3 grid((unsigned)a.ctas, (unsigned)a.B), blk(kSkBulkThreads);
    const size_t smem = (size_t)kSkStages * kSkStageBytes;
    switch (sinkhorn_lpr(a.K)) {
    case 1: return launch_pdl(sinkhorn_out_bulk_kernel<1>, grid, blk, smem, s, a, P, log_u);
    case 2: return launch_pdl(sinkhorn_out_bulk_kernel<2>, grid, blk, smem, s, a, P, log_u);
    case 4: return launch_pdl(sinkhorn_out_bulk_kernel<4>, grid, blk, smem, s, a, P, log_u);
    case 8: return launch_pdl(sinkhorn_out_bulk_kernel<8>, grid, blk, smem, s, a, P, log_u);
    case 16: return launch_pdl(sinkhorn_out_bulk_kernel<16>, grid, blk, smem, s, a, P, log_u);
    default: return launch_pdl(sinkhorn_out_bulk_kernel<32>, grid, blk, smem, s, a, P, log_u);
    }
}

template <int PER>
cudaError_t sinkhorn_launch_t(const SkArgs &a, int iters, float *P, float *log_u, float *log_v,
                              cudaStream_t s, int *launches)
{
    cudaError_t e = cudaSuccess;
    const dim3 grid((unsigned)a.ctas, (unsigned)a.B);
    const dim3 rgrid((unsigned)((a.K + 31) / 32), (unsigned)a.B);
    const bool bulk = a.K % 4 == 0;
    for (int t = 0; t < iters && e == cudaSuccess; ++t) {
        prof_begin("sinkhorn_sweep", s);
        if (bulk)
            e = sinkhorn_bulk_sweep(a, s);
        else
            e = launch_pdl(sinkhorn_sweep_kernel<PER>, grid, dim3(kSkThreads), 0, s, a);
        prof_end(s);
        if (e != cudaSuccess) break;
        prof_begin("sinkhorn_reduce", s);
        e = launch_pdl(sinkhorn_reduce_kernel, rgrid, dim3(kSkThreads), 0, s, a,
                       t + 1 == iters ? log_v : static_cast<float *>(nullptr));
        prof_end(s);
        *launches += 2;
    }
    if (e == cudaSuccess && (P || log_u)) {
        const int rows = (a.n + kSkWarps - 1) / kSkWarps;
        const int octas = min((4 * 152 + a.B - 1) / a.B, rows);
        prof_begin("sinkhorn_out", s);
        if (bulk && P)
            e = sinkhorn_bulk_out(a, P, log_u, s);
        else
            e = launch_pdl(sinkhorn_out_kernel<PER>, dim3((unsigned)octas, (unsigned)a.B),
                           dim3(kSkThreads), 0, s, a, P, log_u);
        prof_end(s);
        *launches += 1;
    }
    return e;
}

// The bulk sweep's dynamic shared memory (once per process and lane count).
cudaError_t sinkhorn_preflight(int K)
{
    static std::once_flag once[6];
    static cudaError_t err[6];
    const int lpr = sinkhorn_lpr(K);
    const int idx = lpr == 1 ? 0 : lpr == 2 ? 1 : lpr == 4 ? 2 : lpr == 8 ? 3 : lpr == 16 ? 4 : 5;
    std::call_once(once[idx], [&] {
        const int bytes = kSkStages * kSkStageBytes;
        const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
#define FOCUS_SK_ATTR(L)                                                              \
    (cudaFuncSetAttribute(sinkhorn_sweep_bulk_kernel<L>, at, bytes) != cudaSuccess        \
         ? cudaErrorInvalidValue                                                          \
         : cudaFuncSetAttribute(sinkhorn_out_bulk_kernel<L>, at, bytes))
        switch (idx) {
        case 0: err[0] = FOCUS_SK_ATTR(1); break;
        case 1: err[1] = FOCUS_SK_ATTR(2); break;
        case 2: err[2] = FOCUS_SK_ATTR(4); break;
        case 3: err[3] = FOCUS_SK_ATTR(8); break;
        case 4: err[4] = FOCUS_SK_ATTR(16); break;
        default: err[5] = FOCUS_SK_ATTR(32); break;
        }
#undef FOCUS_SK_ATTR
    });
    return err[idx];
}

}  // namespace

int sinkhorn_ctas(int B, int n, int K)
{
    if (K % 4 == 0) {
        // bulk-copy sweep: one CTA per SM of 152 over the batch, at least
        // one chunk of rows each
        const int rc = kSkStageBytes / (4 * K);
        const int chunks = (n + rc - 1) / rc;
        const int want = (152 + B - 1) / B;
        return want < chunks ? want : chunks;
    }
    // about four CTAs per SM over the batch, at least one row per warp
    const int want = (4 * 152 + B - 1) / B;
    const int rows = (n + kSkWarps - 1) / kSkWarps;
    return want < rows ? want : (rows < 1 ? 1 : rows);
}

size_t sinkhorn_ws_bytes(int B, int n, int K)
{
    const size_t a256 = 255;
    const size_t v = ((size_t)B * K * 4 + a256) & ~a256;
    const size_t u = ((size_t)B * n * 4 + a256) & ~a256;
    const size_t p = ((size_t)B * sinkhorn_ctas(B, n, K) * K * 4 + a256) & ~a256;
    return v + u + p;
}

cudaError_t launch_sinkhorn(const float *S, int B, int n, int K, float tau, int iters, float *P,
                            float *log_u, float *log_v, void *ws, const WaitCtl &wc,
                            cudaStream_t s, int *launches)
{
    const size_t a256 = 255;
    uint8_t *w = static_cast<uint8_t *>(ws);
    SkArgs a;
    a.S = S;
    a.B = B;
    a.n = n;
    a.K = K;
    a.ctas = sinkhorn_ctas(B, n, K);
    a.k2 = 1.4426950408889634f / tau;
    a.wc = wc;
    a.v2 = reinterpret_cast<float *>(w);
    w += ((size_t)B * K * 4 + a256) & ~a256;
    a.u2 = reinterpret_cast<float *>(w);
    w += ((size_t)B * n * 4 + a256) & ~a256;
    a.part = reinterpret_cast<float *>(w);
    cudaError_t e = sinkhorn_preflight(K);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.v2, 0, (size_t)B * K * 4, s);   // v = 1
    if (e != cudaSuccess) return e;
    if (K <= 32) return sinkhorn_launch_t<1>(a, iters, P, log_u, log_v, s, launches);
    if (K <= 64) return sinkhorn_launch_t<2>(a, iters, P, log_u, log_v, s, launches);
    if (K <= 128) return sinkhorn_launch_t<4>(a, iters, P, log_u, log_v, s, launches);
    if (K <= 256) return sinkhorn_launch_t<8>(a, iters, P, log_u, log_v, s, launches);
    if (K <= 512) return sinkhorn_launch_t<16>(a, iters, P, log_u, log_v, s, launches);
    return sinkhorn_launch_t<32>(a, iters, P, log_u, log_v, s, launches);
}

}  // namespace focus
