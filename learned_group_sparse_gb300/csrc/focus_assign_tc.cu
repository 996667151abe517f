// Centroid scoring and hard top-k on the tensor cores (Focus, gist.science/zh
// technical summary 2.1.1 and 2.1.3).
//
// The scores s = (X W_g) C^T are formed as s = X M with M = W_g C^T
// ([hidden, K], fp32, once per call).  X is exactly bf16, so splitting M into
// two bf16 parts M = M_hi + M_lo (residual below 2^-17 of |M|) and running
// tcgen05 bf16 MMAs with fp32 accumulation gives fp32-accurate scores.  The
// two parts are stacked as one B operand [M_hi; M_lo] ([2 Kp, hidden]), so one
// MMA of N = 2 Kp (two of N = Kp when 2 Kp > 256) yields
//   S_hi[128 tokens, Kp] = X_tile . M_hi^T and S_lo = X_tile . M_lo^T
// in TMEM, and the epilogue adds them.
// The epilogue keeps each token's top-(k+1) scores in registers (one thread
// per token = TMEM lane), in descending order with ties to the lower id, and
// writes the ids and the smallest gap between consecutive kept scores.
//
// CTA: warps 0-3 epilogue, warp 4 TMA producer, warp 5 TMEM allocator + MMA.
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"
#include "focus_ptx.cuh"
#include "focus_wait.cuh"
#include "focus_topk.cuh"

namespace focus {

namespace {

constexpr int kTokens = 128;   // tokens per CTA (MMA M)
constexpr int kHK = 64;        // hidden per pipeline stage (one 128-byte swizzle row)

// M^T split: mhi[c][h], mlo[c][h] for c < Kp (rows >= K are zero).  Block:
// 32 centroids x 32 hidden rows, both operands staged in shared memory; lane
// l takes hidden row h0 + l and warp w centroids c0 + w + 8 j, so that a
// warp's stores cover 32 consecutive hidden entries of one centroid row.
__global__ void __launch_bounds__(256) assign_prep_kernel(const float *__restrict__ Wg,
                                                          const float *__restrict__ C,
                                                          int hidden, int dg, int K, int Kp,
                                                          __nv_bfloat16 *__restrict__ mhi,
                                                          __nv_bfloat16 *__restrict__ mlo)
{
    grid_dep_sync();
    extern __shared__ float psm[];
    float *csm = psm;                  // [dg][32]: C rows c0..c0+31, transposed
    float *wsm = psm + 32 * dg;        // [32][dg + 1]: W_g rows h0..h0+31
    const int c0 = blockIdx.y * 32, h0 = blockIdx.x * 32;
#pragma unroll 8   // several loads in flight per thread
    for (int i = threadIdx.x; i < 32 * dg; i += blockDim.x) {
        const int r = i / dg, e = i - r * dg;
        csm[e * 32 + r] = (c0 + r < K) ? C[(int64_t)(c0 + r) * dg + e] : 0.f;
        wsm[r * (dg + 1) + e] = (h0 + r < hidden) ? Wg[(int64_t)(h0 + r) * dg + e] : 0.f;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int e = 0; e < dg; ++e) {
        const float wv = wsm[lane * (dg + 1) + e];   // (dg + 1): no bank conflicts
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = fmaf(wv, csm[e * 32 + w + 8 * j], acc[j]);
    }
    const int h = h0 + lane;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = c0 + w + 8 * j;
        if (c < Kp && h < hidden) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(acc[j]);
            const __nv_bfloat16 lo = __float2bfloat16_rn(acc[j] - __bfloat162float(hi));
            mhi[(int64_t)c * hidden + h] = hi;
            mlo[(int64_t)c * hidden + h] = lo;
        }
    }
}

struct TcArgs {
    int64_t ntok;
    int hidden, K, Kp, topk, stages;
    int32_t *ids;
    float *margin;
    WaitCtl wc;
};

__device__ __forceinline__ uint32_t tc_stage_bytes(int Kp) { return 128u * kTokens + 2u * 128u * Kp; }

// Epilogue for top-NS lists (NS = min(k + 1, K)): this thread's row of
// S_hi + S_lo (the warp-collective TMEM loads are executed by all lanes, even
// after a timeout).
template <int NS>
__device__ __forceinline__ void tc_epilogue(const TcArgs &a, uint32_t tmem, bool ok, int64_t t0)
{
    const int warp = threadIdx.x >> 5;
    const int r = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    TopList<NS> L;
    L.init();
    // the first chunk (min(32, K) >= NS candidates) fills the list; the rest
    // arrive with higher ids than every kept one
#pragma unroll 1
    for (int c0 = 0; c0 < a.Kp; c0 += 32) {
        float v[32], vl[32];
        tmem_ld32(tmem + lane_off + c0, v);
        tmem_ld32(tmem + lane_off + a.Kp + c0, vl);
        if (c0 == 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (e < a.K) L.offer_first(v[e] + vl[e], e);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (c0 + e < a.K) L.offer_next(v[e] + vl[e], c0 + e);
        }
    }
    const int64_t tok = t0 + r;
    if (ok && tok < a.ntok) {
#pragma unroll
        for (int q = 0; q < NS; ++q)
            if (q < a.topk) a.ids[tok * a.topk + q] = L.i[q];
        if (a.margin) a.margin[tok] = L.gap(min(a.topk + 1, a.K));
    }
}

__global__ void __launch_bounds__(192, 2) assign_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const __grid_constant__ CUtensorMap tmM,
                                                           const TcArgs a)
{
    grid_dep_sync();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t stage_bytes = tc_stage_bytes(a.Kp);   // multiple of 1024
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.stages * stage_bytes);
    // bars: full[stages], empty[stages], done, drain
    uint64_t *drain = bars + 2 * a.stages + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * a.stages + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsteps = a.hidden / kHK;
    const int64_t t0 = (int64_t)blockIdx.x * kTokens;
    uint32_t ncols = 32;
    while ((int)ncols < 2 * a.Kp) ncols <<= 1;     // S_hi at column 0, S_lo at column Kp

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&bars[s], 1);
            mbar_init(&bars[a.stages + s], 1);
        }
        mbar_init(&bars[2 * a.stages], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmM);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        if (lane == 0) {
            int k = 0;
            for (; k < nsteps; ++k) {
                const int st = k % a.stages;
                if (k >= a.stages &&
                    !mbar_wait(&bars[a.stages + st], ((k / a.stages) - 1) & 1, abort_flag, a.wc))
                    break;
                uint8_t *base = sm + st * stage_bytes;
                mbar_arrive_expect_tx(&bars[st], stage_bytes);
                tma_load_2d(base, &tmX, &bars[st], k * kHK, (int)t0);
                // [M_hi; M_lo] rows in boxes of up to 256
                for (int r0 = 0; r0 < 2 * a.Kp; r0 += 256)
                    tma_load_2d(base + 128 * kTokens + 128 * r0, &tmM, &bars[st], k * kHK, r0);
            }
            if (*abort_flag) {
                // let the copies of the last issued stages land
                const uint64_t deadline = global_timer_ns() + 200000000ull;
                for (int t = k > a.stages ? k - a.stages : 0; t < k; ++t)
                    mbar_wait_until(&bars[t % a.stages], (t / a.stages) & 1, deadline);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            // one MMA of N = 2 Kp over [M_hi; M_lo], or two of N = Kp
            const bool one = 2 * a.Kp <= 256;
            const uint32_t idesc = idesc_bf16_f32(kTokens, one ? 2 * a.Kp : a.Kp, false, false);
            bool ok = true;
            for (int k = 0; k < nsteps && ok; ++k) {
                const int st = k % a.stages;
                ok = mbar_wait(&bars[st], (k / a.stages) & 1, abort_flag, a.wc);
                if (!ok) break;
                tc_fence_after();
                const uint32_t xa = smem_u32(sm + st * stage_bytes);
                const uint32_t hb = xa + 128 * kTokens;
                const uint32_t lb = hb + 128 * a.Kp;
#pragma unroll
                for (int kk = 0; kk < kHK / 16; ++kk) {
                    const uint64_t ad = sdesc_sw128(xa + kk * 32, 16, 1024);
                    const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
                    tc_mma_bf16(tmem, ad, sdesc_sw128(hb + kk * 32, 16, 1024), idesc, acc);
                    if (!one)
                        tc_mma_bf16(tmem + a.Kp, ad, sdesc_sw128(lb + kk * 32, 16, 1024), idesc,
                                    acc);
                }
                tc_commit(&bars[a.stages + st]);
            }
            if (ok) tc_commit(&bars[2 * a.stages]);
            // every issued MMA completes before TMEM is released
            tc_commit(drain);
            mbar_wait_until(drain, 0, global_timer_ns() + 500000000ull);
        }
        __syncwarp();
    } else {
        // epilogue: thread = token row = TMEM lane
        const bool ok = mbar_wait(&bars[2 * a.stages], 0, abort_flag, a.wc);
        tc_fence_after();
        switch (min(a.topk + 1, a.K)) {
        case 1: tc_epilogue<1>(a, tmem, ok, t0); break;
        case 2: tc_epilogue<2>(a, tmem, ok, t0); break;
        case 3: tc_epilogue<3>(a, tmem, ok, t0); break;
        case 4: tc_epilogue<4>(a, tmem, ok, t0); break;
        case 5: tc_epilogue<5>(a, tmem, ok, t0); break;
        case 6: tc_epilogue<6>(a, tmem, ok, t0); break;
        case 7: tc_epilogue<7>(a, tmem, ok, t0); break;
        case 8: tc_epilogue<8>(a, tmem, ok, t0); break;
        default: tc_epilogue<9>(a, tmem, ok, t0); break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

int assign_tc_kp(int K) { return (K + 15) / 16 * 16; }

}  // namespace

bool assign_tc_supported(int hidden, int K, int topk)
{
    return K <= 256 && hidden % kHK == 0 && topk <= 8;
}

size_t assign_tc_ws_bytes(int hidden, int K)
{
    if (K > 256) return 0;
    return 2 * (size_t)assign_tc_kp(K) * hidden * sizeof(__nv_bfloat16) + 256;
}

cudaError_t assign_tc_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan)
{
    const int Kp = assign_tc_kp(p.K);
    plan->path = 1;
    plan->p = p;
    plan->wc = wc;
    plan->Kp = Kp;
    plan->mhi = ws;   // [M_hi; M_lo]: [2 Kp, hidden]
    const uint32_t stage = 128u * kTokens + 2u * 128u * Kp;
    // Stages within ~110 KB so that two CTAs share an SM: one streams X while
    // the other runs its top-k epilogue.
    int st = (int)(113u * 1024u / stage);
    plan->stages = st > 4 ? 4 : (st < 2 ? 2 : st);
    plan->smem = (size_t)plan->stages * stage + (2 * plan->stages + 2) * 8 + 16 + 1024;
    plan->smem2 = sizeof(float) * ((size_t)32 * p.dg + (size_t)32 * (p.dg + 1));
    plan->grid = (p.ntok + kTokens - 1) / kTokens;
    if (p.ntok > 0 &&
        (!make_map_2d(&plan->map[0], p.X, (uint64_t)p.hidden, (uint64_t)p.ntok, kHK, kTokens,
                      false) ||
         !make_map_2d(&plan->map[1], plan->mhi, (uint64_t)p.hidden, (uint64_t)(2 * Kp), kHK,
                      (uint32_t)(2 * Kp <= 256 ? 2 * Kp : 256), false)))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(assign_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan->smem2);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(assign_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)plan->smem);
}

cudaError_t assign_tc_launch(const AssignPlan &plan, cudaStream_t s, int *launches)
{
    const AssignLaunch &p = plan.p;
    const int Kp = plan.Kp;
    __nv_bfloat16 *mhi = static_cast<__nv_bfloat16 *>(plan.mhi);
    __nv_bfloat16 *mlo = mhi + (size_t)Kp * p.hidden;
    {
        const dim3 grid((unsigned)((p.hidden + 31) / 32), (unsigned)((Kp + 31) / 32));
        prof_begin("assign_prep", s);
        cudaError_t e = launch_pdl(assign_prep_kernel, grid, dim3(256), plan.smem2, s, p.Wg, p.C,
                                   p.hidden, p.dg, p.K, Kp, mhi, mlo);
        prof_end(s);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (p.ntok == 0) return cudaSuccess;
    TcArgs a;
    a.ntok = p.ntok;
    a.hidden = p.hidden;
    a.K = p.K;
    a.Kp = Kp;
    a.topk = p.topk;
    a.stages = plan.stages;
    a.ids = p.ids;
    a.margin = p.margin;
    a.wc = plan.wc;
    prof_begin("assign", s);
    cudaError_t e = launch_pdl(assign_tc_kernel, dim3((unsigned)plan.grid), dim3(192), plan.smem,
                               s, plan.map[0], plan.map[1], a);
    prof_end(s);
    *launches += 1;
    return e;
}

// ----------------------------------------------------------- path choice
int assign_path(int hidden, int dg, int K, int topk)
{
    if (assign_z_supported(hidden, dg, K, topk)) return 2;
    if (assign_tc_supported(hidden, K, topk)) return 1;
    return 0;
}

size_t assign_ws_bytes(int64_t ntok, int hidden, int dg, int K, int topk)
{
    switch (assign_path(hidden, dg, K, topk)) {
    case 2: return assign_z_ws_bytes(ntok, hidden, dg, K);
    case 1: return assign_tc_ws_bytes(hidden, K);
    default: return 0;
    }
}

cudaError_t assign_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan)
{
    switch (assign_path(p.hidden, p.dg, p.K, p.topk)) {
    case 2: return assign_z_prepare(p, ws, wc, plan);
    case 1: return assign_tc_prepare(p, ws, wc, plan);
    default:
        plan->path = 0;
        plan->p = p;
        plan->wc = wc;
        return cudaSuccess;
    }
}

cudaError_t assign_launch(const AssignPlan &plan, cudaStream_t s, int *launches)
{
    switch (plan.path) {
    case 2: return assign_z_launch(plan, s, launches);
    case 1: return assign_tc_launch(plan, s, launches);
    default: return launch_assign(plan.p, s, launches);
    }
}

}  // namespace focus
