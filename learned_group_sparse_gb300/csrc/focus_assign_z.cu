// Centroid scoring in the pages' own order when there are more centroids than
// centroid dimensions (Focus, gist.science/zh technical summary 2.1.1: hidden
// states are projected into centroid space, then scored against every
// centroid; 2.1.3: at inference a token joins its k best groups).
//
//   z = x W_g   (d_g values per token),   s_c = z . C_c,   top-k of s.
//
// For K > d_g this is cheaper than s = x (W_g C^T): the long contraction over
// the hidden size runs with N = d_g instead of N = K.  Two kernels:
//
//  assign_z_gemm   persistent tcgen05 GEMM Z = X W_g.  A CTA takes 256 tokens
//                  (two 128-row MMA tiles) per step of its loop, so that each
//                  W_g stage brought into shared memory feeds both tiles; W_g
//                  (fp32) is split into two bf16 parts W_hi + W_lo and both
//                  are accumulated into one fp32 TMEM accumulator (X is exact
//                  in bf16, so the product is fp32-accurate).  TMEM holds two
//                  such accumulators, so the epilogue of one step overlaps the
//                  next step's MMAs.  The epilogue scales each row of Z by a
//                  power of two 2^-e that puts its largest |z| in
//                  [2^14, 2^15), splits it into fp16 hi + lo parts (22-bit
//                  significand at any magnitude) and writes them with 2^e.
//  assign_z_score  persistent: S = Z C^T as three fp16 tcgen05 products
//                  Z_hi C_hi + Z_hi C_lo + Z_lo C_hi (fp32 accumulation), with
//                  C resident in shared memory, and the per-token top-(k+1)
//                  epilogue (one thread per token = TMEM lane).  The ranking is
//                  unchanged by the row's power-of-two scale; the margin is
//                  scaled back.
//
// CTA of both kernels: warps 0-3 epilogue, warp 4 TMA producer, warp 5 TMEM
// allocator + MMA issuer.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"
#include "focus_ptx.cuh"
#include "focus_wait.cuh"
#include "focus_topk.cuh"

namespace focus {

namespace {

constexpr int kZTok = 128;     // tokens per MMA tile (M)
constexpr int kZHK = 64;       // hidden per pipeline stage (one 128-byte swizzle row)
constexpr int kZSel = 9;       // top-(k+1), k <= 8
constexpr int kZEpiWarps = 8;  // two per TMEM lane quarter, each half of the columns

// WT [2 dgp][hidden] bf16: row d < dgp = bf16 hi part of column d of W_g,
// row dgp + d = its lo part (zero rows for d >= d_g).  CH [2 Kp][dgp] fp16:
// row c < Kp = hi part of centroid c, row Kp + c = its lo part (zero past K
// and past d_g).  Blocks [0, nwt): 32 x 32 transpose tiles of W_g; the rest:
// 256 entries of C each.
__global__ void __launch_bounds__(256) assign_z_prep_kernel(const float *__restrict__ Wg,
                                                            const float *__restrict__ C,
                                                            int hidden, int dg, int dgp, int K,
                                                            int Kp, __nv_bfloat16 *__restrict__ WT,
                                                            __half *__restrict__ CH)
{
    grid_dep_sync();
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int th = hidden / 32;
    const int nwt = th * (dgp / 32);
    if ((int)blockIdx.x < nwt) {
        const int h0 = (blockIdx.x % th) * 32, d0 = (blockIdx.x / th) * 32;
        for (int y = ty; y < 32; y += 8) {
            const int d = d0 + tx;
            tile[y][tx] = d < dg ? Wg[(int64_t)(h0 + y) * dg + d] : 0.f;
        }
        __syncthreads();
        for (int y = ty; y < 32; y += 8) {
            const float v = tile[tx][y];   // W_g[h0 + tx][d0 + y]
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            WT[(int64_t)(d0 + y) * hidden + h0 + tx] = hi;
            WT[(int64_t)(dgp + d0 + y) * hidden + h0 + tx] = lo;
        }
    } else {
        const int64_t i = (int64_t)(blockIdx.x - nwt) * 256 + threadIdx.x;
        if (i < (int64_t)Kp * dgp) {
            const int c = (int)(i / dgp), d = (int)(i - (int64_t)c * dgp);
            const float v = (c < K && d < dg) ? C[(int64_t)c * dg + d] : 0.f;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            CH[(int64_t)c * dgp + d] = hi;
            CH[(int64_t)(Kp + c) * dgp + d] = lo;
        }
    }
}

struct ZGemmArgs {
    int64_t ntok;
    int hidden, dgp, stages;
    __half *Z;        // [ntok][2 dgp]: fp16 hi part, then lo part, of z * 2^-e
    float *zscale;    // [ntok]: 2^e
    WaitCtl wc;
};

// One stage: X rows of the two token tiles [128 x 64] bf16 (16 KB each), then
// W_hi and W_lo [dgp x 64] bf16.
__host__ __device__ inline uint32_t z_stage_bytes(int dgp) { return 32768u + 256u * (uint32_t)dgp; }

__global__ void __launch_bounds__(192, 1) assign_z_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                                                               const __grid_constant__ CUtensorMap tmW,
                                                               const ZGemmArgs a)
{
    grid_dep_sync();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int S = a.stages, dgp = a.dgp;
    const uint32_t SB = z_stage_bytes(dgp);   // multiple of 1024
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + S * SB);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;       // [2] accumulator buffer b complete
    uint64_t *tempty = tfull + 2;      // [2] accumulator buffer b read by the epilogue
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsteps = a.hidden / kZHK;
    const int64_t nsup = (a.ntok + 2 * kZTok - 1) / (2 * kZTok);
    uint32_t ncols = 32;
    while ((int)ncols < 4 * dgp) ncols <<= 1;   // buffer b, tile t at column (2 b + t) dgp

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);   // one lane per epilogue warp
        }
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
        tma_prefetch_desc(&tmW);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int64_t g = 0;   // stage loads issued
            bool ok = true;
            for (int64_t j = blockIdx.x; ok && j < nsup; j += gridDim.x) {
                const int row0 = (int)(j * 2 * kZTok);
                for (int k = 0; k < nsteps; ++k, ++g) {
                    const int st = (int)(g % S);
                    if (g >= S &&
                        !(ok = mbar_wait(&empty[st], (uint32_t)((g / S) - 1) & 1u, abort_flag,
                                         a.wc)))
                        break;
                    uint8_t *base = sm + (size_t)st * SB;
                    mbar_arrive_expect_tx(&full[st], SB);
                    tma_load_2d(base, &tmX, &full[st], k * kZHK, row0);
                    tma_load_2d(base + 16384, &tmX, &full[st], k * kZHK, row0 + kZTok);
                    tma_load_2d(base + 32768, &tmW, &full[st], k * kZHK, 0);
                    tma_load_2d(base + 32768 + 128 * dgp, &tmW, &full[st], k * kZHK, dgp);
                }
            }
            if (!ok) {
                // let the copies of the last S issued stages land
                const uint64_t deadline = global_timer_ns() + 200000000ull;
                for (int64_t t = g > S ? g - S : 0; t < g; ++t)
                    mbar_wait_until(&full[t % S], (uint32_t)(t / S) & 1u, deadline);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kZTok, dgp, false, false);
            int64_t g = 0;
            int jj = 0;        // steps of this CTA
            bool ok = true;
            for (int64_t j = blockIdx.x; ok && j < nsup; j += gridDim.x, ++jj) {
                const int b = jj & 1;
                if (jj >= 2 &&
                    !(ok = mbar_wait(&tempty[b], (uint32_t)((jj >> 1) - 1) & 1u, abort_flag,
                                     a.wc)))
                    break;
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)(2 * b * dgp);
                for (int k = 0; k < nsteps; ++k, ++g) {
                    const int st = (int)(g % S);
                    if (!(ok = mbar_wait(&full[st], (uint32_t)(g / S) & 1u, abort_flag, a.wc)))
                        break;
                    tc_fence_after();
                    const uint32_t xa = smem_u32(sm + (size_t)st * SB);
                    const uint32_t wh = xa + 32768, wl = wh + 128 * dgp;
#pragma unroll
                    for (int kk = 0; kk < kZHK / 16; ++kk) {
                        const uint64_t bh = sdesc_sw128(wh + kk * 32, 16, 1024);
                        const uint64_t bl = sdesc_sw128(wl + kk * 32, 16, 1024);
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint64_t ad = sdesc_sw128(xa + t * 16384 + kk * 32, 16, 1024);
                            const uint32_t dt = d0 + (uint32_t)(t * dgp);
                            tc_mma_bf16(dt, ad, bh, idesc, (k > 0 || kk > 0) ? 1u : 0u);
                            tc_mma_bf16(dt, ad, bl, idesc, 1u);
                        }
                    }
                    tc_commit(&empty[st]);
                }
                if (ok) tc_commit(&tfull[b]);
            }
            // every issued MMA completes before TMEM is released
            tc_commit(drain);
            mbar_wait_until(drain, 0, global_timer_ns() + 500000000ull);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int r = threadIdx.x;   // TMEM lane = row of each tile
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int jj = 0;
        for (int64_t j = blockIdx.x; j < nsup; j += gridDim.x, ++jj) {
            const int b = jj & 1;
            // warp-uniform: tcgen05.ld below is warp-collective
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&tfull[b], (uint32_t)(jj >> 1) & 1u, abort_flag, a.wc)))
                break;
            tc_fence_after();
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const int64_t row = j * 2 * kZTok + t * kZTok + r;
                const uint32_t col = tmem + lane_off + (uint32_t)((2 * b + t) * dgp);
                // the row's largest |z| (first pass over TMEM)
                float amax = 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < dgp; c0 += 32) {
                    float v[32];
                    tmem_ld32(col + c0, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
                }
                int ex = 0;
                if (amax > 0.f && amax < CUDART_INF_F) frexpf(amax, &ex);   // amax < 2^ex
                ex = max(ex, -100);   // keeps both scale factors normal floats
                const float down = __int_as_float((127 + 15 - ex) << 23);   // 2^(15 - ex)
                // second pass: scaled rows into fp16 hi + lo
                uint16_t *zrow = reinterpret_cast<uint16_t *>(a.Z) + row * 2 * dgp;
#pragma unroll 1
                for (int c0 = 0; c0 < dgp; c0 += 32) {
                    float v[32];
                    tmem_ld32(col + c0, v);
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float x0 = v[2 * q] * down, x1 = v[2 * q + 1] * down;
                        const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
                        hi[q] = (uint32_t)__half_as_ushort(h0) |
                                ((uint32_t)__half_as_ushort(h1) << 16);
                        lo[q] = pack_f16x2(x0 - __half2float(h0), x1 - __half2float(h1));
                    }
                    if (row < a.ntok) {
                        st_global_v8(zrow + c0, hi);
                        st_global_v8(zrow + c0 + 16, hi + 8);
                        st_global_v8(zrow + dgp + c0, lo);
                        st_global_v8(zrow + dgp + c0 + 16, lo + 8);
                    }
                }
                if (row < a.ntok) a.zscale[row] = __int_as_float((127 - 15 + ex) << 23);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

struct ZScoreArgs {
    int64_t ntok;
    int K, Kp, dgp, topk, stages;
    const float *zscale;
    int32_t *ids;
    float *margin;
    WaitCtl wc;
};

// Shared memory: C_hi / C_lo as [dgp / 64 chunks][2 Kp rows][128 B], then the
// Z stages, each one 64-column chunk of Z_hi and Z_lo of a token tile
// ([128 x 64] fp16, 16 KB each), then the lists that the second warp of a lane
// quarter hands to the first ([2 tiles][128 rows][kZSel] scores and ids).
__host__ __device__ inline uint32_t zs_c_bytes(int Kp, int dgp) { return 4u * (uint32_t)Kp * dgp; }
constexpr uint32_t kZsStage = 32768u;
constexpr uint32_t kZsMerge = 2u * 128u * kZSel * 8u;

// The scoring epilogue for top-NS lists (NS = min(k + 1, K)).  Warp w takes
// the rows of TMEM lane quarter w mod 4 over half w / 4 of the columns; the
// second half's lists go through shared memory to the first, which merges
// them (its ids are the lower ones, so equal scores keep its entry) and
// writes the ids and the margin.
template <int NS>
__device__ __forceinline__ void z_score_epilogue(const ZScoreArgs &a, uint32_t tmem,
                                                 uint64_t *tfull, uint64_t *tempty,
                                                 volatile int *abort_flag, float *xs, int *xi,
                                                 int64_t ntiles)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int nch = (a.Kp + 31) / 32, nch0 = (nch + 1) / 2;
    const int cb = hf ? 32 * nch0 : 0, ce = hf ? 32 * nch : 32 * nch0;
    const int nsel = min(a.topk + 1, a.K);
    int jj = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++jj) {
        const int b = jj & 1;
        const bool ok = mbar_wait(&tfull[b], (uint32_t)(jj >> 1) & 1u, abort_flag, a.wc);
        // the two warps of the quarter leave together: they meet at a named
        // barrier below, and tcgen05.ld is warp-collective
        if (!named_bar_and(1 + q4, 64, ok)) break;
        tc_fence_after();
        TopList<NS> L;
        L.init();
        const uint32_t col = tmem + lane_off + (uint32_t)(b * a.Kp);
        // the first chunk (at least NS candidates) fills the list; the rest
        // arrive with higher ids than every kept one
        {
            float v[32];
            tmem_ld32(col + cb, v);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (cb + e < a.K) L.offer_first(v[e], cb + e);
        }
#pragma unroll 1
        for (int c0 = cb + 32; c0 < ce; c0 += 32) {
            float v[32];
            tmem_ld32(col + c0, v);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (c0 + e < a.K) L.offer_next(v[e], c0 + e);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        float *ps = xs + ((size_t)b * 128 + r) * kZSel;
        int *pi = xi + ((size_t)b * 128 + r) * kZSel;
        if (hf) {
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                ps[q] = L.s[q];
                pi[q] = L.i[q];
            }
        }
        named_bar_sync(1 + q4, 64);
        if (!hf) {
            L.merge(ps, pi);
            const int64_t tok = t * kZTok + r;
            if (tok < a.ntok) {
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    if (q < a.topk) a.ids[tok * a.topk + q] = L.i[q];
                if (a.margin) a.margin[tok] = L.gap(nsel) * a.zscale[tok];   // the row's 2^e
            }
        }
    }
}

__global__ void __launch_bounds__(320, 1) assign_z_score_kernel(const __grid_constant__ CUtensorMap tmZ,
                                                                const __grid_constant__ CUtensorMap tmC,
                                                                const ZScoreArgs a)
{
    grid_dep_sync();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int S = a.stages, Kp = a.Kp, dgp = a.dgp;
    const int nchunk = dgp / 64;
    const uint32_t CB = zs_c_bytes(Kp, dgp);          // multiple of 1024
    uint8_t *sC = sm;
    uint8_t *sZ = sm + CB;
    float *xs = reinterpret_cast<float *>(sZ + (size_t)S * kZsStage);
    int *xi = reinterpret_cast<int *>(xs + 2 * 128 * kZSel);
    uint64_t *full = reinterpret_cast<uint64_t *>(xi + 2 * 128 * kZSel);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *cbar = tempty + 2;
    uint64_t *drain = cbar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (a.ntok + kZTok - 1) / kZTok;
    uint32_t ncols = 32;
    while ((int)ncols < 2 * Kp) ncols <<= 1;   // buffer b at column b Kp

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kZEpiWarps);
        }
        mbar_init(cbar, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kZEpiWarps + 1) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    if (warp == kZEpiWarps && lane == 0) {
        tma_prefetch_desc(&tmZ);
        tma_prefetch_desc(&tmC);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kZEpiWarps) {
        if (lane == 0) {
            // C once: chunk c holds rows [0, 2 Kp) of columns [64 c, 64 c + 64)
            mbar_arrive_expect_tx(cbar, CB);
            for (int c = 0; c < nchunk; ++c) {
                uint8_t *dst = sC + (size_t)c * 2 * Kp * 128;
                tma_load_2d(dst, &tmC, cbar, c * 64, 0);
                tma_load_2d(dst + (size_t)Kp * 128, &tmC, cbar, c * 64, Kp);
            }
            int64_t g = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                for (int c = 0; c < nchunk; ++c, ++g) {
                    const int st = (int)(g % S);
                    if (g >= S &&
                        !(ok = mbar_wait(&empty[st], (uint32_t)((g / S) - 1) & 1u, abort_flag,
                                         a.wc)))
                        break;
                    uint8_t *base = sZ + (size_t)st * kZsStage;
                    mbar_arrive_expect_tx(&full[st], kZsStage);
                    tma_load_2d(base, &tmZ, &full[st], c * 64, (int)(t * kZTok));
                    tma_load_2d(base + 16384, &tmZ, &full[st], dgp + c * 64, (int)(t * kZTok));
                }
            }
            if (!ok) {
                const uint64_t deadline = global_timer_ns() + 200000000ull;
                mbar_wait_until(cbar, 0, deadline);
                for (int64_t t = g > S ? g - S : 0; t < g; ++t)
                    mbar_wait_until(&full[t % S], (uint32_t)(t / S) & 1u, deadline);
            }
        }
        __syncwarp();
    } else if (warp == kZEpiWarps + 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kZTok, Kp);
            bool ok = mbar_wait(cbar, 0, abort_flag, a.wc);
            int64_t g = 0;
            int jj = 0;
            for (int64_t t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++jj) {
                const int b = jj & 1;
                if (jj >= 2 &&
                    !(ok = mbar_wait(&tempty[b], (uint32_t)((jj >> 1) - 1) & 1u, abort_flag,
                                     a.wc)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * Kp);
                for (int c = 0; c < nchunk; ++c, ++g) {
                    const int st = (int)(g % S);
                    if (!(ok = mbar_wait(&full[st], (uint32_t)(g / S) & 1u, abort_flag, a.wc)))
                        break;
                    tc_fence_after();
                    const uint32_t zh = smem_u32(sZ + (size_t)st * kZsStage), zl = zh + 16384;
                    const uint32_t ch = smem_u32(sC + (size_t)c * 2 * Kp * 128),
                                   cl = ch + (uint32_t)Kp * 128;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ah = sdesc_sw128(zh + kk * 32, 16, 1024);
                        const uint64_t al = sdesc_sw128(zl + kk * 32, 16, 1024);
                        const uint64_t bh = sdesc_sw128(ch + kk * 32, 16, 1024);
                        const uint64_t bl = sdesc_sw128(cl + kk * 32, 16, 1024);
                        tc_mma_bf16(d, ah, bh, idesc, (c > 0 || kk > 0) ? 1u : 0u);
                        tc_mma_bf16(d, ah, bl, idesc, 1u);
                        tc_mma_bf16(d, al, bh, idesc, 1u);
                    }
                    tc_commit(&empty[st]);
                }
                if (ok) tc_commit(&tfull[b]);
            }
            tc_commit(drain);
            mbar_wait_until(drain, 0, global_timer_ns() + 500000000ull);
        }
        __syncwarp();
    } else {
        const int nsel = min(a.topk + 1, a.K);
        switch (nsel) {
        case 1: z_score_epilogue<1>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 2: z_score_epilogue<2>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 3: z_score_epilogue<3>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 4: z_score_epilogue<4>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 5: z_score_epilogue<5>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 6: z_score_epilogue<6>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 7: z_score_epilogue<7>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        case 8: z_score_epilogue<8>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        default: z_score_epilogue<9>(a, tmem, tfull, tempty, abort_flag, xs, xi, ntiles); break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kZEpiWarps + 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// fp16 2-D tensor map [outer, inner] (inner contiguous), box {64, box_outer},
// 128-byte swizzle.
bool make_map_2d_f16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                     uint32_t box_outer)
{
    return make_map_2d(m, base, inner, outer, 64, box_outer, true);
}

inline size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

int assign_z_dgp(int dg) { return (dg + 63) / 64 * 64; }

bool assign_z_supported(int hidden, int dg, int K, int topk)
{
    const int Kp = (K + 15) / 16 * 16, dgp = assign_z_dgp(dg);
    return K <= 256 && topk <= 8 && hidden % 64 == 0 && dgp <= 128 && Kp > dgp;
}

size_t assign_z_ws_bytes(int64_t ntok, int hidden, int dg, int K)
{
    const int Kp = (K + 15) / 16 * 16, dgp = assign_z_dgp(dg);
    return al256((size_t)2 * dgp * hidden * 2) + al256((size_t)2 * Kp * dgp * 2) +
           al256((size_t)ntok * 2 * dgp * 2) + al256((size_t)ntok * 4) + 256;
}

cudaError_t assign_z_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan)
{
    const int Kp = (p.K + 15) / 16 * 16, dgp = assign_z_dgp(p.dg);
    uint8_t *base = static_cast<uint8_t *>(ws);
    size_t off = 0;
    plan->wt = base + off;     off += al256((size_t)2 * dgp * p.hidden * 2);
    plan->ch = base + off;     off += al256((size_t)2 * Kp * dgp * 2);
    plan->z = base + off;      off += al256((size_t)p.ntok * 2 * dgp * 2);
    plan->zscale = reinterpret_cast<float *>(base + off);
    plan->Kp = Kp;
    plan->dgp = dgp;
    plan->wc = wc;
    plan->p = p;
    plan->path = 2;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    // GEMM: stages of 32 KB of X plus 256 dgp bytes of W_g within ~200 KB
    const uint32_t sb = z_stage_bytes(dgp);
    int st = (int)(200u * 1024u / sb);
    plan->stages = st > 4 ? 4 : (st < 2 ? 2 : st);
    plan->smem = (size_t)plan->stages * sb + (2 * plan->stages + 5) * 8 + 16 + 1024;
    const int64_t nsup = (p.ntok + 255) / 256;
    plan->grid = nsup < sms ? nsup : sms;
    // score kernel: C resident, then as many 32 KB Z stages as fit (2 to 4)
    const uint32_t cb = zs_c_bytes(Kp, dgp);
    const size_t fixed = (size_t)cb + kZsMerge + (2 * 4 + 6) * 8 + 16 + 1024;
    int st2 = (int)((kMaxSmemPerBlock - fixed) / kZsStage);
    plan->stages2 = st2 > 4 ? 4 : st2;
    if (plan->stages2 < 2) return cudaErrorInvalidConfiguration;
    plan->smem2 = (size_t)cb + (size_t)plan->stages2 * kZsStage + kZsMerge +
                  (2 * plan->stages2 + 6) * 8 + 16 + 1024;
    const int64_t ntiles = (p.ntok + 127) / 128;
    plan->grid2 = ntiles < sms ? ntiles : sms;
    if (p.ntok > 0) {
        if (!make_map_2d(&plan->map[0], p.X, (uint64_t)p.hidden, (uint64_t)p.ntok, 64, 128, false) ||
            !make_map_2d(&plan->map[1], plan->wt, (uint64_t)p.hidden, (uint64_t)(2 * dgp), 64,
                         (uint32_t)dgp, false) ||
            !make_map_2d_f16(&plan->map[2], plan->z, (uint64_t)(2 * dgp), (uint64_t)p.ntok, 128) ||
            !make_map_2d_f16(&plan->map[3], plan->ch, (uint64_t)dgp, (uint64_t)(2 * Kp),
                             (uint32_t)Kp))
            return cudaErrorInvalidValue;
    }
    if ((e = cudaFuncSetAttribute(assign_z_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)plan->smem)) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(assign_z_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)plan->smem2);
}

cudaError_t assign_z_launch(const AssignPlan &plan, cudaStream_t s, int *launches)
{
    const AssignLaunch &p = plan.p;
    const int Kp = plan.Kp, dgp = plan.dgp;
    cudaError_t e;
    {
        const int nwt = (p.hidden / 32) * (dgp / 32);
        const int64_t nc = ((int64_t)Kp * dgp + 255) / 256;
        prof_begin("assign_prep", s);
        e = launch_pdl(assign_z_prep_kernel, dim3((unsigned)(nwt + nc)), dim3(256), 0, s, p.Wg,
                       p.C, p.hidden, p.dg, dgp, p.K, Kp,
                       static_cast<__nv_bfloat16 *>(plan.wt), static_cast<__half *>(plan.ch));
        prof_end(s);
        if (e != cudaSuccess) return e;
        *launches += 1;
    }
    if (p.ntok == 0) return cudaSuccess;
    ZGemmArgs ga;
    ga.ntok = p.ntok;
    ga.hidden = p.hidden;
    ga.dgp = dgp;
    ga.stages = plan.stages;
    ga.Z = static_cast<__half *>(plan.z);
    ga.zscale = plan.zscale;
    ga.wc = plan.wc;
    prof_begin("assign", s);
    e = launch_pdl(assign_z_gemm_kernel, dim3((unsigned)plan.grid), dim3(192), plan.smem, s,
                   plan.map[0], plan.map[1], ga);
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    ZScoreArgs sa;
    sa.ntok = p.ntok;
    sa.K = p.K;
    sa.Kp = Kp;
    sa.dgp = dgp;
    sa.topk = p.topk;
    sa.stages = plan.stages2;
    sa.zscale = plan.zscale;
    sa.ids = p.ids;
    sa.margin = p.margin;
    sa.wc = plan.wc;
    prof_begin("assign_score", s);
    e = launch_pdl(assign_z_score_kernel, dim3((unsigned)plan.grid2),
                   dim3(32 * (kZEpiWarps + 2)), plan.smem2, s,
                   plan.map[2], plan.map[3], sa);
    prof_end(s);
    *launches += 1;
    return e;
}

}  // namespace focus
