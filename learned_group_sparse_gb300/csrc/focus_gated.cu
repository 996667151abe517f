// Soft-gated attention of training and its backward (Focus, gist.science/zh
// technical summary 2.1.2 "gated attention": the score is
//     s_ij = q_i . k_j * (1_local + (1 - 1_local) * sigma(lambda * a_ij)),
// computed for every causal pair while training; gist.science/nl
// Kerncomponent 4: soft gates over all pairs in training, hard top-k at
// inference).  Readings: 1_local = [i - j < w]; a_ij = g_i . g_j, the dot
// product of the tokens' soft group assignments (rows of G); q . k is scaled
// by `scale` before the gate; causal softmax over j <= i.
//
// The forward and the backward run on the 5th-generation tensor cores
// (focus_gated_tc.cu, focus_gated_bwd_tc.cu).  This file holds their small
// companions: the fp16 copy of G (its columns padded to a multiple of 16
// with zeros) that feeds the products A = G_q G_k^T, the backward's
// D_i = dO_i . O_i, the sum of the dG partials (one per query-head chunk from
// the query side, one per kv head from the key side) and of the d lambda
// partials, each in a fixed order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "focus_internal.h"
#include "focus_ptx.cuh"

namespace focus {

namespace {

constexpr int kGT = 64;               // d lambda partials: at most one per 64 query rows

struct GatedArgs {
    const __nv_bfloat16 *q, *k, *v;   // [B, n, Hq | Hkv, D]
    const __half *g;                  // [B, n, kp] fp16, zero-padded columns
    const __nv_bfloat16 *o, *dO;      // [B, n, Hq, D]
    const float *lse;                 // [B, Hq, n] natural log
    const float *rowv;                // [2][B, Hq, npad]: -lse log2(e) (-inf past n) and
                                      // -dO . O (0 past n), npad = n rounded up to 128
    __nv_bfloat16 *out;               // O (forward)
    float *lse_out;                   // forward
    float *dq, *dk, *dv, *dg;         // [B, n, Hq, D], [B, n, Hkv, D] x 2, [B, n, Kg]
    float *dlam_part;                 // [B, nhc, n / 64] partial d lambda
    float *dg_part;                   // [nhc + Hkv][B, n, Kg]: row side per head chunk, column
                                      // side per kv head
    int B, n, Hq, Hkv, kp, Kg, window, npad;
    int hc, nhc;                      // query heads per dG chunk, chunks
    float scale, lambda;
};

// G [B, n, Kg] fp32 -> [B, n, kp] fp16 with zero columns past Kg.
__global__ void gated_g16_kernel(const float *__restrict__ G, int64_t rows, int Kg, int kp,
                                 __half *__restrict__ g16)
{
    grid_dep_sync();
    const int64_t total = rows * kp;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = x / kp;
        const int c = (int)(x - r * kp);
        g16[x] = __float2half_rn(c < Kg ? G[r * Kg + c] : 0.f);
    }
}

// The backward's per-(row, head) values, D / 8 lanes each (16 bytes of O and
// of dO per lane): -lse_i log2(e) and
// -D_i = -dO_i . O_i (bf16 inputs, fp32 sum), in rows padded to npad (-inf
// and 0 past n) so that a kernel can copy any 64-row run of them whole.
template <int D>
__global__ void gated_bwd_prep_kernel(const GatedArgs a, float *__restrict__ rowv)
{
    constexpr int LPR = D / 8;   // lanes per (row, head): 16 bytes of O and of dO each
    grid_dep_sync();
    const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t w = g / LPR;
    const int sub = (int)(g % LPR);
    const bool live = w < (int64_t)a.B * a.npad * a.Hq;   // whole groups of LPR lanes
    const int64_t bi = w / a.Hq;     // b * npad + i
    const int h = (int)(w - bi * a.Hq);
    const int64_t b = bi / a.npad, i = bi - b * a.npad;
    float sum = 0.f;
    if (live && i < a.n) {
        const int64_t x = ((b * a.n + i) * a.Hq + h) * D + sub * 8;
        const uint4 ov = *reinterpret_cast<const uint4 *>(a.o + x);
        const uint4 gv = *reinterpret_cast<const uint4 *>(a.dO + x);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[q]));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[q]));
            sum = fmaf(of.x, gf.x, sum);
            sum = fmaf(of.y, gf.y, sum);
        }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (live && sub == 0) {
        const int64_t y = (b * a.Hq + h) * a.npad + i;
        const int64_t plane = (int64_t)a.B * a.Hq * a.npad;
        rowv[y] = i < a.n ? -a.lse[(b * a.Hq + h) * a.n + i] * 1.4426950408889634f : -CUDART_INF_F;
        rowv[plane + y] = -sum;
    }
}

// dG = the sum over head chunks of both sides' partials, in a fixed order.
__global__ void gated_dg_reduce_kernel(const GatedArgs a)
{
    grid_dep_sync();
    const int64_t total = (int64_t)a.B * a.n * a.Kg;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int c = 0; c < a.nhc + a.Hkv; ++c) s += a.dg_part[(int64_t)c * total + x];
        a.dg[x] = s;
    }
}

// d lambda = sum of the query-tile partials, in a fixed order (one warp).
__global__ void gated_dlam_kernel(const float *__restrict__ part, int count,
                                  float *__restrict__ out)
{
    grid_dep_sync();
    // lane l sums partials l, l + 32, ... in double, then a fixed shuffle tree
    double s = 0.0;
    for (int x = threadIdx.x; x < count; x += 32) s += (double)part[x];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (threadIdx.x == 0) *out = (float)s;
}

}  // namespace

size_t gated_ws_bytes(int B, int n, int Hq, int Hkv, int Kg)
{
    const size_t a256 = 255;
    const int kp = (Kg + 15) / 16 * 16;
    const int nqt = (n + kGT - 1) / kGT;
    const int nhc = (Hq + kGatedHeadChunk - 1) / kGatedHeadChunk;
    const size_t npad = ((size_t)n + 127) / 128 * 128;
    return (((size_t)B * n * kp * 2 + a256) & ~a256) +
           (((size_t)2 * B * Hq * npad * 4 + a256) & ~a256) +
           (((size_t)B * nhc * nqt * 4 + a256) & ~a256) +
           (((size_t)(nhc + Hkv) * B * n * Kg * 4 + a256) & ~a256);
}

namespace {

GatedArgs gated_args(const GatedLaunch &p, void *ws)
{
    const size_t a256 = 255;
    GatedArgs a{};
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.o = p.o;
    a.dO = p.dO;
    a.lse = p.lse;
    a.out = p.out;
    a.lse_out = p.lse_out;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.dg = p.dg;
    a.B = p.B;
    a.n = p.n;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.Kg = p.Kg;
    a.kp = (p.Kg + 15) / 16 * 16;
    a.window = p.window;
    a.scale = p.scale;
    a.lambda = p.lambda;
    uint8_t *w = static_cast<uint8_t *>(ws);
    a.g = reinterpret_cast<const __half *>(w);
    w += ((size_t)p.B * p.n * a.kp * 2 + a256) & ~a256;
    a.npad = (p.n + 127) / 128 * 128;
    a.rowv = reinterpret_cast<const float *>(w);
    w += ((size_t)2 * p.B * p.Hq * a.npad * 4 + a256) & ~a256;
    a.hc = kGatedHeadChunk < p.Hq ? kGatedHeadChunk : p.Hq;
    a.nhc = (p.Hq + a.hc - 1) / a.hc;
    a.dlam_part = reinterpret_cast<float *>(w);
    const int nqt = (p.n + kGT - 1) / kGT;
    w += ((size_t)p.B * a.nhc * nqt * 4 + a256) & ~a256;
    a.dg_part = reinterpret_cast<float *>(w);
    return a;
}

cudaError_t launch_g16(const GatedLaunch &p, const GatedArgs &a, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.B * p.n;
    const int64_t total = rows * a.kp;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256, 152 * 16);
    return launch_pdl(gated_g16_kernel, dim3(blocks), dim3(256), 0, s, p.G, rows, p.Kg, a.kp,
                      const_cast<__half *>(a.g));
}

template <int D>
cudaError_t gated_bwd_t(const GatedLaunch &p, const GatedArgs &a, const GatedBwTcPlan &plan,
                        cudaStream_t s, int *launches)
{
    cudaError_t e;
    const int64_t warps = (int64_t)p.B * a.npad * p.Hq;   // (row, head) groups
    prof_begin("gated_bwd_prep", s);
    e = launch_pdl(gated_bwd_prep_kernel<D>, dim3((unsigned)((warps * (D / 8) + 255) / 256)),
                   dim3(256),
                   0, s, a, const_cast<float *>(a.rowv));
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    if ((e = gated_bwd_tc_launch(plan, a.rowv, a.npad, a.dlam_part, a.dg_part, s, launches)) !=
        cudaSuccess)
        return e;
    const int64_t dgn = (int64_t)p.B * p.n * p.Kg;
    prof_begin("gated_dg_reduce", s);
    e = launch_pdl(gated_dg_reduce_kernel,
                   dim3((unsigned)std::min<int64_t>((dgn + 255) / 256, 152 * 8)), dim3(256), 0, s,
                   a);
    prof_end(s);
    if (e != cudaSuccess) return e;
    prof_begin("gated_dlam", s);
    e = launch_pdl(gated_dlam_kernel, dim3(1), dim3(32), 0, s, a.dlam_part,
                   gated_bwd_tc_dlam_count(p.B, p.n, p.Hq), p.dlam);
    prof_end(s);
    *launches += 2;
    return e;
}

}  // namespace

cudaError_t launch_gated_fwd(const GatedLaunch &p, void *ws, cudaStream_t s, int *launches)
{
    const GatedArgs a = gated_args(p, ws);
    GatedTcPlan plan;
    cudaError_t e = gated_tc_prepare(p, a.g, a.kp, &plan);   // enqueues nothing
    if (e != cudaSuccess) return e;
    if ((e = launch_g16(p, a, s)) != cudaSuccess) return e;
    *launches += 1;
    return gated_tc_launch(plan, s, launches);
}

cudaError_t launch_gated_bwd(const GatedLaunch &p, void *ws, cudaStream_t s, int *launches)
{
    const GatedArgs a = gated_args(p, ws);
    GatedBwTcPlan plan;
    cudaError_t e = gated_bwd_tc_prepare(p, a.g, a.kp, &plan);   // enqueues nothing
    if (e != cudaSuccess) return e;
    if ((e = launch_g16(p, a, s)) != cudaSuccess) return e;
    *launches += 1;
    return p.d == 64 ? gated_bwd_t<64>(p, a, plan, s, launches)
                     : gated_bwd_t<128>(p, a, plan, s, launches);
}

}  // namespace focus
