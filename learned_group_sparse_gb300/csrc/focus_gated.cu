// Soft-gated attention of training and its backward (Focus, gist.science/zh
// technical summary 2.1.2 "gated attention": the score is
//     s_ij = q_i . k_j * (1_local + (1 - 1_local) * sigma(lambda * a_ij)),
// computed for every causal pair while training; gist.science/nl
// Kerncomponent 4: soft gates over all pairs in training, hard top-k at
// inference).  Readings: 1_local = [i - j < w]; a_ij = g_i . g_j, the dot
// product of the tokens' soft group assignments (rows of G); q . k is scaled
// by `scale` before the gate; causal softmax over j <= i.
//
// The forward runs on the 5th-generation tensor cores (focus_gated_tc.cu):
// the fp16 copy of G made here (its columns padded to a multiple of 16 with
// zeros) feeds a second product A = G_q G_k^T beside S = Q K^T in TMEM.
// The backward kernels here tile queries and keys by 64; a warp owns 16 rows
// of a tile and runs m16n8k16 tensor-core MMAs (`mma.sync`, fp32
// accumulation): S = Q K^T in bf16 and A = G_q G_k^T in fp16, the gate and
// P in registers, then the gradient products.  Each kernel recomputes P
// from the forward's log-sum-exp, so none needs atomics and every sum has a
// fixed order:
//   gated_bwd_prep_kernel   D_i = dO_i . O_i per (row, head)
//   gated_bwd_q_kernel      rows = queries (CTA: 64 queries, 4 heads,
//                           batch): dQ, the row side of dG, sum_j da_ij g_j,
//                           and d lambda
//   gated_bwd_k_kernel      rows = keys (CTA: 64 keys, kv head, batch, over
//                           its query heads): dK, dV and the column side of
//                           dG, sum_i da_ij g_i
//   gated_dg_reduce_kernel  dG = the sum of the per-chunk partials
// with dS_ij = P_ij (dP_ij - D_i), dP_ij = dO_i . v_j, and for a gated pair
// d gate_ij = dS_ij t_ij, da_ij = d gate_ij lambda sigma (1 - sigma).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "focus_internal.h"
#include "focus_ptx.cuh"

namespace focus {

namespace {

constexpr int kGT = 64;               // rows per tile (queries or keys)
constexpr int kGWarps = 4;            // 16 rows per warp
constexpr int kGThreads = kGWarps * 32;
constexpr int kGMaxKs = 8;            // k-steps of 16 over the padded groups: K_g <= 128
constexpr int kGHeadChunk = 4;        // query heads per CTA of the dG kernels (partials per chunk)

struct GatedArgs {
    const __nv_bfloat16 *q, *k, *v;   // [B, n, Hq | Hkv, D]
    const __half *g;                  // [B, n, kp] fp16, zero-padded columns
    const __nv_bfloat16 *o, *dO;      // [B, n, Hq, D]
    const float *lse;                 // [B, Hq, n] natural log
    const float *Dd;                  // [B, Hq, n] dO . O
    __nv_bfloat16 *out;               // O (forward)
    float *lse_out;                   // forward
    float *dq, *dk, *dv, *dg;         // [B, n, Hq, D], [B, n, Hkv, D] x 2, [B, n, Kg]
    float *dlam_part;                 // [B, nhc, n / 64] partial d lambda
    float *dg_part;                   // [nhc + Hkv][B, n, Kg]: row side per head chunk, column
                                      // side per kv head
    int B, n, Hq, Hkv, kp, Kg, window;
    int hc, nhc;                      // query heads per dG chunk, chunks
    float scale, lambda;
};

__device__ __forceinline__ void g_ldsm_x4(const void *p, uint32_t *r)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void g_ldsm_x4_t(const void *p, uint32_t *r)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// c += A B, m16n8k16, bf16 or fp16 inputs, fp32 accumulation
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment of a 16 x 16 block of rows stored [row][col] with `stride` bytes
// per row, at (row 0, column c0).
__device__ __forceinline__ void lda(const uint8_t *base, int stride, int c0, int lane,
                                    uint32_t *a)
{
    const int r = lane & 15, c = c0 + ((lane >> 4) << 3);
    g_ldsm_x4(base + r * stride + c * 2, a);
}

// B fragments of two n-tiles (rows 0..7 and 8..15 of a [n][k] array, k = c0
// .. c0 + 15): b[0], b[1] for the first n-tile, b[2], b[3] for the second.
__device__ __forceinline__ void ldb_nk(const uint8_t *base, int stride, int c0, int lane,
                                       uint32_t *b)
{
    const int r = ((lane >> 4) << 3) + (lane & 7), c = c0 + (((lane >> 3) & 1) << 3);
    g_ldsm_x4(base + r * stride + c * 2, b);
}

// B fragments of two n-tiles from a [k][n] array (k rows 0..15, n columns
// c0 .. c0 + 15): transposed loads.
__device__ __forceinline__ void ldb_kn(const uint8_t *base, int stride, int c0, int lane,
                                       uint32_t *b)
{
    const int r = (((lane >> 3) & 1) << 3) + (lane & 7), c = c0 + ((lane >> 4) << 3);
    g_ldsm_x4_t(base + r * stride + c * 2, b);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// rows [r0, r0 + 64) of a [B, n, H, W] (16-bit) tensor, head h, into shared
// rows of `stride` bytes; rows past n are zero-filled
__device__ __forceinline__ void load_tile(uint8_t *dst, int stride, const void *src, int b, int n,
                                          int H, int h, int W, int r0, int tid)
{
    const int units = W / 8;   // 16-byte units per row
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    for (int x = tid; x < kGT * units; x += kGThreads) {
        const int r = x / units, u = x - r * units;
        const int row = r0 + r;
        const bool ok = row < n;
        const int64_t off = ((((int64_t)b * n + (ok ? row : 0)) * H + h) * W + u * 8) * 2;
        cp_async16(dst + r * stride + u * 16, s8 + off, ok ? 16u : 0u);
    }
}

// sigma(z) = 1/2 + tanh(z / 2) / 2 with the hardware tanh approximation
// (relative error about 2^-11: below the fp16 rounding of the G products).
__device__ __forceinline__ float sigmoidf_(float z)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}

// Where a 64 x 64 tile of queries [q0, q0 + 64) and keys [k0, k0 + 64) lies
// against the window: every pair inside it, or some pair inside it.
__device__ __forceinline__ bool tile_all_local(int q0, int k0, int window)
{
    return q0 + kGT - 1 - k0 < window;
}
__device__ __forceinline__ bool tile_any_local(int q0, int k0, int window)
{
    return q0 - (k0 + kGT - 1) < window;
}


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

// D[b, h, i] = dO_i . O_i (bf16 inputs, fp32 sum): one warp per (row, head).
template <int D>
__global__ void gated_bwd_prep_kernel(const GatedArgs a, float *__restrict__ Dd)
{
    grid_dep_sync();
    const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= (int64_t)a.B * a.n * a.Hq) return;
    const int64_t row = w / a.Hq;   // b * n + i
    const int h = (int)(w - row * a.Hq);
    const __nv_bfloat16 *o = a.o + w * D, *g = a.dO + w * D;
    float sum = 0.f;
#pragma unroll
    for (int e = lane; e < D; e += 32) sum += __bfloat162float(o[e]) * __bfloat162float(g[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) {
        const int64_t b = row / a.n, i = row - b * a.n;
        Dd[(b * a.Hq + h) * a.n + i] = sum;
    }
}

// Shared layout of a backward CTA: the tiles of its own rows (queries:
// Q, dO, G_q; keys: K, V, G_k), then one stage of the other side's tiles,
// then the other side's log-sum-exp and D (key orientation only).
template <int D>
struct GatedBwdSmem {
    static constexpr int kRow = D * 2 + 16;
    static __host__ __device__ int side(int kp) { return kGT * (2 * kRow + kp * 2 + 16); }
    // + the dG_k tile of the key side, [64][kp + 8] floats
    static __host__ __device__ int bytes(int kp)
    {
        return 2 * side(kp) + 2 * kGT * 4 + kGT * (kp + 8) * 4;
    }
};

// Backward with rows = queries, CTA (64 queries, chunk of hc heads, batch):
// for every head of the chunk and every key tile up to the diagonal, taken
// in two halves of 32 keys (so that the tiles' scores fit the registers next
// to both accumulators): S = Q K^T, A = G_q G_k^T, P = exp(gated logit -
// LSE), dP = dO V^T, dS = P (dP - D); then dQ += (dS gate scale) K (written
// per head) and, for gated pairs, dG_q += (dS t lambda sigma') G_k and
// d lambda += dS t a sigma' (both summed over the chunk's heads).
template <int D>
__global__ void __launch_bounds__(kGThreads, 2) gated_bwd_q_kernel(const GatedArgs a)
{
    using L = GatedBwdSmem<D>;
    constexpr int kRow = L::kRow;
    constexpr int NG = 2 * kGMaxKs;   // n-tiles of the dG accumulator
    grid_dep_sync();
    extern __shared__ __align__(128) uint8_t gsm[];
    const int gRow = a.kp * 2 + 16;
    uint8_t *Qs = gsm, *dOs = gsm + kGT * kRow, *Gqs = gsm + 2 * kGT * kRow;
    uint8_t *Ks = gsm + L::side(a.kp), *Vs = Ks + kGT * kRow, *Gks = Ks + 2 * kGT * kRow;
    const int qt = gridDim.x - 1 - blockIdx.x;
    const int b = blockIdx.z;
    const int h0 = (int)blockIdx.y * a.hc, h1 = min(a.Hq, h0 + a.hc);
    const int gqa = a.Hq / a.Hkv;
    const int q0 = qt * kGT;
    const int nks = a.kp / 16;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rbase = q0 + 16 * warp + (lane >> 2);
    const float l2e = 1.4426950408889634f;

    float gacc[NG][4];
#pragma unroll
    for (int x = 0; x < NG; ++x) gacc[x][0] = gacc[x][1] = gacc[x][2] = gacc[x][3] = 0.f;
    float dlam = 0.f;
    load_tile(Gqs, gRow, a.g, b, a.n, 1, 0, a.kp, q0, tid);
    for (int h = h0; h < h1; ++h) {
        const int kvh = h / gqa;
        load_tile(Qs, kRow, a.q, b, a.n, a.Hq, h, D, q0, tid);
        load_tile(dOs, kRow, a.dO, b, a.n, a.Hq, h, D, q0, tid);
        float lse2[2], dd[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = rbase + 8 * r;
            const int64_t at = ((int64_t)b * a.Hq + h) * a.n + i;
            lse2[r] = i < a.n ? a.lse[at] * l2e : 0.f;
            dd[r] = i < a.n ? a.Dd[at] : 0.f;
        }
        float qacc[D / 8][4];
#pragma unroll
        for (int x = 0; x < D / 8; ++x) qacc[x][0] = qacc[x][1] = qacc[x][2] = qacc[x][3] = 0.f;
        for (int kt = 0; kt <= qt; ++kt) {
            const int k0 = kt * kGT;
            const bool all_local = tile_all_local(q0, k0, a.window);
            const bool any_local = tile_any_local(q0, k0, a.window);
            load_tile(Ks, kRow, a.k, b, a.n, a.Hkv, kvh, D, k0, tid);
            load_tile(Vs, kRow, a.v, b, a.n, a.Hkv, kvh, D, k0, tid);
            if (!all_local) load_tile(Gks, gRow, a.g, b, a.n, 1, 0, a.kp, k0, tid);
            cp_async_wait_all();
            __syncthreads();
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int c0 = 32 * hf;   // first key of the half in the tile
                float s[4][4], ag[4][4], dp[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] = ag[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t qa[4], oa[4];
                    lda(Qs + 16 * warp * kRow, kRow, 16 * kk, lane, qa);
                    lda(dOs + 16 * warp * kRow, kRow, 16 * kk, lane, oa);
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        uint32_t bb[4];
                        ldb_nk(Ks + (c0 + 16 * np) * kRow, kRow, 16 * kk, lane, bb);
                        mma_bf16(s[2 * np], qa, bb[0], bb[1]);
                        mma_bf16(s[2 * np + 1], qa, bb[2], bb[3]);
                        ldb_nk(Vs + (c0 + 16 * np) * kRow, kRow, 16 * kk, lane, bb);
                        mma_bf16(dp[2 * np], oa, bb[0], bb[1]);
                        mma_bf16(dp[2 * np + 1], oa, bb[2], bb[3]);
                    }
                }
                if (!all_local)
#pragma unroll
                    for (int ks = 0; ks < kGMaxKs; ++ks)
                        if (ks < nks) {
                            uint32_t ga[4];
                            lda(Gqs + 16 * warp * gRow, gRow, 16 * ks, lane, ga);
#pragma unroll
                            for (int np = 0; np < 2; ++np) {
                                uint32_t bb[4];
                                ldb_nk(Gks + (c0 + 16 * np) * gRow, gRow, 16 * ks, lane, bb);
                                mma_f16(ag[2 * np], ga, bb[0], bb[1]);
                                mma_f16(ag[2 * np + 1], ga, bb[2], bb[3]);
                            }
                        }
                // dt = dS gate scale into s, da = dS t lambda sigma' into ag
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = e >> 1;
                        const int i = rbase + 8 * r;
                        const int j = k0 + c0 + 8 * nt + 2 * (lane & 3) + (e & 1);
                        const bool valid = j <= i && i < a.n;
                        const bool local = all_local || (any_local && i - j < a.window);
                        const float t = s[nt][e] * a.scale;
                        const float sg = local ? 1.f : sigmoidf_(a.lambda * ag[nt][e]);
                        const float P = valid ? exp2f(t * sg * l2e - lse2[r]) : 0.f;
                        const float ds = P * (dp[nt][e] - dd[r]);
                        const float sp = sg * (1.f - sg);
                        const bool gated = valid && !local;
                        dlam += gated ? ds * t * ag[nt][e] * sp : 0.f;
                        s[nt][e] = ds * sg * a.scale;
                        ag[nt][e] = gated ? ds * t * a.lambda * sp : 0.f;
                    }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t pa[4] = {pack_bf16x2(s[2 * kk][0], s[2 * kk][1]),
                                            pack_bf16x2(s[2 * kk][2], s[2 * kk][3]),
                                            pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                            pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
                    for (int dq = 0; dq < D / 16; ++dq) {
                        uint32_t bb[4];
                        ldb_kn(Ks + (c0 + 16 * kk) * kRow, kRow, 16 * dq, lane, bb);
                        mma_bf16(qacc[2 * dq], pa, bb[0], bb[1]);
                        mma_bf16(qacc[2 * dq + 1], pa, bb[2], bb[3]);
                    }
                    if (!all_local) {
                        const uint32_t ha[4] = {pack_h2(ag[2 * kk][0], ag[2 * kk][1]),
                                                pack_h2(ag[2 * kk][2], ag[2 * kk][3]),
                                                pack_h2(ag[2 * kk + 1][0], ag[2 * kk + 1][1]),
                                                pack_h2(ag[2 * kk + 1][2], ag[2 * kk + 1][3])};
#pragma unroll
                        for (int c = 0; c < kGMaxKs; ++c)
                            if (c < nks) {
                                uint32_t bb[4];
                                ldb_kn(Gks + (c0 + 16 * kk) * gRow, gRow, 16 * c, lane, bb);
                                mma_f16(gacc[2 * c], ha, bb[0], bb[1]);
                                mma_f16(gacc[2 * c + 1], ha, bb[2], bb[3]);
                            }
                    }
                }
            }
            __syncthreads();   // the key tiles are rewritten next
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = rbase + 8 * r;
            if (i >= a.n) continue;
            float *row = a.dq + (((int64_t)b * a.n + i) * a.Hq + h) * D;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                *reinterpret_cast<float2 *>(row + 8 * nt + 2 * (lane & 3)) =
                    make_float2(qacc[nt][2 * r], qacc[nt][2 * r + 1]);
        }
        __syncthreads();   // the query tiles are rewritten for the next head
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = rbase + 8 * r;
        if (i >= a.n) continue;
        float *row = a.dg_part + (((int64_t)blockIdx.y * a.B + b) * a.n + i) * a.Kg;
#pragma unroll
        for (int nt = 0; nt < NG; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 8 * nt + 2 * (lane & 3) + e;
                if (c < a.Kg) row[c] = gacc[nt][2 * r + e];
            }
    }
    // d lambda of the CTA's pairs, in a fixed order
    __shared__ float red[kGWarps];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, off);
    if (lane == 0) red[warp] = dlam;
    __syncthreads();
    if (tid == 0)
        a.dlam_part[((int64_t)b * gridDim.y + blockIdx.y) * gridDim.x + qt] =
            (red[0] + red[1]) + (red[2] + red[3]);
}

// Backward with rows = keys, CTA (64 keys, kv head, batch), over the query
// heads of the kv head: dK, dV and the column side of dG.  For each query
// tile from the diagonal on, in two halves of 32 queries: S^T = K Q^T,
// A^T = G_k G_q^T, P^T from the queries' LSE, dP^T = V dO^T,
// dS^T = P^T (dP^T - D); then dV += P^T dO, dK += (dS^T gate scale) Q and,
// for gated pairs, dG_k += (dS^T t lambda sigma') G_q.  dK and dV stay in
// registers; the dG_k products are added into a shared [64][kp] tile (each
// element owned by one lane), written at the end as this kv head's partial.
template <int D>
__global__ void __launch_bounds__(kGThreads, 2) gated_bwd_k_kernel(const GatedArgs a)
{
    using L = GatedBwdSmem<D>;
    constexpr int kRow = L::kRow;
    grid_dep_sync();
    extern __shared__ __align__(128) uint8_t gsm[];
    const int gRow = a.kp * 2 + 16;
    const int gStride = a.kp + 8;   // floats per row of the dG_k tile
    uint8_t *Ks = gsm, *Vs = gsm + kGT * kRow, *Gks = gsm + 2 * kGT * kRow;
    uint8_t *Qs = gsm + L::side(a.kp), *dOs = Qs + kGT * kRow, *Gqs = Qs + 2 * kGT * kRow;
    float *lse2s = reinterpret_cast<float *>(gsm + 2 * L::side(a.kp));
    float *dds = lse2s + kGT;
    float *dgs = dds + kGT;         // [64][gStride]
    const int kt = blockIdx.x;      // the first key tiles have the most query tiles
    const int b = blockIdx.z;
    const int gqa = a.Hq / a.Hkv;
    const int kvh = blockIdx.y;
    const int h0 = kvh * gqa, h1 = h0 + gqa;
    const int k0 = kt * kGT;
    const int nqt = (a.n + kGT - 1) / kGT;
    const int nks = a.kp / 16;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rbase = k0 + 16 * warp + (lane >> 2);
    const float l2e = 1.4426950408889634f;

    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int x = 0; x < D / 8; ++x) {
        dk[x][0] = dk[x][1] = dk[x][2] = dk[x][3] = 0.f;
        dv[x][0] = dv[x][1] = dv[x][2] = dv[x][3] = 0.f;
    }
    for (int x = tid; x < kGT * gStride; x += kGThreads) dgs[x] = 0.f;
    load_tile(Gks, gRow, a.g, b, a.n, 1, 0, a.kp, k0, tid);
    load_tile(Ks, kRow, a.k, b, a.n, a.Hkv, kvh, D, k0, tid);
    load_tile(Vs, kRow, a.v, b, a.n, a.Hkv, kvh, D, k0, tid);
    for (int h = h0; h < h1; ++h) {
        for (int qt = kt; qt < nqt; ++qt) {
            const int q0 = qt * kGT;
            const bool all_local = tile_all_local(q0, k0, a.window);
            const bool any_local = tile_any_local(q0, k0, a.window);
            load_tile(Qs, kRow, a.q, b, a.n, a.Hq, h, D, q0, tid);
            load_tile(dOs, kRow, a.dO, b, a.n, a.Hq, h, D, q0, tid);
            if (!all_local) load_tile(Gqs, gRow, a.g, b, a.n, 1, 0, a.kp, q0, tid);
            if (tid < kGT) {
                const int i = q0 + tid;
                const int64_t at = ((int64_t)b * a.Hq + h) * a.n + i;
                lse2s[tid] = i < a.n ? a.lse[at] * l2e : 0.f;
                dds[tid] = i < a.n ? a.Dd[at] : 0.f;
            }
            cp_async_wait_all();
            __syncthreads();
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int c0 = 32 * hf;   // first query of the half in the tile
                float s[4][4], ag[4][4], dp[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] = ag[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t ka[4], va[4];
                    lda(Ks + 16 * warp * kRow, kRow, 16 * kk, lane, ka);
                    lda(Vs + 16 * warp * kRow, kRow, 16 * kk, lane, va);
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        uint32_t bb[4];
                        ldb_nk(Qs + (c0 + 16 * np) * kRow, kRow, 16 * kk, lane, bb);
                        mma_bf16(s[2 * np], ka, bb[0], bb[1]);
                        mma_bf16(s[2 * np + 1], ka, bb[2], bb[3]);
                        ldb_nk(dOs + (c0 + 16 * np) * kRow, kRow, 16 * kk, lane, bb);
                        mma_bf16(dp[2 * np], va, bb[0], bb[1]);
                        mma_bf16(dp[2 * np + 1], va, bb[2], bb[3]);
                    }
                }
                if (!all_local)
#pragma unroll
                    for (int ks = 0; ks < kGMaxKs; ++ks)
                        if (ks < nks) {
                            uint32_t ga[4];
                            lda(Gks + 16 * warp * gRow, gRow, 16 * ks, lane, ga);
#pragma unroll
                            for (int np = 0; np < 2; ++np) {
                                uint32_t bb[4];
                                ldb_nk(Gqs + (c0 + 16 * np) * gRow, gRow, 16 * ks, lane, bb);
                                mma_f16(ag[2 * np], ga, bb[0], bb[1]);
                                mma_f16(ag[2 * np + 1], ga, bb[2], bb[3]);
                            }
                        }
                // P^T into dp, dt into s, da into ag
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = rbase + 8 * (e >> 1);                      // key
                        const int cl = c0 + 8 * nt + 2 * (lane & 3) + (e & 1);   // query in the tile
                        const int i = q0 + cl;
                        const bool valid = j <= i && i < a.n && j < a.n;
                        const bool local = all_local || (any_local && i - j < a.window);
                        const float t = s[nt][e] * a.scale;
                        const float sg = local ? 1.f : sigmoidf_(a.lambda * ag[nt][e]);
                        const float P = valid ? exp2f(t * sg * l2e - lse2s[cl]) : 0.f;
                        const float ds = P * (dp[nt][e] - dds[cl]);
                        s[nt][e] = ds * sg * a.scale;
                        dp[nt][e] = P;
                        ag[nt][e] = (valid && !local) ? ds * t * a.lambda * sg * (1.f - sg) : 0.f;
                    }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t ta[4] = {pack_bf16x2(s[2 * kk][0], s[2 * kk][1]),
                                            pack_bf16x2(s[2 * kk][2], s[2 * kk][3]),
                                            pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                            pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
                    const uint32_t pa[4] = {pack_bf16x2(dp[2 * kk][0], dp[2 * kk][1]),
                                            pack_bf16x2(dp[2 * kk][2], dp[2 * kk][3]),
                                            pack_bf16x2(dp[2 * kk + 1][0], dp[2 * kk + 1][1]),
                                            pack_bf16x2(dp[2 * kk + 1][2], dp[2 * kk + 1][3])};
#pragma unroll
                    for (int dq = 0; dq < D / 16; ++dq) {
                        uint32_t bb[4];
                        ldb_kn(Qs + (c0 + 16 * kk) * kRow, kRow, 16 * dq, lane, bb);
                        mma_bf16(dk[2 * dq], ta, bb[0], bb[1]);
                        mma_bf16(dk[2 * dq + 1], ta, bb[2], bb[3]);
                        ldb_kn(dOs + (c0 + 16 * kk) * kRow, kRow, 16 * dq, lane, bb);
                        mma_bf16(dv[2 * dq], pa, bb[0], bb[1]);
                        mma_bf16(dv[2 * dq + 1], pa, bb[2], bb[3]);
                    }
                }
                if (!all_local) {
                    // dG_k += da G_q over the half's 32 queries, two n-tiles
                    // (16 group columns) at a time, added into the shared tile
                    uint32_t ha[2][4];
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        ha[kk][0] = pack_h2(ag[2 * kk][0], ag[2 * kk][1]);
                        ha[kk][1] = pack_h2(ag[2 * kk][2], ag[2 * kk][3]);
                        ha[kk][2] = pack_h2(ag[2 * kk + 1][0], ag[2 * kk + 1][1]);
                        ha[kk][3] = pack_h2(ag[2 * kk + 1][2], ag[2 * kk + 1][3]);
                    }
                    for (int c = 0; c < nks; ++c) {
                        float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            uint32_t bb[4];
                            ldb_kn(Gqs + (c0 + 16 * kk) * gRow, gRow, 16 * c, lane, bb);
                            mma_f16(g0, ha[kk], bb[0], bb[1]);
                            mma_f16(g1, ha[kk], bb[2], bb[3]);
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            float *row = dgs + (16 * warp + (lane >> 2) + 8 * r) * gStride +
                                         16 * c + 2 * (lane & 3);
                            float2 *p0 = reinterpret_cast<float2 *>(row);
                            float2 *p1 = reinterpret_cast<float2 *>(row + 8);
                            const float2 v0 = *p0, v1 = *p1;
                            *p0 = make_float2(v0.x + g0[2 * r], v0.y + g0[2 * r + 1]);
                            *p1 = make_float2(v1.x + g1[2 * r], v1.y + g1[2 * r + 1]);
                        }
                    }
                }
            }
            __syncthreads();   // the query tiles are rewritten next
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int j = rbase + 8 * r;
        if (j >= a.n) continue;
        const int64_t off = (((int64_t)b * a.n + j) * a.Hkv + kvh) * D + 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            *reinterpret_cast<float2 *>(a.dk + off + 8 * nt) =
                make_float2(dk[nt][2 * r], dk[nt][2 * r + 1]);
            *reinterpret_cast<float2 *>(a.dv + off + 8 * nt) =
                make_float2(dv[nt][2 * r], dv[nt][2 * r + 1]);
        }
    }
    // this kv head's partial of the column side of dG (its rows only)
    __syncthreads();
    float *part = a.dg_part + ((((int64_t)a.nhc + kvh) * a.B + b) * a.n) * a.Kg;
    for (int x = tid; x < kGT * a.Kg; x += kGThreads) {
        const int r = x / a.Kg, c = x - r * a.Kg;
        if (k0 + r < a.n) part[(int64_t)(k0 + r) * a.Kg + c] = dgs[r * gStride + c];
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

// d lambda = sum of the query-tile partials, in a fixed order (one thread).
__global__ void gated_dlam_kernel(const float *__restrict__ part, int count, float *__restrict__ out)
{
    grid_dep_sync();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        double s = 0.0;
        for (int x = 0; x < count; ++x) s += (double)part[x];
        *out = (float)s;
    }
}

}  // namespace

size_t gated_ws_bytes(int B, int n, int Hq, int Hkv, int Kg)
{
    const size_t a256 = 255;
    const int kp = (Kg + 15) / 16 * 16;
    const int nqt = (n + kGT - 1) / kGT;
    const int nhc = (Hq + kGHeadChunk - 1) / kGHeadChunk;
    return (((size_t)B * n * kp * 2 + a256) & ~a256) + (((size_t)B * Hq * n * 4 + a256) & ~a256) +
           (((size_t)B * nhc * nqt * 4 + a256) & ~a256) +
           (((size_t)(nhc + Hkv) * B * n * Kg * 4 + a256) & ~a256);
}

namespace {

template <int D>
cudaError_t gated_preflight_d(int kp)
{
    const int bwd = GatedBwdSmem<D>::bytes(kp);
    const cudaFuncAttribute at = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e = cudaFuncSetAttribute(gated_bwd_q_kernel<D>, at, bwd);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gated_bwd_k_kernel<D>, at, bwd);
    return e;
}

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
    a.Dd = reinterpret_cast<const float *>(w);
    w += ((size_t)p.B * p.Hq * p.n * 4 + a256) & ~a256;
    a.hc = kGHeadChunk < p.Hq ? kGHeadChunk : p.Hq;
    a.nhc = (p.Hq + a.hc - 1) / a.hc;
    a.dlam_part = reinterpret_cast<float *>(w);
    const int nqt = (p.n + kGT - 1) / kGT;
    w += ((size_t)p.B * ((p.Hq + kGHeadChunk - 1) / kGHeadChunk) * nqt * 4 + a256) & ~a256;
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
cudaError_t gated_bwd_t(const GatedLaunch &p, GatedArgs a, cudaStream_t s, int *launches)
{
    const int nqt = (p.n + kGT - 1) / kGT;
    const size_t smem = GatedBwdSmem<D>::bytes(a.kp);
    const dim3 blk(kGThreads);
    cudaError_t e;
    const int64_t warps = (int64_t)p.B * p.n * p.Hq;
    prof_begin("gated_bwd_prep", s);
    e = launch_pdl(gated_bwd_prep_kernel<D>, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256),
                   0, s, a, const_cast<float *>(a.Dd));
    prof_end(s);
    if (e != cudaSuccess) return e;
    prof_begin("gated_bwd_dq", s);
    e = launch_pdl(gated_bwd_q_kernel<D>, dim3(nqt, a.nhc, p.B), blk, smem, s, a);
    prof_end(s);
    if (e != cudaSuccess) return e;
    prof_begin("gated_bwd_dkv", s);
    e = launch_pdl(gated_bwd_k_kernel<D>, dim3(nqt, p.Hkv, p.B), blk, smem, s, a);
    prof_end(s);
    if (e != cudaSuccess) return e;
    const int64_t dgn = (int64_t)p.B * p.n * p.Kg;
    prof_begin("gated_dg_reduce", s);
    e = launch_pdl(gated_dg_reduce_kernel,
                   dim3((unsigned)std::min<int64_t>((dgn + 255) / 256, 152 * 8)), dim3(256), 0, s,
                   a);
    prof_end(s);
    if (e != cudaSuccess) return e;
    prof_begin("gated_dlam", s);
    e = launch_pdl(gated_dlam_kernel, dim3(1), dim3(32), 0, s, a.dlam_part, p.B * a.nhc * nqt,
                   p.dlam);
    prof_end(s);
    *launches += 5;
    return e;
}

}  // namespace

cudaError_t gated_preflight(int d, int Kg)
{
    const int kp = (Kg + 15) / 16 * 16;
    return d == 64 ? gated_preflight_d<64>(kp) : gated_preflight_d<128>(kp);
}

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
    cudaError_t e = launch_g16(p, a, s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return p.d == 64 ? gated_bwd_t<64>(p, a, s, launches) : gated_bwd_t<128>(p, a, s, launches);
}

}  // namespace focus
