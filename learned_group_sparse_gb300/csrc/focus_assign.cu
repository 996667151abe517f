// Centroid scoring and hard top-k group membership (Focus, gist.science/zh
// technical summary 2.1.1 and 2.1.3): z = x W_g, s_c = z . C_c, and each
// token keeps the k highest-scoring groups (descending, ties to lower id).
//
// One CTA of 256 threads handles 64 tokens:
//   phase A  z[64][d_g] = X[64][hidden] . W_g, fp32 FMA over hidden chunks
//            of 32 staged in shared memory (bf16 X widened on load);
//   phase B  scores for 64 centroids at a time into shared memory;
//   phase C  one warp per token merges the new scores into its running
//            top-(k+1) list with k+1 rounds of warp arg-max.
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"

namespace focus {

namespace {

constexpr int kTM = 64;        // tokens per CTA
constexpr int kKC = 32;        // hidden chunk
constexpr int kCC = 64;        // centroids per phase-B chunk
constexpr int kMaxSel = 9;     // top-(k+1), k <= 8

// (score, id) ordering: larger score first, equal scores -> lower id first.
__device__ __forceinline__ bool better(float s1, int i1, float s2, int i2)
{
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

template <int NJ>   // d_g <= 128 * NJ; thread columns tx*4 + 128*j
__global__ void __launch_bounds__(256) assign_kernel(const __nv_bfloat16 *__restrict__ X,
                                                     const float *__restrict__ Wg,
                                                     const float *__restrict__ C, int64_t ntok,
                                                     int hidden, int dg, int K, int topk,
                                                     int32_t *__restrict__ ids,
                                                     float *__restrict__ margin)
{
    grid_dep_sync();
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    // layout (floats): z [kTM][dgp] | work area (max of phase A and phase B)
    const int dgp = 128 * NJ;
    float *zs = sm;                                        // [kTM][dgp]
    float *work = zs + kTM * dgp;
    // phase A: Xs [kTM][kKC] (fp32) | Ws [kKC][dgp]
    float *Xs = work;
    float *Ws = Xs + kTM * kKC;
    // phase B/C: Cs [dgp][kCC] | Ss [kTM][kCC] | best [kTM][kMaxSel] (score) + ids
    float *Cs = work;
    float *Ss = Cs + dgp * kCC;
    float *bestS = Ss + kTM * kCC;
    int *bestI = reinterpret_cast<int *>(bestS + kTM * kMaxSel);

    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * kTM;

    // ------------------------------------------------------------ phase A
    float acc[8][4 * NJ];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 4 * NJ; ++c) acc[a][c] = 0.f;

    for (int k0 = 0; k0 < hidden; k0 += kKC) {
        // X chunk: 64 tokens x 32 values; 256 threads x 8 values
        {
            const int tok = tid >> 2, part = tid & 3;
            const int64_t gt = t0 + tok;
            float v[8];
            if (gt < ntok && k0 + part * 8 < hidden) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(X + gt * hidden + k0 + part * 8);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[2 * e] = __uint_as_float(w[e] << 16);
                    v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Xs[tok * kKC + part * 8 + e] = v[e];
        }
        // W chunk: 32 rows x dgp columns (zero beyond d_g / hidden)
        for (int idx = tid; idx < kKC * dgp; idx += 256) {
            const int kr = idx / dgp, c = idx - kr * dgp;
            const int gk = k0 + kr;
            Ws[idx] = (gk < hidden && c < dg) ? __ldg(Wg + (int64_t)gk * dg + c) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kKC; ++kk) {
            float xv[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) xv[a] = Xs[(ty * 8 + a) * kKC + kk];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float4 w = *reinterpret_cast<const float4 *>(Ws + kk * dgp + j * 128 + tx * 4);
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    acc[a][4 * j + 0] = fmaf(xv[a], w.x, acc[a][4 * j + 0]);
                    acc[a][4 * j + 1] = fmaf(xv[a], w.y, acc[a][4 * j + 1]);
                    acc[a][4 * j + 2] = fmaf(xv[a], w.z, acc[a][4 * j + 2]);
                    acc[a][4 * j + 3] = fmaf(xv[a], w.w, acc[a][4 * j + 3]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            *reinterpret_cast<float4 *>(zs + (ty * 8 + a) * dgp + j * 128 + tx * 4) =
                make_float4(acc[a][4 * j], acc[a][4 * j + 1], acc[a][4 * j + 2], acc[a][4 * j + 3]);

    const int nsel = min(topk + 1, K);
    for (int i = tid; i < kTM * kMaxSel; i += 256) {
        bestS[i] = -CUDART_INF_F;
        bestI[i] = 0x7fffffff;
    }
    __syncthreads();

    // ---------------------------------------------------- phases B and C
    for (int c0 = 0; c0 < K; c0 += kCC) {
        // Cs[e][c] = C[c0 + c][e]
        for (int idx = tid; idx < kCC * dgp; idx += 256) {
            const int c = idx / dgp, e = idx - c * dgp;
            Cs[e * kCC + c] = (c0 + c < K && e < dg) ? __ldg(C + (int64_t)(c0 + c) * dg + e) : 0.f;
        }
        __syncthreads();
        {
            // thread: tokens ty*8..+7, centroids tx and tx+32 of this chunk
            float s0[8], s1[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) s0[a] = s1[a] = 0.f;
            for (int e = 0; e < dg; ++e) {
                const float c_a = Cs[e * kCC + tx], c_b = Cs[e * kCC + tx + 32];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const float z = zs[(ty * 8 + a) * dgp + e];
                    s0[a] = fmaf(z, c_a, s0[a]);
                    s1[a] = fmaf(z, c_b, s1[a]);
                }
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                Ss[(ty * 8 + a) * kCC + tx] = s0[a];
                Ss[(ty * 8 + a) * kCC + tx + 32] = s1[a];
            }
        }
        __syncthreads();
        // phase C: warp ty merges tokens ty*8..+7
        for (int a = 0; a < 8; ++a) {
            const int tok = ty * 8 + a;
            float cs[3];
            int ci[3];
            cs[0] = (c0 + tx < K) ? Ss[tok * kCC + tx] : -CUDART_INF_F;
            ci[0] = c0 + tx;
            cs[1] = (c0 + tx + 32 < K) ? Ss[tok * kCC + tx + 32] : -CUDART_INF_F;
            ci[1] = c0 + tx + 32;
            cs[2] = (tx < nsel) ? bestS[tok * kMaxSel + tx] : -CUDART_INF_F;
            ci[2] = (tx < nsel) ? bestI[tok * kMaxSel + tx] : 0x7fffffff;
            if (cs[0] != cs[0]) cs[0] = -CUDART_INF_F;
            if (cs[1] != cs[1]) cs[1] = -CUDART_INF_F;
            float selS = -CUDART_INF_F;
            int selI = 0x7fffffff;
            for (int rnd = 0; rnd < nsel; ++rnd) {
                // lane-local best of its three candidates
                int lb = 0;
                if (better(cs[1], ci[1], cs[lb], ci[lb])) lb = 1;
                if (better(cs[2], ci[2], cs[lb], ci[lb])) lb = 2;
                float bs = cs[lb];
                int bi = ci[lb];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (better(os, oi, bs, bi)) {
                        bs = os;
                        bi = oi;
                    }
                }
                // remove the winner (ids are unique across lanes' candidates)
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    if (ci[q] == bi) {
                        cs[q] = -CUDART_INF_F;
                        ci[q] = 0x7fffffff;
                    }
                if (tx == rnd) {
                    selS = bs;
                    selI = bi;
                }
            }
            __syncwarp();
            if (tx < nsel) {
                bestS[tok * kMaxSel + tx] = selS;
                bestI[tok * kMaxSel + tx] = selI;
            }
            __syncwarp();
        }
        __syncthreads();
    }

    // ------------------------------------------------------------ output
    for (int tok = tid; tok < kTM; tok += 256) {
        const int64_t gt = t0 + tok;
        if (gt >= ntok) continue;
        for (int s = 0; s < topk; ++s) ids[gt * topk + s] = bestI[tok * kMaxSel + s];
        if (margin) {
            float gap = CUDART_INF_F;
            for (int s = 1; s < nsel; ++s)
                gap = fminf(gap, bestS[tok * kMaxSel + s - 1] - bestS[tok * kMaxSel + s]);
            margin[gt] = gap;
        }
    }
}

template <int NJ>
size_t assign_smem_bytes()
{
    const int dgp = 128 * NJ;
    const size_t phaseA = (size_t)kTM * kKC + (size_t)kKC * dgp;
    const size_t phaseB = (size_t)dgp * kCC + (size_t)kTM * kCC + 2 * (size_t)kTM * kMaxSel;
    return sizeof(float) * ((size_t)kTM * dgp + (phaseA > phaseB ? phaseA : phaseB));
}

template <int NJ>
cudaError_t launch_assign_nj(const AssignLaunch &p, cudaStream_t s)
{
    const size_t smem = assign_smem_bytes<NJ>();
    cudaError_t e = cudaFuncSetAttribute(assign_kernel<NJ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (p.ntok + kTM - 1) / kTM;
    if (blocks == 0) return cudaSuccess;
    prof_begin("assign", s);
    e = launch_pdl(assign_kernel<NJ>, dim3((unsigned)blocks), dim3(256), smem, s, p.X, p.Wg, p.C,
                   p.ntok, p.hidden, p.dg, p.K, p.topk, p.ids, p.margin);
    prof_end(s);
    return e;
}

}  // namespace

cudaError_t launch_assign(const AssignLaunch &p, cudaStream_t s, int *launches)
{
    *launches += p.ntok > 0 ? 1 : 0;
    if (p.dg <= 128) return launch_assign_nj<1>(p, s);
    return launch_assign_nj<2>(p, s);
}

}  // namespace focus
