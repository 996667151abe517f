// Forward of soft-gated training attention on the 5th-generation tensor cores
// (Focus, gist.science/zh technical summary 2.1.2 "gated attention": for
// every causal pair, s_ij = q_i . k_j * scale * gate_ij with gate_ij = 1
// inside the local window (i - j < w) and sigma(lambda * g_i . g_j)
// elsewhere; gist.science/nl Kerncomponent 4: soft gates over all pairs while
// training).
//
// The warp-specialised layout of the prefill attention kernel with a second
// product per key tile.  One CTA takes two 128-row query tiles, its halves
// h = 0, 1 (two heads that share a key/value head, or two consecutive query
// tiles of one head), against one stream of 64-row key tiles.  One thread
// issues, per key tile u,
//   S_h = Q_h K_u^T       bf16, fp32 accumulation
//   A_h = Gq_h Gk_u^T     fp16 soft assignments (K_g padded to 16 with zeros);
//                         skipped when every pair of the tile is local
//   O_h += P_h V_u        P_h in TMEM (bf16, over the first 32 columns of S_h)
// in the order S_0 A_0 (u), O_1 += P_1 V (u-1), S_1 A_1 (u), O_0 += P_0 V (u),
// so that one half's softmax overlaps the other half's products; the tensor
// pipe runs in issue order, so S_h(u) complete implies O_h += P_h(u-1) V
// complete.  A softmax thread owns one query row (TMEM lane): one 128-column
// TMEM load brings S_h and A_h of its row, it forms the base-2 logits
// x = s * scale * log2(e) * gate, masks j > i, and writes P = 2^(x - ref).
// TMEM columns: S_0 [0,64), A_0 [64,128), S_1 [128,192), A_1 [192,256),
// O_0 [256, 256+D), O_1 [384, 384+D).
//
// Persistent (one CTA per SM walks the work items, heaviest first); TMA loads
// Q and Gq per half and K, V and Gk per key tile (a 3-deep ring when it fits
// in shared memory); every wait is bounded and a CTA that gives up drains its
// copies and MMAs before it releases shared memory and TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "focus_attn_kernel.cuh"
#include "focus_internal.h"

namespace focus {

namespace {

constexpr int kGM = 128;   // query rows per tile (one TMEM lane each)
constexpr int kGN = 64;    // key rows per tile

// mbarrier slots: [half] pairs, then [stage] triples
enum {
    G_QFULL = 0, G_QEMPTY = 2, G_SFULL = 4, G_PFULL = 6, G_ODONE = 8, G_IFULL = 10,
    G_IEMPTY = 12, G_KFULL = 14, G_KEMPTY = 17, G_VFULL = 20, G_VEMPTY = 23, G_DRAIN = 26,
    kGBars = 27
};

// Shared memory of one CTA: D columns of bf16 per Q/K/V row, KPC chunks of 64
// fp16 per G row; every tile is a whole number of 1024-byte swizzle atoms.
template <int D, int KPC>
struct GtcSmem {
    static constexpr int NS = (D == 128 && KPC == 2) ? 2 : 3;   // K/V/Gk stages
    static constexpr uint32_t kQT = kGM * D * 2;        // query tile: D/64 chunks of 16 KB
    static constexpr uint32_t kGqT = kGM * KPC * 128;   // Gq tile: chunks of 16 KB
    static constexpr uint32_t kKT = kGN * D * 2;        // key or value tile: chunks of 8 KB
    static constexpr uint32_t kGkT = kGN * KPC * 128;   // Gk tile: chunks of 8 KB
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kGq = kQ + 2 * kQT;
    static constexpr uint32_t kK = kGq + 2 * kGqT;
    static constexpr uint32_t kV = kK + NS * kKT;
    static constexpr uint32_t kGk = kV + NS * kKT;
    static constexpr uint32_t kBar = kGk + NS * kGkT;
    static constexpr uint32_t kRing = kBar + 256;       // 2 work-item slots of 64 bytes
    static constexpr uint32_t kMisc = kRing + 128;      // TMEM base, abort flag
    static constexpr uint32_t kBytes = kMisc + 16 + 1024;   // + alignment slack
    static_assert(kGBars * 8 <= 256, "barrier block");
    static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct GtcArgs {
    int B, n, Hq, Hkv, nks, window, pair_heads;
    float scale2;        // scale * log2(e)
    float half_scale2;   // scale2 / 2
    float half_lambda;   // lambda / 2
    __nv_bfloat16 *out;  // [B, n, Hq, D]
    float *lse;          // [B, Hq, n], natural log
    int *status;
};

// A work item: half h has query rows [q0[h], qend[h]) of head hd[h] and key
// tiles [0, uhi[h]) (none when uhi[h] = 0); the item streams nkv key tiles.
struct GItem {
    int b, nkv, hd[2], q0[2], qend[2], uhi[2];
};

__device__ __forceinline__ void gput(int *p, const GItem &w)
{
    p[0] = w.b;
    p[1] = w.nkv;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        p[2 + h] = w.hd[h];
        p[4 + h] = w.q0[h];
        p[6 + h] = w.qend[h];
        p[8 + h] = w.uhi[h];
    }
}

__device__ __forceinline__ GItem gget(const int *p)
{
    GItem w;
    w.b = p[0];
    w.nkv = p[1];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        w.hd[h] = p[2 + h];
        w.q0[h] = p[4 + h];
        w.qend[h] = p[6 + h];
        w.uhi[h] = p[8 + h];
    }
    return w;
}

__host__ __device__ __forceinline__ int gtc_query_pairs(int n, int pair_heads)
{
    const int nqt = (n + kGM - 1) / kGM;
    return pair_heads ? nqt : (nqt + 1) / 2;
}

__host__ __device__ __forceinline__ int gtc_items(int B, int n, int Hq, int pair_heads)
{
    return B * gtc_query_pairs(n, pair_heads) * (pair_heads ? Hq / 2 : Hq);
}

// Work item -> its two query tiles.  Head slots vary fastest (items that
// share key tiles run side by side), the last query tiles (most keys) first.
__device__ __forceinline__ GItem gdecode(const GtcArgs &a, int item)
{
    GItem w;
    const int hsl = a.pair_heads ? a.Hq / 2 : a.Hq;
    const int hs = item % hsl;
    const int rest = item / hsl;
    const int nq = gtc_query_pairs(a.n, a.pair_heads);
    const int qp = nq - 1 - rest % nq;
    w.b = rest / nq;
    const int t0 = a.pair_heads ? qp : 2 * qp;
    w.nkv = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        w.hd[h] = a.pair_heads ? 2 * hs + h : hs;
        w.q0[h] = kGM * ((a.pair_heads || h == 0) ? t0 : t0 + 1);
        w.qend[h] = min(w.q0[h] + kGM, a.n);
        if (w.qend[h] <= w.q0[h]) {
            w.qend[h] = w.q0[h];
            w.uhi[h] = 0;
        } else {
            w.uhi[h] = (w.qend[h] + kGN - 1) / kGN;   // causal: keys [0, qend)
        }
        w.nkv = max(w.nkv, w.uhi[h]);
    }
    return w;
}

// Some pair of the tile (rows up to qend - 1, keys from kvb) lies outside
// the window, so the tile needs the gate product.
__device__ __forceinline__ bool tile_gated(int qend, int kvb, int window)
{
    return qend - 1 - kvb >= window;
}

// tanh with the hardware approximation (relative error about 2^-11, below
// the fp16 rounding of the G products)
__device__ __forceinline__ float tanh_fast(float x)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
    return t;
}

// (x0, x1) * s on two fp32 lanes in one instruction.
__device__ __forceinline__ void mul2(float &d0, float &d1, float x0, float x1, float s)
{
    asm("{\n\t.reg .b64 rx, rs, rd;\n\t"
        "mov.b64 rx, {%2, %3};\n\t"
        "mov.b64 rs, {%4, %4};\n\t"
        "mul.rn.f32x2 rd, rx, rs;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(x0), "f"(x1), "f"(s));
}

// (x0, x1) * (y0, y1) on two fp32 lanes in one instruction.
__device__ __forceinline__ void mulv2(float &x0, float &x1, float y0, float y1)
{
    asm("{\n\t.reg .b64 rx, ry, rd;\n\t"
        "mov.b64 rx, {%0, %1};\n\t"
        "mov.b64 ry, {%2, %3};\n\t"
        "mul.rn.f32x2 rd, rx, ry;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(y0), "f"(y1));
}

template <int D, int KPC>
__global__ void __launch_bounds__(kThreads, 1)
    gated_tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmGq,
                        const __grid_constant__ CUtensorMap tmGk, const GtcArgs a)
{
    using L = GtcSmem<D, KPC>;
    constexpr int NS = L::NS;
    constexpr int kChunks = D / 64;

    const int nitems = gtc_items(a.B, a.n, a.Hq, a.pair_heads);
    if ((int)blockIdx.x >= nitems) return;
    const int kv_per_q = a.Hq / a.Hkv;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sQ = sm + L::kQ;
    uint8_t *sGq = sm + L::kGq;
    uint8_t *sK = sm + L::kK;
    uint8_t *sV = sm + L::kV;
    uint8_t *sGk = sm + L::kGk;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kBar);
    int *ring = reinterpret_cast<int *>(sm + L::kRing);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bars[G_QFULL + h], 1);
            mbar_init(&bars[G_QEMPTY + h], 1);
            mbar_init(&bars[G_SFULL + h], 1);
            mbar_init(&bars[G_PFULL + h], 4);    // one lane per warp of the half
            mbar_init(&bars[G_ODONE + h], 1);
            mbar_init(&bars[G_IFULL + h], 32);   // the producer warp
            mbar_init(&bars[G_IEMPTY + h], 9);   // 8 softmax warps + the MMA thread
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars[G_KFULL + s], 1);
            mbar_init(&bars[G_KEMPTY + s], 1);
            mbar_init(&bars[G_VFULL + s], 1);
            mbar_init(&bars[G_VEMPTY + s], 1);
        }
        mbar_init(&bars[G_DRAIN], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmGq);
        tma_prefetch_desc(&tmGk);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 256;   // O_0; O_1 at + 128
    // (set-up above touches no global memory; launched with launch_pdl after
    // the kernel that converts G to fp16)
    grid_dep_sync();

    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
        if (warp == kProducerWarp) {
            // ------------------------------------------------- TMA producer
            int T = 0;                    // key tiles issued so far
            int iq[2] = {0, 0};           // query tiles loaded per half
            bool ok = true;
            for (int k = 0, item = blockIdx.x; ok && item < nitems;
                 item = item_of(++k, blockIdx.x, gridDim.x)) {
                // ring slot k & 1 is free once item k - 2 is fully consumed
                if (k >= 2 && lane == 0)
                    ok = mbar_wait(&bars[G_IEMPTY + (k & 1)], ((k >> 1) - 1) & 1, abort_flag,
                                   a.status);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                const GItem w = gdecode(a, item);
                if (lane == 0) gput(ring + (k & 1) * 16, w);
                __syncwarp();
                mbar_arrive(&bars[G_IFULL + (k & 1)]);
                if (w.nkv == 0) continue;
                const int kvh = w.hd[0] / kv_per_q;
                // Q_h and Gq_h: free once the last products of the half's
                // previous item are done
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (w.uhi[h] == 0) continue;
                    if (iq[h] >= 1 && lane == 0)
                        ok = mbar_wait(&bars[G_QEMPTY + h], (iq[h] - 1) & 1, abort_flag, a.status);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[G_QFULL + h], L::kQT + L::kGqT);
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_4d(sQ + h * L::kQT + c * 16384, &tmQ, &bars[G_QFULL + h],
                                        c * 64, w.hd[h], w.q0[h], w.b);
                        for (int c = 0; c < KPC; ++c)
                            tma_load_4d(sGq + h * L::kGqT + c * 16384, &tmGq, &bars[G_QFULL + h],
                                        c * 64, 0, w.q0[h], w.b);
                    }
                    ++iq[h];
                }
                if (!ok) break;
                for (int u = 0; u < w.nkv; ++u, ++T) {
                    const int st = T % NS;
                    const uint32_t par = ((T / NS) & 1) ^ 1;   // phase of the stage's last use
                    if (T >= NS && lane == 0)
                        ok = mbar_wait(&bars[G_KEMPTY + st], par, abort_flag, a.status);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[G_KFULL + st], L::kKT + L::kGkT);
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_4d(sK + st * L::kKT + c * 8192, &tmK, &bars[G_KFULL + st],
                                        c * 64, kvh, kGN * u, w.b);
                        for (int c = 0; c < KPC; ++c)
                            tma_load_4d(sGk + st * L::kGkT + c * 8192, &tmGk, &bars[G_KFULL + st],
                                        c * 64, 0, kGN * u, w.b);
                    }
                    if (T >= NS && lane == 0)
                        ok = mbar_wait(&bars[G_VEMPTY + st], par, abort_flag, a.status);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[G_VFULL + st], L::kKT);
                        for (int c = 0; c < kChunks; ++c)
                            tma_load_4d(sV + st * L::kKT + c * 8192, &tmV, &bars[G_VFULL + st],
                                        c * 64, kvh, kGN * u, w.b);
                    }
                    __syncwarp();
                }
            }
            // A CTA that gave up lets the copies already issued land before
            // shared memory is released.
            if (*abort_flag && lane == 0) {
                const uint64_t t0 = global_timer_ns();
                for (int h = 0; h < 2; ++h)
                    while (iq[h] > 0 && !mbar_try_wait(&bars[G_QFULL + h], (iq[h] - 1) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                for (int t = max(0, T - NS); t <= T; ++t) {
                    const int st = t % NS;
                    const uint32_t par = (t / NS) & 1;
                    while (!mbar_try_wait(&bars[G_KFULL + st], par) &&
                           global_timer_ns() - t0 < 200000000ull) {
                    }
                    while (!mbar_try_wait(&bars[G_VFULL + st], par) &&
                           global_timer_ns() - t0 < 300000000ull) {
                    }
                }
            }
        } else if (warp == kMmaWarp) {
            // -------------------------------------------------- MMA issuer
            if (lane == 0) {
                constexpr uint32_t kIdQK = idesc_bf16_f32(kGM, kGN, false, false);
                constexpr uint32_t kIdA = idesc_f16_f32(kGM, kGN);
                constexpr uint32_t kIdPV = idesc_bf16_f32(kGM, D, false, true);
                constexpr uint32_t kHi = sdesc_hi(1024);
                // low descriptor words of the first tile of each buffer; a
                // tile or a step inside one is an added constant
                const uint32_t dq0 = sdesc_lo(smem_u32(sQ), 16);
                const uint32_t dgq0 = sdesc_lo(smem_u32(sGq), 16);
                const uint32_t dk0 = sdesc_lo(smem_u32(sK), 16);
                const uint32_t dgk0 = sdesc_lo(smem_u32(sGk), 16);
                // V is MN-major: the second 64-column chunk of D lies one
                // 64-row chunk (8 KB) further (leading offset)
                const uint32_t dv0 = sdesc_lo(smem_u32(sV), kGN * 128);
                int T = 0;
                int iq[2] = {0, 0};   // Q loads consumed per half
                int np[2] = {0, 0};   // P.V products issued per half
                bool ok = true;
                for (int k = 0, item = blockIdx.x; ok && item < nitems;
                     item = item_of(++k, blockIdx.x, gridDim.x)) {
                    ok = mbar_wait(&bars[G_IFULL + (k & 1)], (k >> 1) & 1, abort_flag, a.status);
                    if (!ok) break;
                    const GItem w = gget(ring + (k & 1) * 16);
                    mbar_arrive(&bars[G_IEMPTY + (k & 1)]);
                    if (w.nkv == 0) continue;
                    bool qready[2] = {false, false}, first[2] = {true, true};
                    int kready = -1, vready = -1;
                    // S_h = Q_h K_u^T and, for a gated tile, A_h = Gq_h Gk_u^T
                    auto issue_qk = [&](int h, int u) -> bool {
                        const int t = T + u, st = t % NS;
                        if (kready < u) {
                            if (!mbar_wait(&bars[G_KFULL + st], (t / NS) & 1, abort_flag, a.status))
                                return false;
                            kready = u;
                        }
                        if (!qready[h]) {
                            if (!mbar_wait(&bars[G_QFULL + h], iq[h] & 1, abort_flag, a.status))
                                return false;
                            qready[h] = true;
                        }
                        tc_fence_after();
                        const uint32_t qd = dq0 + h * (L::kQT >> 4), kd = dk0 + st * (L::kKT >> 4);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // 16 columns = 32 bytes; 64 columns = one chunk
                            const uint32_t qo = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                            const uint32_t ko = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                            tc_mma_bf16_lo<kHi, kHi>(tmem + h * 128, qd + qo, kd + ko, kIdQK,
                                                     kk > 0 ? 1u : 0u);
                        }
                        if (tile_gated(w.qend[h], kGN * u, a.window)) {
                            const uint32_t gq = dgq0 + h * (L::kGqT >> 4);
                            const uint32_t gk = dgk0 + st * (L::kGkT >> 4);
#pragma unroll
                            for (int ks = 0; ks < 4 * KPC; ++ks) {
                                if (ks >= a.nks) break;
                                const uint32_t qo = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                                const uint32_t ko = ((ks >> 2) * 8192 + (ks & 3) * 32) >> 4;
                                tc_mma_bf16_lo<kHi, kHi>(tmem + h * 128 + 64, gq + qo, gk + ko,
                                                         kIdA, ks > 0 ? 1u : 0u);
                            }
                        }
                        tc_commit(&bars[G_SFULL + h]);
                        if (u == w.uhi[h] - 1) tc_commit(&bars[G_QEMPTY + h]);
                        return true;
                    };
                    // O_h += P_h(u) V_u
                    auto issue_pv = [&](int h, int u) -> bool {
                        const int t = T + u, st = t % NS;
                        if (vready < u) {
                            if (!mbar_wait(&bars[G_VFULL + st], (t / NS) & 1, abort_flag, a.status))
                                return false;
                            vready = u;
                        }
                        if (!mbar_wait(&bars[G_PFULL + h], np[h] & 1, abort_flag, a.status))
                            return false;
                        tc_fence_after();
                        const uint32_t vd = dv0 + st * (L::kKT >> 4);
                        const uint32_t acc0 = first[h] ? 0u : 1u;
#pragma unroll
                        for (int kk = 0; kk < kGN / 16; ++kk)
                            // A = P_h: 16 keys = 8 TMEM columns; B = V: 16 key rows of
                            // 128 bytes (2 KB) per step
                            tc_mma_bf16_ts_lo<kHi>(tmem_o + h * 128, tmem + h * 128 + kk * 8,
                                                   vd + ((kk * 2048) >> 4), kIdPV,
                                                   kk > 0 ? 1u : acc0);
                        first[h] = false;
                        ++np[h];
                        if (u == w.uhi[h] - 1) tc_commit(&bars[G_ODONE + h]);
                        return true;
                    };
                    const int nkv = w.nkv;
                    for (int u = 0; ok && u <= nkv; ++u) {
                        if (u < nkv && u < w.uhi[0]) ok = issue_qk(0, u);
                        if (ok && u >= 1) {
                            if (u - 1 < w.uhi[1]) ok = issue_pv(1, u - 1);
                            if (ok) tc_commit(&bars[G_VEMPTY + (T + u - 1) % NS]);   // V(u-1) read
                        }
                        if (ok && u < nkv) {
                            if (u < w.uhi[1]) ok = issue_qk(1, u);
                            if (ok) tc_commit(&bars[G_KEMPTY + (T + u) % NS]);       // K, Gk(u) read
                        }
                        if (ok && u < nkv && u < w.uhi[0]) ok = issue_pv(0, u);
                    }
                    T += nkv;
#pragma unroll
                    for (int h = 0; h < 2; ++h) iq[h] += w.uhi[h] > 0 ? 1 : 0;
                }
                // every MMA issued completes before TMEM is released
                tc_commit(&bars[G_DRAIN]);
                mbar_wait_until(&bars[G_DRAIN], 0, global_timer_ns() + 500000000ull);
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------ softmax of half hh = warp / 4
        const int hh = warp >> 2;
        const int r = threadIdx.x & 127;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_off + hh * 128;    // S_h, then A_h
        const uint32_t o_col = tmem_o + lane_off + hh * 128;  // O_h
        int ns = 0;     // S_h tiles consumed
        int nod = 0;    // O_h completions
        bool ok = true;
        for (int k = 0, item = blockIdx.x; ok && item < nitems;
             item = item_of(++k, blockIdx.x, gridDim.x)) {
            const int slot = k & 1;
            ok = mbar_wait(&bars[G_IFULL + slot], (k >> 1) & 1, abort_flag, a.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int *wi = ring + slot * 16;
            const int wb = wi[0], hd = wi[2 + hh], q0 = wi[4 + hh], qend = wi[6 + hh];
            const int uhi = wi[8 + hh];
            const int i = q0 + r;               // this row's query token
            const bool qvalid = i < qend;
            float m_ref = -CUDART_INF_F;        // reference max (base 2) of O_h and l
            float l = 0.f;
            for (int u = 0; u < uhi; ++u) {
                const int kvb = kGN * u;
                ok = mbar_wait(&bars[G_SFULL + hh], ns & 1, abort_flag, a.status);
                ++ns;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                float s[128];
                tmem_ld128(s_col, s);   // S_h: columns 0-63, A_h: 64-127
                // base-2 logits x = s * scale * log2(e) * gate
                const int lim = qvalid ? i - kvb : -1;   // keys c <= lim are causal
                const int loc = i - kvb - a.window;      // keys c <= loc are gated
                if (!tile_gated(qend, kvb, a.window)) {
#pragma unroll
                    for (int c = 0; c < kGN; c += 2) mul2(s[c], s[c + 1], s[c], s[c + 1], a.scale2);
                } else if (__all_sync(0xffffffffu, loc >= kGN - 1)) {
                    // every pair of the warp's rows is gated:
                    // scale2 * sigma(lambda a) = scale2/2 + scale2/2 * tanh(lambda a / 2)
#pragma unroll
                    for (int c = 0; c < kGN; c += 2) {
                        float z0, z1, g0, g1;
                        mul2(z0, z1, s[kGN + c], s[kGN + c + 1], a.half_lambda);
                        fma2(g0, g1, tanh_fast(z0), tanh_fast(z1), a.half_scale2, a.half_scale2);
                        mulv2(s[c], s[c + 1], g0, g1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kGN; ++c) {
                        const float g =
                            fmaf(a.half_scale2, tanh_fast(a.half_lambda * s[kGN + c]), a.half_scale2);
                        s[c] *= (c <= loc) ? g : a.scale2;
                    }
                }
                if (__any_sync(0xffffffffu, lim < kGN - 1)) {
#pragma unroll
                    for (int c = 0; c < kGN; ++c) s[c] = (c <= lim) ? s[c] : -CUDART_INF_F;
                }
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float m = fmax3(s[e], s[8 + e], s[16 + e]);
                    m = fmax3(m, s[24 + e], s[32 + e]);
                    m = fmax3(m, s[40 + e], s[48 + e]);
                    mx8[e] = fmaxf(m, s[56 + e]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                // lazy rescaling: keep the reference max unless the row max
                // grows by more than 2^8
                const float m_new = fmaxf(m_ref, mx);
                const bool grow = (m_ref == -CUDART_INF_F) || (m_new > m_ref + 8.f);
                const bool resc = grow && m_ref != -CUDART_INF_F;
                const float new_ref = grow ? m_new : m_ref;
                const float f = resc ? exp2f(m_ref - new_ref) : 1.f;
                const bool any_resc = __any_sync(0xffffffffu, resc);
                m_ref = new_ref;
                const float nref = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;
                // P = 2^(x - ref) in bf16 over the first 32 columns of S_h
                // (keys 2c, 2c+1 in column c): the A operand of P.V
                float rs8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float x0 = s[2 * j], x1 = s[2 * j + 1];
                    add2(x0, x1, nref, nref);
                    const float p0 = exp2f(x0), p1 = exp2f(x1);
                    add2(rs8[2 * (j & 3)], rs8[2 * (j & 3) + 1], p0, p1);
                    pk[j] = pack_bf16x2(p0, p1);
                }
                tmem_st32u(s_col, pk);
                tmem_st_wait();
                l = fmaf(l, f, ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) +
                                   ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7])));
                // O_h += P_h(u-1) V precedes S_h(u) on the tensor pipe: a
                // rescale needs no wait
                if (any_resc) rescale_o<D>(o_col, f);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[G_PFULL + hh]);
            }
            if (!ok) break;

            // ---- epilogue: O / l in bf16, the log-sum-exp (natural log)
            if (uhi > 0) {
                ok = mbar_wait(&bars[G_ODONE + hh], nod & 1, abort_flag, a.status);
                ++nod;
                tc_fence_after();
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            const bool has = l > 0.f;
            const float inv_l = has ? 1.f / l : 0.f;
            float o[D];
            if (uhi > 0) {
                if constexpr (D == 128) {
                    tmem_ld128(o_col, o);
                } else {
                    tmem_ld32(o_col, o);
                    tmem_ld32(o_col + 32, o + 32);
                }
            } else {
#pragma unroll
                for (int e = 0; e < D; ++e) o[e] = 0.f;
            }
            if (qvalid) {
                a.lse[((int64_t)wb * a.Hq + hd) * a.n + i] =
                    has ? (m_ref + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.out + (((int64_t)wb * a.n + i) * a.Hq + hd) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    dst[c] = make_uint4(pack_bf16x2(o[8 * c] * inv_l, o[8 * c + 1] * inv_l),
                                        pack_bf16x2(o[8 * c + 2] * inv_l, o[8 * c + 3] * inv_l),
                                        pack_bf16x2(o[8 * c + 4] * inv_l, o[8 * c + 5] * inv_l),
                                        pack_bf16x2(o[8 * c + 6] * inv_l, o[8 * c + 7] * inv_l));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[G_IEMPTY + slot]);   // ring slot no longer read
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, int KPC>
cudaError_t gtc_preflight_t()
{
    auto kern = gated_tc_fwd_kernel<D, KPC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)GtcSmem<D, KPC>::kBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    // the warpgroups' shares after setmaxnreg must fit in the launch's registers
    if ((int64_t)fa.numRegs * kThreads < 256 * kRegsSoftmax + 128 * kRegsOther)
        return cudaErrorInvalidConfiguration;
    return cudaSuccess;
}

template <int D, int KPC>
cudaError_t gtc_launch_t(const GatedTcPlan &plan, cudaStream_t s, int *launches)
{
    const GatedLaunch &p = plan.p;
    GtcArgs a;
    a.B = p.B;
    a.n = p.n;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.nks = plan.kp / 16;
    a.window = std::min(p.window, p.n);   // i - j < n for every pair
    a.pair_heads = plan.pair_heads;
    a.scale2 = p.scale * 1.4426950408889634f;
    a.half_scale2 = 0.5f * a.scale2;
    a.half_lambda = 0.5f * p.lambda;
    a.out = p.out;
    a.lse = p.lse_out;
    a.status = p.wc.status;
    prof_begin("gated_fwd", s);
    const cudaError_t e =
        launch_pdl(gated_tc_fwd_kernel<D, KPC>, dim3((unsigned)plan.grid), dim3(kThreads),
                   (size_t)GtcSmem<D, KPC>::kBytes, s, plan.map[0], plan.map[1], plan.map[2],
                   plan.map[3], plan.map[4], a);
    prof_end(s);
    *launches += 1;
    return e;
}

}  // namespace

cudaError_t gated_tc_preflight(int d, int Kg)
{
    const bool two = Kg > 64;
    if (d == 64) return two ? gtc_preflight_t<64, 2>() : gtc_preflight_t<64, 1>();
    return two ? gtc_preflight_t<128, 2>() : gtc_preflight_t<128, 1>();
}

cudaError_t gated_tc_prepare(const GatedLaunch &p, const __half *g16, int kp, GatedTcPlan *plan)
{
    cudaError_t e = gated_tc_preflight(p.d, p.Kg);
    if (e != cudaSuccess) return e;
    plan->p = p;
    plan->kp = kp;
    plan->pair_heads = (p.Hq / p.Hkv) % 2 == 0 ? 1 : 0;
    if (!make_map_4d(&plan->map[0], p.q, false, p.B, p.n, p.Hq, p.d, kGM) ||
        !make_map_4d(&plan->map[1], p.k, false, p.B, p.n, p.Hkv, p.d, kGN) ||
        !make_map_4d(&plan->map[2], p.v, false, p.B, p.n, p.Hkv, p.d, kGN) ||
        !make_map_4d(&plan->map[3], g16, true, p.B, p.n, 1, kp, kGM) ||
        !make_map_4d(&plan->map[4], g16, true, p.B, p.n, 1, kp, kGN))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    plan->grid = std::min(gtc_items(p.B, p.n, p.Hq, plan->pair_heads), sms);
    return cudaSuccess;
}

cudaError_t gated_tc_launch(const GatedTcPlan &plan, cudaStream_t s, int *launches)
{
    const bool two = plan.p.Kg > 64;
    if (plan.p.d == 64)
        return two ? gtc_launch_t<64, 2>(plan, s, launches) : gtc_launch_t<64, 1>(plan, s, launches);
    return two ? gtc_launch_t<128, 2>(plan, s, launches) : gtc_launch_t<128, 1>(plan, s, launches);
}

}  // namespace focus
