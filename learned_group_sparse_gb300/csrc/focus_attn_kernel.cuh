// Flash-attention mainloop for sm_103a on the 5th-generation tensor cores:
// TMA loads Q/K/V tiles into 128-byte-swizzled shared memory, one thread
// issues tcgen05.mma into TMEM accumulators, and a warpgroup runs the online
// softmax reading S from TMEM and writing P (bf16) back to shared memory.
//
// One CTA computes one 128-row query tile of one head:
//   warps 0-3  softmax + epilogue (thread r owns query row r = TMEM lane r)
//   warp  4    TMA producer (Q once, K/V double-buffered) + key metadata
//   warp  5    TMEM allocator and MMA issuer
// TMEM columns: S double buffer at [0,128) and [128,256), O at [256,256+D).
//
// Modes (the decomposition of the allowed-pair set of Focus attention,
// gist.science/zh technical summary 2.1.3: within-group causal attention
// plus cross-group local attention):
//   kGroup  : query/key rows are one group's gathered members (ascending
//             token order); causal in that order; a pair whose tokens share
//             several groups is scored only in the lowest shared group.
//   kWindow : original token order; keys with i - window < j <= i that share
//             no group with the query.
//   kDense  : plain causal attention (the comparison baseline).
// kGroup writes normalised fp32 partial outputs plus a base-2 log-sum-exp per
// (group member, head).  kWindow merges, in its epilogue, its own part (still
// in TMEM) with the topk group parts of the row by the exact log-sum-exp rule
// and writes the final bf16 output and natural-log lse, so the output is
// rounded to bf16 once.  kDense writes its output directly.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "focus_ptx.cuh"

namespace focus {

enum AttnMode { kGroup = 0, kWindow = 1, kDense = 2 };

struct AttnArgs {
    int B, n, Hq, Hkv;
    int rows;              // rows per batch of the Q/K/V tensors (n or n*topk packed)
    int window;
    float scale_log2;      // softmax scale * log2(e)
    int K, topk;
    const int32_t *ids;    // [B, n, topk]
    const int32_t *offsets;  // [B, K+1]
    const int32_t *pos;    // [B, n*topk]
    const int2 *tiles;     // kGroup work list: (b*K + g, tile index in group)
    const int *ntiles;     // kGroup: number of valid entries in tiles
    __nv_bfloat16 *out;    // kWindow/kDense: final O [B, n, Hq, D]
    float *lse;            // kWindow/kDense: final lse [B, Hq, n], natural log (nullable)
    float *part_out;       // kGroup: normalised partial O [B, rows, Hq, D] fp32
    float *part_lse_out;   // kGroup: partial lse [B, rows, Hq], base 2
    const float *part_o;   // kWindow: the group partials to merge (= part_out)
    const float *part_lse; // kWindow: their lse (= part_lse_out)
    const int32_t *inv;    // kWindow: [B, n, topk] index of (i, ids[i][s]) in group order
    int *status;           // device status word
    int32_t *pair_count;   // nullable: scored pairs per query (head 0)
};

constexpr int kThreads = 192;
constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // key rows per tile

template <int D>
struct AttnSmem {
    static constexpr uint32_t kTile = kBM * D * 2;           // one bf16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;               // 2 stages
    static constexpr uint32_t kV = kK + 2 * kTile;           // 2 stages
    static constexpr uint32_t kP = kV + 2 * kTile;           // 128 x 128 bf16
    static constexpr uint32_t kTok = kP + kBM * kBN * 2;     // int32 [2][128]
    static constexpr uint32_t kSig = kTok + 2 * kBN * 4;     // uint64 [2][128]
    static constexpr uint32_t kGid = kSig + 2 * kBN * 8;     // int32 [2][128][8]
    static constexpr uint32_t kBar = kGid + 2 * kBN * 8 * 4; // 17 mbarriers
    static constexpr uint32_t kMisc = kBar + 17 * 8;         // tmem slot, abort flag
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;        // slack for 1 KB alignment
};

// mbarrier slots
enum {
    B_QFULL = 0, B_KFULL = 1, B_VFULL = 3, B_KEMPTY = 5, B_VEMPTY = 7, B_SFULL = 9,
    B_SEMPTY = 11, B_PFULL = 13, B_PVDONE = 14, B_META = 15
};

// Bit mask of columns c in [lo, hi] within the 32-column word starting at c0.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int c0)
{
    int a = lo - c0, b = hi - c0;
    if (a < 0) a = 0;
    if (b > 31) b = 31;
    if (a > b) return 0u;
    const uint32_t upto_b = (b == 31) ? 0xffffffffu : ((2u << b) - 1u);
    const uint32_t below_a = (1u << a) - 1u;
    return upto_b & ~below_a;
}

template <int MODE, int D>
__global__ void __launch_bounds__(kThreads, 1)
    focus_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnArgs a)
{
    using L = AttnSmem<D>;
    constexpr int kChunks = D / 64;   // 64-column (128-byte) chunks per row

    // ---------------------------------------------------------- work item
    int h, b, q0, qend, kv_lo, nkv, g = 0, gend = 0;
    if (MODE == kGroup) {
        const int tr = blockIdx.x / a.Hq;
        h = blockIdx.x - tr * a.Hq;
        if (tr >= *a.ntiles) return;             // whole CTA leaves before any set-up
        const int2 tl = a.tiles[tr];
        b = tl.x / a.K;
        g = tl.x - b * a.K;
        const int gs = a.offsets[b * (a.K + 1) + g];
        gend = a.offsets[b * (a.K + 1) + g + 1];
        q0 = gs + kBM * tl.y;
        qend = min(q0 + kBM, gend);
        kv_lo = gs;
        nkv = tl.y + 1;
    } else {
        const int nqt = (a.n + kBM - 1) / kBM;
        h = blockIdx.x % a.Hq;
        const int rest = blockIdx.x / a.Hq;
        int qt = rest % nqt;
        b = rest / nqt;
        if (MODE == kDense) qt = nqt - 1 - qt;   // longest rows first
        q0 = kBM * qt;
        qend = min(q0 + kBM, a.n);
        if (MODE == kDense) {
            kv_lo = 0;
            nkv = qt + 1;
        } else {
            kv_lo = max(0, q0 - a.window + 1);
            nkv = a.window > 0 ? (qend - kv_lo + kBN - 1) / kBN : 0;
        }
    }
    const int kvh = h / (a.Hq / a.Hkv);

    // ------------------------------------------------------------ set-up
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *sQ = sm + L::kQ;
    uint8_t *sK = sm + L::kK;
    uint8_t *sV = sm + L::kV;
    uint8_t *sP = sm + L::kP;
    int32_t *mTok = reinterpret_cast<int32_t *>(sm + L::kTok);
    uint64_t *mSig = reinterpret_cast<uint64_t *>(sm + L::kSig);
    int32_t *mGid = reinterpret_cast<int32_t *>(sm + L::kGid);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars[B_QFULL], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_KFULL + s], 1);
            mbar_init(&bars[B_VFULL + s], 1);
            mbar_init(&bars[B_KEMPTY + s], 1);
            mbar_init(&bars[B_VEMPTY + s], 1);
            mbar_init(&bars[B_SFULL + s], 1);
            mbar_init(&bars[B_SEMPTY + s], 128);
            mbar_init(&bars[B_META + s], 32);
        }
        mbar_init(&bars[B_PFULL], 128);
        mbar_init(&bars[B_PVDONE], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 256;

    if (warp == 4) {
        // ------------------------------------------------- TMA producer
        if (lane == 0 && nkv > 0) {
            mbar_arrive_expect_tx(&bars[B_QFULL], L::kTile);
            for (int c = 0; c < kChunks; ++c)
                tma_load_4d(sQ + c * 16384, &tmQ, &bars[B_QFULL], c * 64, h, q0, b);
        }
        int issued = 0;
        for (int u = 0; u < nkv; ++u) {
            const int st = u & 1;
            const int r0 = kv_lo + kBN * u;
            bool ok = true;
            if (u >= 2 && lane == 0)
                ok = mbar_wait(&bars[B_KEMPTY + st], ((u >> 1) - 1) & 1, abort_flag, a.status);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_KFULL + st], L::kTile);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_4d(sK + st * L::kTile + c * 16384, &tmK, &bars[B_KFULL + st],
                                c * 64, kvh, r0, b);
            }
            if (u >= 2 && lane == 0)
                ok = mbar_wait(&bars[B_VEMPTY + st], ((u >> 1) - 1) & 1, abort_flag, a.status);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (MODE != kDense) {
                // key-row metadata for the mask: token index, group signature, ids
                for (int c = lane; c < kBN; c += 32) {
                    const int row = r0 + c;
                    int tok = -1;
                    if (MODE == kGroup) {
                        if (row < gend) tok = a.pos[(int64_t)b * a.rows + row];
                    } else if (row < a.n) {
                        tok = row;
                    }
                    uint64_t sig = 0;
                    if (tok >= 0) {
                        const int32_t *gp = a.ids + ((int64_t)b * a.n + tok) * a.topk;
                        for (int s = 0; s < a.topk; ++s) {
                            const int gi = gp[s];
                            sig |= 1ull << (gi & 63);
                            mGid[(st * kBN + c) * 8 + s] = gi;
                        }
                    }
                    mTok[st * kBN + c] = tok;
                    mSig[st * kBN + c] = sig;
                }
                mbar_arrive(&bars[B_META + st]);
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_VFULL + st], L::kTile);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_4d(sV + st * L::kTile + c * 16384, &tmV, &bars[B_VFULL + st],
                                c * 64, kvh, r0, b);
            }
            issued = u + 1;
            __syncwarp();
        }
        // If the CTA gave up early, let the copies already issued land before
        // shared memory is released.
        if (*abort_flag && lane == 0) {
            const uint64_t tq = global_timer_ns();
            while (nkv > 0 && !mbar_try_wait(&bars[B_QFULL], 0) &&
                   global_timer_ns() - tq < 100000000ull) {
            }
            for (int u = max(0, issued - 2); u < issued; ++u) {
                const int st = u & 1;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&bars[B_KFULL + st], (u >> 1) & 1) &&
                       global_timer_ns() - t0 < 100000000ull) {
                }
                while (!mbar_try_wait(&bars[B_VFULL + st], (u >> 1) & 1) &&
                       global_timer_ns() - t0 < 200000000ull) {
                }
            }
        }
    } else if (warp == 5) {
        // -------------------------------------------------- MMA issuer
        if (lane == 0 && nkv > 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, false, true);
            const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK);
            const uint32_t v_base = smem_u32(sV), p_base = smem_u32(sP);

            auto issue_pv = [&](int v) -> bool {
                const int st = v & 1;
                if (!mbar_wait(&bars[B_PFULL], v & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(&bars[B_VFULL + st], (v >> 1) & 1, abort_flag, a.status))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // A = P (K-major): 16 keys = 32 bytes inside a 128-byte row.
                    const uint64_t ad =
                        sdesc_sw128(p_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    // B = V (MN-major): 16 key rows of 128 bytes; the second
                    // 64-column half of D lies 16 KB further (LBO).
                    const uint64_t bd =
                        sdesc_sw128(v_base + st * L::kTile + kk * 2048, 16384, 1024);
                    tc_mma_bf16(tmem_o, ad, bd, kIdescPV, (v > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars[B_VEMPTY + st]);
                tc_commit(&bars[B_PVDONE]);
                return true;
            };

            bool ok = mbar_wait(&bars[B_QFULL], 0, abort_flag, a.status);
            for (int u = 0; ok && u < nkv; ++u) {
                const int st = u & 1;
                ok = mbar_wait(&bars[B_KFULL + st], (u >> 1) & 1, abort_flag, a.status);
                if (!ok) break;
                if (u >= 2) {
                    ok = mbar_wait(&bars[B_SEMPTY + st], ((u >> 1) - 1) & 1, abort_flag,
                                   a.status);
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t ad = sdesc_sw128(q_base + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(k_base + st * L::kTile + off, 16, 1024);
                    tc_mma_bf16(tmem + st * kBN, ad, bd, kIdescQK, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars[B_SFULL + st]);
                tc_commit(&bars[B_KEMPTY + st]);
                if (u >= 1) ok = issue_pv(u - 1);
            }
            if (ok) issue_pv(nkv - 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax warpgroup
        const int r = threadIdx.x;                       // row in tile, TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int prow = q0 + r;                         // row in the Q tensor
        bool qvalid;
        int qi;                                          // token index of the row
        uint64_t qsig = 0;
        int qg[8];
        int nq = 0;
        if (MODE == kGroup) {
            qvalid = prow < qend;
            qi = qvalid ? a.pos[(int64_t)b * a.rows + prow] : -1;
            if (qvalid) {
                const int32_t *gp = a.ids + ((int64_t)b * a.n + qi) * a.topk;
                for (int s = 0; s < a.topk; ++s) {
                    const int gi = gp[s];
                    if (gi < g) {            // groups that would own a shared pair first
                        qg[nq++] = gi;
                        qsig |= 1ull << (gi & 63);
                    }
                }
            }
        } else {
            qi = prow;
            qvalid = prow < a.n;
            if (MODE == kWindow && qvalid) {
                const int32_t *gp = a.ids + ((int64_t)b * a.n + qi) * a.topk;
                for (int s = 0; s < a.topk; ++s) {
                    const int gi = gp[s];
                    qg[nq++] = gi;
                    qsig |= 1ull << (gi & 63);
                }
            }
        }
        const bool sig_exact = a.K <= 64;
        float m_ref = -CUDART_INF_F;   // reference max (base-2 domain) applied to O and l
        float l = 0.f;
        int cnt = 0;
        bool ok = true;

        for (int u = 0; u < nkv; ++u) {
            const int st = u & 1;
            const int kvb = kv_lo + kBN * u;             // first key row of the tile
            if (MODE != kDense) {
                if (!mbar_wait(&bars[B_META + st], (u >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
            }
            if (!mbar_wait(&bars[B_SFULL + st], (u >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kBN];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(tmem + lane_off + st * kBN + c4 * 32, s + c4 * 32);
            tc_fence_before();
            mbar_arrive(&bars[B_SEMPTY + st]);

            // ---- which of the 128 keys this row may score
            uint32_t okb[4];
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                uint32_t bits;
                if (!qvalid) {
                    bits = 0u;
                } else if (MODE == kGroup) {
                    bits = range_bits(0, prow - kvb, 32 * w4);          // causal, packed order
                } else if (MODE == kWindow) {
                    bits = range_bits(qi - a.window + 1 - kvb, qi - kvb, 32 * w4);
                } else {
                    bits = range_bits(0, qi - kvb, 32 * w4);
                }
                if (MODE != kDense && nq > 0) {
                    uint32_t cand = bits;
                    while (cand) {
                        const int cc = __ffs(cand) - 1;
                        cand &= cand - 1u;
                        const int c = 32 * w4 + cc;
                        if (mSig[st * kBN + c] & qsig) {
                            bool share = sig_exact;
                            if (!share) {
                                const int32_t *gj = mGid + (st * kBN + c) * 8;
                                for (int x = 0; x < nq && !share; ++x)
                                    for (int y = 0; y < a.topk; ++y)
                                        if (gj[y] == qg[x]) share = true;
                            }
                            if (share) bits &= ~(1u << cc);
                        }
                    }
                }
                okb[w4] = bits;
            }
            if (a.pair_count)
                cnt += __popc(okb[0]) + __popc(okb[1]) + __popc(okb[2]) + __popc(okb[3]);

            float mx = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                const bool on = (okb[c >> 5] >> (c & 31)) & 1u;
                s[c] = on ? s[c] * a.scale_log2 : -CUDART_INF_F;
                mx = fmaxf(mx, s[c]);
            }

            // P(u-1) consumed and O updated by the previous P.V product.
            if (u >= 1) {
                if (!mbar_wait(&bars[B_PVDONE], (u - 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            // Lazy rescaling: keep the reference max unless the row max
            // grows by more than 2^8.
            const float m_new = fmaxf(m_ref, mx);
            const bool grow = (m_ref == -CUDART_INF_F) || (m_new > m_ref + 8.f);
            const bool resc = grow && l > 0.f;
            const float new_ref = grow ? m_new : m_ref;
            if (__any_sync(0xffffffffu, resc)) {
                const float f = resc ? exp2f(m_ref - new_ref) : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem_o + lane_off + c * 32, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= f;
                    tmem_st32(tmem_o + lane_off + c * 32, o);
                }
                tmem_st_wait();
                l *= f;
            }
            m_ref = new_ref;
            const float ref = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;

            // ---- P = 2^(s - ref) in bf16, 128-byte swizzled, K-major
            float rs = 0.f;
            const uint32_t p_row = smem_u32(sP) + r * 128;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) {
                    float p[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = exp2f(s[half * 64 + uu * 8 + e] - ref);
                        rs += p[e];
                    }
                    st_shared_v4(p_row + half * 16384 + ((uu ^ (r & 7)) << 4),
                                 pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                 pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
                }
            }
            l += rs;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL]);
        }

        // ---- epilogue
        if (ok && nkv > 0) {
            ok = mbar_wait(&bars[B_PVDONE], (nkv - 1) & 1, abort_flag, a.status);
            tc_fence_after();
        }
        const bool has = ok && l > 0.f;
        const float lse2 = has ? m_ref + log2f(l) : -CUDART_INF_F;   // this kernel's part
        // Output scale of the TMEM accumulator (which holds sum p v with
        // p = 2^(s - m_ref)) and, for kWindow, the merge with the group parts.
        float fo = has ? 1.f / l : 0.f;
        float L2 = lse2;
        int64_t prt[8];
        float wpart[8];
        if (MODE == kWindow) {
            // Exact softmax over the union of the window part and the topk
            // group parts: L = log2 sum_p 2^{L_p}, O = sum_p 2^{L_p - L} O_p.
            float m = lse2;
            const int nk = a.n * a.topk;     // group-order rows per batch
            for (int s = 0; s < a.topk; ++s) {
                prt[s] = -1;
                wpart[s] = -CUDART_INF_F;
                if (qvalid) {
                    const int r = a.inv[((int64_t)b * a.n + qi) * a.topk + s];
                    if ((unsigned)r < (unsigned)nk) {
                        prt[s] = ((int64_t)b * nk + r) * a.Hq + h;
                        wpart[s] = a.part_lse[prt[s]];
                    }
                }
                m = fmaxf(m, wpart[s]);
            }
            if (m == -CUDART_INF_F) {
                L2 = -CUDART_INF_F;
                fo = 0.f;
                for (int s = 0; s < a.topk; ++s) wpart[s] = 0.f;
            } else {
                float sum = exp2f(lse2 - m);
                for (int s = 0; s < a.topk; ++s) sum += exp2f(wpart[s] - m);
                L2 = m + log2f(sum);
                fo = has ? exp2f(m_ref - L2) : 0.f;     // 2^{L_w - L} / l
                for (int s = 0; s < a.topk; ++s) wpart[s] = exp2f(wpart[s] - L2);
            }
        }
        int64_t orow = 0;
        if (MODE == kGroup)
            orow = ((int64_t)b * a.rows + prow) * a.Hq + h;
        else
            orow = ((int64_t)b * a.n + qi) * a.Hq + h;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float o[32];
            if (nkv > 0) {
                tmem_ld32(tmem_o + lane_off + c * 32, o);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= fo;
            if (!qvalid) continue;
            if (MODE == kGroup) {
                float4 *dst = reinterpret_cast<float4 *>(a.part_out + orow * D + c * 32);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                continue;
            }
            if (MODE == kWindow) {
                for (int s = 0; s < a.topk; ++s) {
                    if (wpart[s] == 0.f) continue;
                    const float4 *src =
                        reinterpret_cast<const float4 *>(a.part_o + prt[s] * D + c * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 v = src[q];
                        o[4 * q] = fmaf(wpart[s], v.x, o[4 * q]);
                        o[4 * q + 1] = fmaf(wpart[s], v.y, o[4 * q + 1]);
                        o[4 * q + 2] = fmaf(wpart[s], v.z, o[4 * q + 2]);
                        o[4 * q + 3] = fmaf(wpart[s], v.w, o[4 * q + 3]);
                    }
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + orow * D);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 v;
                v.x = pack_bf16x2(o[q * 8 + 0], o[q * 8 + 1]);
                v.y = pack_bf16x2(o[q * 8 + 2], o[q * 8 + 3]);
                v.z = pack_bf16x2(o[q * 8 + 4], o[q * 8 + 5]);
                v.w = pack_bf16x2(o[q * 8 + 6], o[q * 8 + 7]);
                dst[c * 4 + q] = v;
            }
        }
        if (qvalid) {
            if (MODE == kGroup) {
                a.part_lse_out[orow] = lse2;
            } else if (a.lse) {
                a.lse[((int64_t)b * a.Hq + h) * a.n + qi] = L2 * 0.69314718055994531f;
            }
            if (a.pair_count && h == 0) atomicAdd(&a.pair_count[(int64_t)b * a.n + qi], cnt);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace focus
