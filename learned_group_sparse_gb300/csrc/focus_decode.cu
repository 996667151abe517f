// Decode: one new token per sequence against a key/value cache whose group
// memberships are kept as per-group position lists (Focus, gist.science/zh
// technical summary 2.1.3 and gist.science/nl Kerncomponent 4: at inference a
// token belongs to its k highest-scoring groups and attends, with an exact
// softmax, to the keys in its local window or sharing one of its groups).
//
// Group lists: glen[b][g] entries of gpos[b][g][0..cap), token positions in
// ascending order.  decode_lists_init copies a prefill's bucketing
// (offsets, pos) into that layout; after the attention the new token joins
// the end of its k lists (positions only grow, so the order holds).
//
// Attention of the new token i = L - 1 over its allowed set, split without
// overlap into
//   window keys  j in [i - w + 1, i]                    (every one allowed;
//                at w = 0 the token's own key, through its own groups), and
//   group keys   j in the list of g, i - j >= w, with g = min(G_i n G_j)
//                (a pair sharing several groups is taken from the lowest).
// The keys form one virtual sequence: the window, then the k lists.
//
// decode_attn_kernel: CTA (split p, kv-head group, batch) takes an equal
// slice of the virtual keys, maps it to positions once for all heads of its
// group (dropping list keys that belong to a lower shared group), and streams
// the kept keys' K and V rows in stages: one bulk copy per key and tensor
// carries the rows of all HG heads of the group, which lie side by side in
// the cache, so HBM sees runs of HG * d * 2 bytes.  A copy warp fills a
// three-stage ring; eight MMA warps each take one (head, 16-key block) of a
// stage: S = Q K^T and O += P V as m16n8k16 bf16 MMAs (the query heads of a
// kv head are the tile's rows, fp32 accumulation) with an online softmax.
// The warps of a head are merged in the CTA; decode_merge_kernel combines
// the P splits per query head and then appends the new tokens to the lists.
// HBM-bound: the K and V rows of the allowed keys are the bytes that matter.
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"
#include "focus_ptx.cuh"
#include "focus_wait.cuh"

namespace focus {

namespace {

constexpr int kDecWarps = 8;                       // MMA warps; one more warp copies
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecBlk = 16;          // keys per warp block: the k of one P V MMA
constexpr int kDecRows = kDecWarps * kDecBlk;      // (key, head) pairs per stage
constexpr int kDecStages = 3;        // stages in flight: the one in use and two more
constexpr int kDecVpt = 4;           // virtual keys per MMA thread in a mapping pass
constexpr int kDecSC = kDecVpt * kDecWarps * 32;   // virtual keys per mapping pass
constexpr int kDecMaxSplits = 256;   // splits per (batch, kv head), at most one per merge thread
constexpr int kDecMaxGqa = 8;        // query heads per kv head: rows 0..7 of the MMA tile
constexpr int kDecMaxTopk = 8;
constexpr int kDecMaxK = 1024;       // groups: the new token's groups as a bit set in shared memory
constexpr int kErrCapacity = 6;     // FOCUS_ERR_CAPACITY

// kv heads per CTA: the largest of 8, 4, 2, 1 dividing Hkv
__host__ __device__ inline int decode_hg(int Hkv)
{
    return Hkv % 8 == 0 ? 8 : Hkv % 4 == 0 ? 4 : Hkv % 2 == 0 ? 2 : 1;
}

__global__ void __launch_bounds__(256) decode_lists_init_kernel(
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ pos, int n, int K, int topk,
    int cap, int32_t *__restrict__ glen, int32_t *__restrict__ gpos, int *status)
{
    grid_dep_sync();
    const int bg = blockIdx.x;                 // b * K + g
    const int b = bg / K, g = bg - b * K;
    const int32_t *off = offsets + (int64_t)b * (K + 1);
    const int o0 = off[g], len = off[g + 1] - o0;
    const int keep = min(len, cap);
    const int32_t *src = pos + (int64_t)b * n * topk + o0;
    int32_t *dst = gpos + (int64_t)bg * cap;
    for (int r = threadIdx.x; r < keep; r += blockDim.x) dst[r] = src[r];
    if (threadIdx.x == 0) {
        glen[bg] = keep;
        if (len > cap) atomicExch(status, kErrCapacity);
    }
}

// The new token i = L - 1 of sequence b joins the lists of its k groups (in
// the order of its ids, so that a repeated id is appended twice, never raced).
__device__ __forceinline__ void decode_append(const int32_t *__restrict__ ids, int b, int Lmax, int L, int K,
                              int topk, int cap, int32_t *__restrict__ glen,
                              int32_t *__restrict__ gpos, int *status)
{
    for (int s = 0; s < topk; ++s) {
        const int g = ids[((int64_t)b * Lmax + (L - 1)) * topk + s];
        if ((unsigned)g >= (unsigned)K) continue;   // an id outside [0, K) joins no list
        const int idx = glen[b * K + g];
        if (idx < cap) {
            gpos[((int64_t)b * K + g) * cap + idx] = L - 1;
            glen[b * K + g] = idx + 1;
        } else {
            atomicExch(status, kErrCapacity);
        }
    }
}

struct DecArgs {
    const __nv_bfloat16 *q;    // [B, Hq, D]
    const __nv_bfloat16 *k;    // [B, Lmax, Hkv, D]
    const __nv_bfloat16 *v;
    const int32_t *ids;        // [B, Lmax, topk]
    const int32_t *glen;       // [B, K]
    const int32_t *gpos;       // [B, K, cap]
    int B, L, Lmax, Hq, Hkv, K, topk, cap, window, P, HG;
    float scale_log2;
    float *opart;              // [B, Hkv, P, gqa, D] unnormalised O of each split
    float2 *mpart;             // [B, Hkv, P, gqa]: {running max (base 2), sum}
    WaitCtl wc;                // wait limit and device status word (a wait that ran out)
};

// Shared memory of a decode CTA for head size D: kDecStages stages, each the
// K rows then the V rows of KS = kDecRows / HG keys (a key's row holds its HG
// heads, HG * D * 2 bytes, plus 16 bytes so that the eight row addresses of
// an ldmatrix, same head and unit of eight consecutive keys, fall in eight
// different bank groups), then the positions of a pass's kept keys.  The
// largest stage is that of HG = 1.  After the key loop the stages hold the
// warps' partial outputs for the CTA merge.
template <int D>
struct DecSmem {
    static constexpr int kStage = 2 * kDecRows * (D * 2 + 16);
    static constexpr int kPos = kDecStages * kStage;            // int [kDecSC]
    static constexpr int kBytes = kPos + kDecSC * 4;
    static_assert(kDecWarps * kDecMaxGqa * (D + 4) * 4 <= kPos, "partial outputs fit the stages");
};

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}

// Rows 0..7 of c += A B for one m16n8k16 bf16 tile with fp32 accumulation.
// Rows 8..15 of A are zero here (the query heads of a kv head fill rows
// 0..7), so only a0 and a2 are passed and the tile's rows 8..15 (c2, c3) are
// dropped: each lane keeps c0 and c1 (row lane / 4, columns 2 (lane % 4) + 0, 1).
__device__ __forceinline__ void mma_16816(float &c0, float &c1, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1)
{
    float d2, d3;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %12};"
        : "=f"(c0), "=f"(c1), "=f"(d2), "=f"(d3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(0.f));
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1) decode_attn_kernel(const DecArgs a)
{
    using L = DecSmem<D>;
    constexpr int kUnits = D / 8;    // 16-byte units per head row = n-tiles of P V
    constexpr int kSteps = D / 16;   // k-steps of Q K^T = n-tile pairs of P V
    extern __shared__ __align__(128) uint8_t dsm[];
    int *spos = reinterpret_cast<int *>(dsm + L::kPos);
    __shared__ int gi[kDecMaxTopk];
    __shared__ int seg[kDecMaxTopk + 1];   // virtual-key bounds: window, then each list
    __shared__ int wcnt[kDecVpt * kDecWarps];
    __shared__ float wm[kDecWarps][kDecMaxGqa], wl[kDecWarps][kDecMaxGqa];
    __shared__ __align__(8) uint64_t full[kDecStages], empty[kDecStages];
    __shared__ int abort_flag;
    __shared__ uint32_t gmask[kDecMaxK / 32];   // the new token's groups

    const int p = blockIdx.x, hgrp = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool copier = warp == kDecWarps;
    const int HG = a.HG;
    const int KS = kDecRows / HG;                 // keys per stage
    const int rowB = HG * D * 2 + 16;             // bytes per key row of a stage
    const int hw = warp % HG, sb = warp / HG;     // an MMA warp's head in the group, key block
    const int gqa = a.Hq / a.Hkv;
    const int i = a.L - 1;
    const int topk = a.topk;
    const int qh = lane >> 2;        // this lane's query head: its row of A and of C

    // Q as MMA A fragments (bf16, row = query head, k = head dim); the inputs
    // of this step are ready, only the lists wait for the previous kernel
    uint32_t qa[kSteps][2];
    {
        const bool live = !copier && qh < gqa;
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(
            a.q + ((int64_t)b * a.Hq + (hgrp * HG + hw) * gqa + (live ? qh : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            qa[kk][0] = live ? qr[kk * 8 + (lane & 3)] : 0u;
            qa[kk][1] = live ? qr[kk * 8 + 4 + (lane & 3)] : 0u;
        }
    }
    if (tid < topk) gi[tid] = a.ids[((int64_t)b * a.Lmax + i) * topk + tid];
    if (tid < kDecStages) {
        mbar_init(&full[tid], 1);
        mbar_init(&empty[tid], kDecWarps);
    }
    if (tid == 0) abort_flag = 0;
    for (int x = tid; x < kDecMaxK / 32; x += kDecThreads) gmask[x] = 0u;
    mbar_fence_init();
    grid_dep_sync();
    __syncthreads();
    if (tid < topk) {
        const int g = gi[tid];
        const bool valid = (unsigned)g < (unsigned)a.K;
        const int len = valid ? a.glen[b * a.K + g] : 0;
        wcnt[tid] = min(max(len, 0), a.cap);
        if (valid) atomicOr(&gmask[g >> 5], 1u << (g & 31));
    }
    __syncthreads();
    int gmin = 0x7fffffff;           // the token's lowest group owns every pair in its list
    for (int s = 0; s < topk; ++s)
        if ((unsigned)gi[s] < (unsigned)a.K) gmin = min(gmin, gi[s]);
    if (tid == 0) {
        // the lists do not hold the new token yet (it is appended after the
        // attention), so its own key is taken as a window key: allowed
        // through the window, or at window 0 through its own groups
        seg[0] = min(max(a.window, gmin < a.K ? 1 : 0), i + 1);
        for (int s = 0; s < topk; ++s) seg[s + 1] = seg[s] + wcnt[s];
    }
    __syncthreads();
    const int nvirt = seg[topk];
    const int nw = seg[0];

    float mrun = -CUDART_INF_F, lrun = 0.f;   // this warp's running max (base 2) and sum
    float o[kUnits][2];                       // O tiles: rows = query heads, n = dims
#pragma unroll
    for (int nt = 0; nt < kUnits; ++nt) o[nt][0] = o[nt][1] = 0.f;
    uint32_t kg = 0;                          // stages of this CTA so far
    uint32_t armed = 0;                       // stages the copy warp has started

    // split p takes the virtual keys [lo, hi), kDecSC per pass
    const int per = (nvirt + a.P - 1) / a.P;
    const int lo = min(nvirt, p * per), hi = min(nvirt, lo + per);
    for (int vs = lo; vs < hi; vs += kDecSC) {
        // ---- positions of the pass's virtual keys, kDecVpt per MMA thread,
        // all loads of a phase in flight together
        int jj[kDecVpt], gs[kDecVpt];
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            const int vk = vs + r * (kDecWarps * 32) + tid;
            jj[r] = -1;
            gs[r] = -1;
            if (!copier && vk < hi) {
                if (vk < nw) {
                    jj[r] = i - vk;
                } else {
                    int sl = 0;
                    while (sl + 1 < topk && vk >= seg[sl + 1]) ++sl;
                    gs[r] = gi[sl];
                    jj[r] = a.gpos[((int64_t)b * a.K + gs[r]) * a.cap + (vk - seg[sl])];
                }
            }
        }
        // a list key counts if it lies before the window and the list's
        // group g is the lowest group it shares with the new token: g is
        // among its groups and none of its groups below g is the token's
        // (the lowest of the token's groups needs no look).  The group ids
        // of all of a thread's keys are loaded before any is used.
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            if (gs[r] >= 0 && !((unsigned)jj[r] < (unsigned)i && i - jj[r] >= a.window)) jj[r] = -1;
        }
        int gx[kDecVpt][kDecMaxTopk];
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            const bool look = gs[r] >= 0 && jj[r] >= 0 && gs[r] != gmin;
            const int32_t *gj = a.ids + ((int64_t)b * a.Lmax + (look ? jj[r] : i)) * topk;
#pragma unroll
            for (int x = 0; x < kDecMaxTopk; ++x) gx[r][x] = (look && x < topk) ? gj[x] : -1;
        }
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            if (gs[r] >= 0 && jj[r] >= 0 && gs[r] != gmin) {
                const int g = gs[r];
                bool found = false, lower = false;
#pragma unroll
                for (int x = 0; x < kDecMaxTopk; ++x) {
                    const int v = gx[r][x];
                    found = found || v == g;
                    if ((unsigned)v < (unsigned)g)
                        lower = lower || ((gmask[v >> 5] >> (v & 31)) & 1u);
                }
                if (!found || lower) jj[r] = -1;
            }
        }
        // ---- compact the kept keys into spos, in virtual-key order
        unsigned bal[kDecVpt];
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            bal[r] = __ballot_sync(0xffffffffu, jj[r] >= 0);
            if (lane == 0 && !copier) wcnt[r * kDecWarps + warp] = __popc(bal[r]);
        }
        __syncthreads();
        int run = 0, basev[kDecVpt];
#pragma unroll
        for (int e = 0; e < kDecVpt * kDecWarps; ++e) {
            if ((e % kDecWarps) == warp) basev[e / kDecWarps] = run;
            run += wcnt[e];
        }
        const int nv = run;
        const unsigned below = (1u << lane) - 1u;
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r)
            if (jj[r] >= 0) spos[basev[r] + __popc(bal[r] & below)] = jj[r];
        __syncthreads();

        // ---- stages of KS kept keys
        const int nst = (nv + KS - 1) / KS;
        if (copier) {
            // one bulk copy per (key, tensor): the key's rows of the group's
            // HG heads; keys past the last kept one repeat the stage's first
            // (their scores are masked)
            for (int k = 0; k < nst; ++k, ++kg) {
                const int st = kg % kDecStages;
                if (kg >= kDecStages &&
                    !mbar_wait(&empty[st], ((kg / kDecStages) - 1) & 1, &abort_flag, a.wc))
                    break;
                if (lane == 0) mbar_arrive_expect_tx(&full[st], 2 * KS * HG * D * 2);
                __syncwarp();
                uint8_t *sbase = dsm + st * L::kStage;
                for (int c = lane; c < 2 * KS; c += 32) {
                    const int which = c >= KS, u = c - which * KS;
                    const int idx = k * KS + u;
                    const int j = spos[idx < nv ? idx : k * KS];
                    const int64_t row = ((int64_t)b * a.Lmax + j) * a.Hkv + hgrp * HG;
                    bulk_load(sbase + (which * KS + u) * rowB, (which ? a.v : a.k) + row * D,
                              HG * D * 2, &full[st]);
                }
                ++armed;
            }
        } else {
            for (int k = 0; k < nst; ++k, ++kg) {
                const int st = kg % kDecStages;
                if (!mbar_wait(&full[st], (kg / kDecStages) & 1, &abort_flag, a.wc)) break;
                const int k0 = k * KS + sb * kDecBlk;   // this warp's first key of the stage
                const int cnt = min(kDecBlk, nv - k0);
                if (cnt > 0) {
                    const uint8_t *kb = dsm + st * L::kStage + (sb * kDecBlk) * rowB + hw * D * 2;
                    const uint8_t *vb = kb + KS * rowB;
                    // S = Q K^T for 16 keys (two n-tiles of 8), two chains per tile
                    float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
                    float e0[2] = {0.f, 0.f}, e1[2] = {0.f, 0.f};
                    {
                        const int ku = ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
                        for (int kk = 0; kk < kSteps; ++kk) {
                            const int x = 2 * kk + ((lane >> 3) & 1);
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4(kb + ku * rowB + (x << 4), r0, r1, r2, r3);
                            if (kk & 1) {
                                mma_16816(e0[0], e0[1], qa[kk][0], qa[kk][1], r0, r1);
                                mma_16816(e1[0], e1[1], qa[kk][0], qa[kk][1], r2, r3);
                            } else {
                                mma_16816(s0[0], s0[1], qa[kk][0], qa[kk][1], r0, r1);
                                mma_16816(s1[0], s1[1], qa[kk][0], qa[kk][1], r2, r3);
                            }
                        }
                    }
                    // online softmax for head qh over keys 2c, 2c + 1, 8 + 2c, 9 + 2c
                    const int c2 = 2 * (lane & 3);
                    const float sc = a.scale_log2;
                    const float t0 = c2 < cnt ? (s0[0] + e0[0]) * sc : -CUDART_INF_F;
                    const float t1 = c2 + 1 < cnt ? (s0[1] + e0[1]) * sc : -CUDART_INF_F;
                    const float t2 = c2 + 8 < cnt ? (s1[0] + e1[0]) * sc : -CUDART_INF_F;
                    const float t3 = c2 + 9 < cnt ? (s1[1] + e1[1]) * sc : -CUDART_INF_F;
                    float mx = fmaxf(fmaxf(t0, t1), fmaxf(t2, t3));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float mnew = fmaxf(mrun, mx);       // finite: key 0 of a block is kept
                    const float alpha = exp2f(mrun - mnew);   // 0 on the first block
                    const float p0 = exp2f(t0 - mnew), p1 = exp2f(t1 - mnew);
                    const float p2 = exp2f(t2 - mnew), p3 = exp2f(t3 - mnew);
                    lrun = lrun * alpha + ((p0 + p1) + (p2 + p3));
                    mrun = mnew;
#pragma unroll
                    for (int nt = 0; nt < kUnits; ++nt) {
                        o[nt][0] *= alpha;
                        o[nt][1] *= alpha;
                    }
                    // O += P V (P as the A fragment straight from the S tiles)
                    const uint32_t pa0 = pack_bf16x2(p0, p1), pa2 = pack_bf16x2(p2, p3);
                    const int vu = (((lane >> 3) & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int jp = 0; jp < kSteps; ++jp) {
                        const int x = 2 * jp + (lane >> 4);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_t(vb + vu * rowB + (x << 4), r0, r1, r2, r3);
                        mma_16816(o[2 * jp][0], o[2 * jp][1], pa0, pa2, r0, r1);
                        mma_16816(o[2 * jp + 1][0], o[2 * jp + 1][1], pa0, pa2, r2, r3);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);   // this warp is done with the stage
            }
        }
        __syncthreads();    // spos and wcnt are rewritten by the next pass
        if (abort_flag) break;
    }
    if (abort_flag) {
        // a wait ran out: the copy warp lets its copies still in flight land,
        // then the CTA leaves without a result (the status word holds the timeout)
        if (copier) {
            const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
            for (uint32_t u = armed > kDecStages ? armed - kDecStages : 0; u < armed; ++u)
                mbar_wait_until(&full[u % kDecStages], (u / kDecStages) & 1, deadline);
        }
        return;
    }

    // ---- merge the warps of each head, then write this split's unnormalised
    // result for the group's HG kv heads
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 1);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 2);
    if (!copier && (lane & 3) == 0 && qh < gqa) {
        wm[warp][qh] = mrun;
        wl[warp][qh] = lrun;
    }
    __syncthreads();
    // [warp][query head][D + 4]: the padding puts the eight query heads' rows
    // of a float2 store in different bank groups
    constexpr int kRowF = D + 4;
    float *ob = reinterpret_cast<float *>(dsm);
    if (!copier && qh < gqa) {
        float M = -CUDART_INF_F;
        for (int w = hw; w < kDecWarps; w += HG) M = fmaxf(M, wm[w][qh]);
        const float wt = mrun == -CUDART_INF_F ? 0.f : exp2f(mrun - M);
        float *orow = ob + (warp * kDecMaxGqa + qh) * kRowF + 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < kUnits; ++nt)
            *reinterpret_cast<float2 *>(orow + nt * 8) = make_float2(o[nt][0] * wt, o[nt][1] * wt);
    }
    __syncthreads();
    const int64_t hbase = (int64_t)b * a.Hkv + hgrp * HG;   // first kv head of the group
    {
        // rows r = (head hh, query head qq) of the group, a float4 per thread
        constexpr int kV = D / 4;
        constexpr int kRowsPer = kDecThreads / kV;
        const int c4 = tid % kV;
        for (int r = tid / kV; r < HG * gqa; r += kRowsPer) {
            const int hh = r / gqa, qq = r - hh * gqa;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = hh; w < kDecWarps; w += HG) {
                const float4 v = *reinterpret_cast<const float4 *>(
                    ob + (w * kDecMaxGqa + qq) * kRowF + 4 * c4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4 *>(a.opart + (((hbase + hh) * a.P + p) * gqa + qq) * D +
                                        4 * c4) = acc;
        }
    }
    if (tid < HG * gqa) {
        const int hh = tid / gqa, qq = tid - hh * gqa;
        float M = -CUDART_INF_F, Ls = 0.f;
        for (int w = hh; w < kDecWarps; w += HG) M = fmaxf(M, wm[w][qq]);
        for (int w = hh; w < kDecWarps; w += HG)
            if (wm[w][qq] != -CUDART_INF_F) Ls += wl[w][qq] * exp2f(wm[w][qq] - M);
        a.mpart[((hbase + hh) * a.P + p) * gqa + qq] = make_float2(M, Ls);
    }
}

// O = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p for every query head.
// Block (query head, 32 columns): warp g takes splits g, g + 8, ... of its
// 32 columns, all of them in flight before the weights are known; the
// splits' {max, sum} are read one per thread.  After the attention has read
// the lists, the grid's last block appends the new tokens to them.
struct DecAppend {
    const int32_t *ids;
    int B, Lmax, L, K, topk, cap;
    int32_t *glen, *gpos;
    int *status;
};

constexpr int kMrgCols = 32;                       // columns per merge block
constexpr int kMrgWarps = 8;
constexpr int kMrgThreads = kMrgWarps * 32;
static_assert(kMrgThreads >= kDecMaxSplits, "one merge thread per split for the weights");

template <int D>
__global__ void __launch_bounds__(kMrgThreads) decode_merge_kernel(const float *__restrict__ opart,
                                                                   const float2 *__restrict__ mpart,
                                                                   int Hq, int Hkv, int P,
                                                                   __nv_bfloat16 *__restrict__ O,
                                                                   float *__restrict__ lse,
                                                                   const DecAppend ap)
{
    constexpr int kPer = kDecMaxSplits / kMrgWarps;   // splits per thread, at most
    constexpr int kChunks = D / kMrgCols;
    grid_dep_sync();
    __shared__ float wgt[kDecMaxSplits];
    __shared__ float red[kMrgWarps], part[kMrgWarps][kMrgCols];
    __shared__ float Msh, Lsh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == gridDim.x - 1) {       // the last block appends
        for (int bb = tid; bb < ap.B; bb += blockDim.x)
            decode_append(ap.ids, bb, ap.Lmax, ap.L, ap.K, ap.topk, ap.cap, ap.glen, ap.gpos,
                          ap.status);
        return;
    }
    const int bh = blockIdx.x / kChunks;     // b * Hq + hq
    const int col = (blockIdx.x - bh * kChunks) * kMrgCols + lane;
    const int b = bh / Hq, hq = bh - b * Hq;
    const int gqa = Hq / Hkv, h = hq / gqa, q = hq - h * gqa;
    const int64_t base = ((int64_t)b * Hkv + h) * P;
    float ov[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pp = warp + kMrgWarps * k;
        ov[k] = pp < P ? opart[((base + pp) * gqa + q) * D + col] : 0.f;
    }
    float2 ml = make_float2(-CUDART_INF_F, 0.f);
    if (tid < P) ml = mpart[(base + tid) * gqa + q];
    float mx = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float M = -CUDART_INF_F;
        for (int w = 0; w < kMrgWarps; ++w) M = fmaxf(M, red[w]);
        Msh = M;
    }
    __syncthreads();
    const float M = Msh;
    const float wv = (tid < P && ml.x != -CUDART_INF_F) ? exp2f(ml.x - M) : 0.f;
    if (tid < P) wgt[tid] = wv;
    float ls = wv * ml.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    __syncthreads();
    if (lane == 0) red[warp] = ls;
    __syncthreads();
    if (tid == 0) {
        float Lt = 0.f;
        for (int w = 0; w < kMrgWarps; ++w) Lt += red[w];
        Lsh = Lt;
    }
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pp = warp + kMrgWarps * k;
        if (pp < P) acc += wgt[pp] * ov[k];
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (tid < kMrgCols) {
        const float lsum = Lsh;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kMrgWarps; ++w) tot += part[w][tid];
        O[(int64_t)bh * D + col] = __float2bfloat16_rn(lsum > 0.f ? tot / lsum : 0.f);
        if (lse && col == 0)
            lse[bh] = lsum > 0.f ? (M + log2f(lsum)) * 0.69314718055994531f : -CUDART_INF_F;
    }
}

}  // namespace

int decode_splits(int B, int Hkv)
{
    // about one CTA per SM of 152 over all (batch, kv-head group) pairs
    const int ctas = B * (Hkv / decode_hg(Hkv));
    const int want = (152 + ctas - 1) / ctas;
    return want < 1 ? 1 : (want > kDecMaxSplits ? kDecMaxSplits : want);
}

size_t decode_ws_bytes(int B, int Hq, int Hkv, int d)
{
    const int P = decode_splits(B, Hkv);
    const size_t rows = (size_t)B * Hkv * P * (Hq / Hkv);
    return ((rows * d * 4 + 255) & ~(size_t)255) + rows * 8 + 256;
}

cudaError_t launch_decode_lists_init(const int32_t *offsets, const int32_t *pos, int B, int n,
                                     int K, int topk, int cap, int32_t *glen, int32_t *gpos,
                                     int *status, cudaStream_t s, int *launches)
{
    prof_begin("decode_lists_init", s);
    const cudaError_t e = launch_pdl(decode_lists_init_kernel, dim3((unsigned)(B * K)), dim3(256),
                                     0, s, offsets, pos, n, K, topk, cap, glen, gpos, status);
    prof_end(s);
    *launches += 1;
    return e;
}

cudaError_t launch_decode(const DecodeLaunch &p, cudaStream_t s, int *launches)
{
    cudaError_t e;
    const int P = decode_splits(p.B, p.Hkv);
    const int HG = decode_hg(p.Hkv);
    const size_t rows = (size_t)p.B * p.Hkv * P * (p.Hq / p.Hkv);
    uint8_t *ws = static_cast<uint8_t *>(p.ws);
    DecArgs a;
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.ids = p.ids;
    a.glen = p.glen;
    a.gpos = p.gpos;
    a.B = p.B;
    a.L = p.L;
    a.Lmax = p.Lmax;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.K = p.K;
    a.topk = p.topk;
    a.cap = p.cap;
    a.window = p.window;
    a.P = P;
    a.HG = HG;
    a.scale_log2 = p.scale_log2;
    a.opart = reinterpret_cast<float *>(ws);
    a.mpart = reinterpret_cast<float2 *>(ws + ((rows * p.d * 4 + 255) & ~(size_t)255));
    a.wc = p.wc;
    const dim3 grid((unsigned)P, (unsigned)(p.Hkv / HG), (unsigned)p.B);
    prof_begin("decode_attn", s);
    if (p.d == 64)
        e = launch_pdl(decode_attn_kernel<64>, grid, dim3(kDecThreads), DecSmem<64>::kBytes, s, a);
    else
        e = launch_pdl(decode_attn_kernel<128>, grid, dim3(kDecThreads), DecSmem<128>::kBytes, s,
                       a);
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    DecAppend ap;
    ap.ids = p.ids;
    ap.B = p.B;
    ap.Lmax = p.Lmax;
    ap.L = p.L;
    ap.K = p.K;
    ap.topk = p.topk;
    ap.cap = p.cap;
    ap.glen = p.glen;
    ap.gpos = p.gpos;
    ap.status = p.status;
    prof_begin("decode_merge", s);
    const unsigned mblocks = (unsigned)(p.B * p.Hq * (p.d / kMrgCols) + 1);   // + the append
    if (p.d == 64)
        e = launch_pdl(decode_merge_kernel<64>, dim3(mblocks), dim3(kMrgThreads), 0, s, a.opart,
                       a.mpart, p.Hq, p.Hkv, P, p.O, p.lse, ap);
    else
        e = launch_pdl(decode_merge_kernel<128>, dim3(mblocks), dim3(kMrgThreads), 0, s, a.opart,
                       a.mpart, p.Hq, p.Hkv, P, p.O, p.lse, ap);
    prof_end(s);
    *launches += 1;
    return e;
}

size_t decode_smem_bytes(int d) { return d == 64 ? DecSmem<64>::kBytes : DecSmem<128>::kBytes; }

cudaError_t decode_preflight(int d)
{
    if (d == 64)
        return cudaFuncSetAttribute(decode_attn_kernel<64>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    DecSmem<64>::kBytes);
    return cudaFuncSetAttribute(decode_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DecSmem<128>::kBytes);
}

}  // namespace focus
