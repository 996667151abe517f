// Decode: one new token per sequence against a key/value cache whose group
// memberships are kept as per-group position lists (Focus, gist.science/zh
// technical summary 2.1.3 and gist.science/nl Kerncomponent 4: at inference a
// token belongs to its k highest-scoring groups and attends, with an exact
// softmax, to the keys in its local window or sharing one of its groups).
//
// Group lists: glen[b][g] entries of gpos[b][g][0..cap), token positions in
// ascending order.  decode_lists_init copies a prefill's bucketing
// (offsets, pos) into that layout; decode_append puts the new token at the
// end of its k lists (positions only grow, so the order holds).
//
// Attention of the new token i = L - 1 over its allowed set, split without
// overlap into
//   window keys  j in [i - w + 1, i]                    (every one allowed), and
//   group keys   j in the list of g, i - j >= w, with g = min(G_i n G_j)
//                (a pair sharing several groups is taken from the lowest).
// The keys form one virtual sequence: the window, then the k lists.
// decode_attn_kernel: CTA (p, kv head, batch) takes chunks p, p + P, ... of
// 64 virtual keys, maps them to positions, drops the group keys that are not
// its own (window or a lower shared group), copies the K and V rows of the
// rest into shared memory (16-byte asynchronous copies), and runs an online
// softmax for the query heads of the kv head in fp32.  decode_merge_kernel
// combines the P partial results per query head.  HBM-bound: the K and V rows
// of the allowed keys are the bytes that matter.
#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "focus_internal.h"
#include "focus_ptx.cuh"

namespace focus {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecCtasPerSm = 2;     // resident decode CTAs per SM (registers)
constexpr int kDecBlk = 16;          // kept keys per warp block: the k of one P V MMA
constexpr int kDecStages = 3;        // blocks of a warp in flight: the current and two more
constexpr int kDecVpt = 4;           // virtual keys per thread in a mapping pass
constexpr int kDecSC = kDecVpt * kDecThreads;   // virtual keys per mapping pass
constexpr int kDecMaxSplits = 128;   // splits per (batch, kv head), at most one per merge thread
constexpr int kDecMaxGqa = 8;        // query heads per kv head: rows 0..7 of the MMA tile
constexpr int kDecMaxTopk = 8;
constexpr int kDecMaxK = 1024;       // groups: the new token's groups as a bit set in shared memory
constexpr int kErrCapacity = 6;     // FOCUS_ERR_CAPACITY

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
    int B, L, Lmax, Hq, Hkv, K, topk, cap, window, P;
    float scale_log2;
    float *opart;              // [B, Hkv, P, gqa, D] unnormalised O of each CTA
    float2 *mpart;             // [B, Hkv, P, gqa]: {running max (base 2), sum}
    int *status;               // device status word (a wait that ran out)
};

// Shared memory of a decode CTA for head size D: per warp, kDecStages stages
// of the K rows and the V rows of a block of kDecBlk kept keys, then the
// positions of a pass's kept keys.  A row takes 16 bytes more than it holds,
// so that the eight row addresses of an ldmatrix (same 16-byte unit, eight
// consecutive rows) fall in eight different bank groups.  After the key loop
// the stages hold the warps' partial outputs for the CTA merge.
template <int D>
struct DecSmem {
    static constexpr int kRow = D * 2 + 16;                     // bytes per cached row
    static constexpr int kBlk = kDecBlk * kRow;                 // K (or V) rows of a block
    static constexpr int kWarp = kDecStages * 2 * kBlk;         // stages of K and V
    static constexpr int kPos = kDecWarps * kWarp;              // int [kDecSC]
    static constexpr int kBytes = kPos + kDecSC * 4;
    static_assert(kDecWarps * kDecMaxGqa * D * 4 <= kPos, "partial outputs fit the stages");
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
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm) decode_attn_kernel(const DecArgs a)
{
    using L = DecSmem<D>;
    constexpr int kUnits = D / 8;    // 16-byte units per row = n-tiles of P V
    constexpr int kSteps = D / 16;   // k-steps of Q K^T = n-tile pairs of P V
    extern __shared__ __align__(128) uint8_t dsm[];
    int *spos = reinterpret_cast<int *>(dsm + L::kPos);
    __shared__ int gi[kDecMaxTopk];
    __shared__ int seg[kDecMaxTopk + 1];   // virtual-key bounds: window, then each list
    __shared__ int wcnt[kDecVpt * kDecWarps];
    __shared__ float wm[kDecWarps][kDecMaxGqa], wl[kDecWarps][kDecMaxGqa];
    __shared__ __align__(8) uint64_t bars[kDecWarps][kDecStages];   // one per warp stage
    __shared__ int abort_flag;
    __shared__ uint32_t gmask[kDecMaxK / 32];   // the new token's groups

    const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gqa = a.Hq / a.Hkv;
    const int i = a.L - 1;
    const int topk = a.topk;
    const int qh = lane >> 2;        // this lane's query head: its row of A and of C

    // Q as MMA A fragments (bf16, row = query head, k = head dim); the inputs
    // of this step are ready, only the lists wait for the previous kernel
    uint32_t qa[kSteps][2];
    {
        const bool live = qh < gqa;
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(
            a.q + ((int64_t)b * a.Hq + h * gqa + (live ? qh : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            qa[kk][0] = live ? qr[kk * 8 + (lane & 3)] : 0u;
            qa[kk][1] = live ? qr[kk * 8 + 4 + (lane & 3)] : 0u;
        }
    }
    if (tid < topk) gi[tid] = a.ids[((int64_t)b * a.Lmax + i) * topk + tid];
    if (tid < kDecWarps * kDecStages) mbar_init(&bars[tid / kDecStages][tid % kDecStages], 1);
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
    uint8_t *wbuf = dsm + warp * L::kWarp;
    uint32_t issued = 0, used = 0;   // blocks this warp has issued / consumed (stage = n % 3)

    // K and V rows of kept keys [16 t, 16 t + 16) into the next stage: one
    // bulk copy per lane (lanes 0..15 the K rows, 16..31 the V rows).  Rows
    // past the last kept key repeat the block's first key; their scores are
    // masked.
    auto issue = [&](int t, int nv) {
        const int st = issued % kDecStages;
        uint64_t *bar = &bars[warp][st];
        if (lane == 0) mbar_arrive_expect_tx(bar, 2 * kDecBlk * D * 2);
        __syncwarp();
        const int u = lane & (kDecBlk - 1);
        const int idx = t * kDecBlk + u;
        const int j = spos[idx < nv ? idx : t * kDecBlk];
        const int64_t row = ((int64_t)b * a.Lmax + j) * a.Hkv + h;
        const __nv_bfloat16 *src = (lane < kDecBlk ? a.k : a.v) + row * D;
        uint8_t *dst = wbuf + st * 2 * L::kBlk + (lane < kDecBlk ? 0 : L::kBlk) + u * L::kRow;
        bulk_load(dst, src, D * 2, bar);
        ++issued;
    };

    // split p takes the virtual keys [lo, hi), kDecSC per pass
    const int per = (nvirt + a.P - 1) / a.P;
    const int lo = min(nvirt, p * per), hi = min(nvirt, lo + per);
    for (int vs = lo; vs < hi; vs += kDecSC) {
        // ---- positions of the pass's virtual keys, kDecVpt per thread, all
        // loads of a phase in flight together
        int jj[kDecVpt], gs[kDecVpt];
#pragma unroll
        for (int r = 0; r < kDecVpt; ++r) {
            const int vk = vs + r * kDecThreads + tid;
            jj[r] = -1;
            gs[r] = -1;
            if (vk < hi) {
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
            if (lane == 0) wcnt[r * kDecWarps + warp] = __popc(bal[r]);
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

        // ---- blocks of kDecBlk kept keys: warp w takes blocks w, w + 4, ...
        // with the copies of its next two blocks in flight during the current one
        const int nb = (nv + kDecBlk - 1) / kDecBlk;
        for (int t = warp, k = 0; t < nb && k < kDecStages - 1; t += kDecWarps, ++k) issue(t, nv);
        for (int t = warp; t < nb; t += kDecWarps) {
            const int ahead = (kDecStages - 1) * kDecWarps;
            if (t + ahead < nb) issue(t + ahead, nv);   // into the stage freed last
            const int st = used % kDecStages;
            if (!mbar_wait(&bars[warp][st], (used / kDecStages) & 1, &abort_flag, a.status))
                break;
            ++used;
            const uint8_t *kb = wbuf + st * 2 * L::kBlk;
            const uint8_t *vb = kb + L::kBlk;
            const int cnt = min(kDecBlk, nv - t * kDecBlk);
            // S = Q K^T for 16 keys (two n-tiles of 8)
            float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
            {
                const int ku = ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < kSteps; ++kk) {
                    const int x = 2 * kk + ((lane >> 3) & 1);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kb + ku * L::kRow + (x << 4), r0, r1, r2, r3);
                    mma_16816(s0[0], s0[1], qa[kk][0], qa[kk][1], r0, r1);
                    mma_16816(s1[0], s1[1], qa[kk][0], qa[kk][1], r2, r3);
                }
            }
            // online softmax for head qh over keys 2c, 2c + 1, 8 + 2c, 9 + 2c
            const int c2 = 2 * (lane & 3);
            const float t0 = c2 < cnt ? s0[0] * a.scale_log2 : -CUDART_INF_F;
            const float t1 = c2 + 1 < cnt ? s0[1] * a.scale_log2 : -CUDART_INF_F;
            const float t2 = c2 + 8 < cnt ? s1[0] * a.scale_log2 : -CUDART_INF_F;
            const float t3 = c2 + 9 < cnt ? s1[1] * a.scale_log2 : -CUDART_INF_F;
            float mx = fmaxf(fmaxf(t0, t1), fmaxf(t2, t3));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(mrun, mx);          // finite: key 0 of a block is kept
            const float alpha = exp2f(mrun - mnew);      // 0 on the first block
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
            {
                const int vu = (((lane >> 3) & 1) << 3) + (lane & 7);
#pragma unroll
                for (int jp = 0; jp < kSteps; ++jp) {
                    const int x = 2 * jp + (lane >> 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(vb + vu * L::kRow + (x << 4), r0, r1, r2, r3);
                    mma_16816(o[2 * jp][0], o[2 * jp][1], pa0, pa2, r0, r1);
                    mma_16816(o[2 * jp + 1][0], o[2 * jp + 1][1], pa0, pa2, r2, r3);
                }
            }
            __syncwarp();   // the stage is free for the copies issued next
        }
        __syncthreads();    // spos and wcnt are rewritten by the next pass
        if (abort_flag) break;
    }
    if (abort_flag) {
        // a wait ran out: let this warp's copies still in flight land, then
        // leave without a result (the status word holds the timeout)
        const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
        for (; used < issued; ++used)
            mbar_wait_until(&bars[warp][used % kDecStages], (used / kDecStages) & 1, deadline);
        return;
    }

    // ---- merge the four warps, then write this split's unnormalised result
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 1);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 2);
    if ((lane & 3) == 0 && qh < gqa) {
        wm[warp][qh] = mrun;
        wl[warp][qh] = lrun;
    }
    __syncthreads();
    float *ob = reinterpret_cast<float *>(dsm);   // [warp][head][D]
    if (qh < gqa) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w][qh]);
        const float wt = mrun == -CUDART_INF_F ? 0.f : exp2f(mrun - M);
        float *orow = ob + (warp * kDecMaxGqa + qh) * D + 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < kUnits; ++nt)
            *reinterpret_cast<float2 *>(orow + nt * 8) = make_float2(o[nt][0] * wt, o[nt][1] * wt);
    }
    __syncthreads();
    const int64_t base = (((int64_t)b * a.Hkv + h) * a.P + p) * gqa;
    for (int e = tid; e < gqa * D; e += kDecThreads) {
        const int hq = e / D, d = e - hq * D;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) acc += ob[(w * kDecMaxGqa + hq) * D + d];
        a.opart[(base + hq) * D + d] = acc;
    }
    if (tid < gqa) {
        float M = -CUDART_INF_F, Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w][tid]);
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w)
            if (wm[w][tid] != -CUDART_INF_F) Ls += wl[w][tid] * exp2f(wm[w][tid] - M);
        a.mpart[base + tid] = make_float2(M, Ls);
    }
}

// O = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p for every query head.
// Four groups of D threads take every fourth split; each thread has its
// column of all of its splits in flight before the weights are known.  After
// the attention has read the lists, block 0 appends the new tokens to them.
struct DecAppend {
    const int32_t *ids;
    int B, Lmax, L, K, topk, cap;
    int32_t *glen, *gpos;
    int *status;
};

template <int D>
__global__ void __launch_bounds__(4 * D, 1) decode_merge_kernel(const float *__restrict__ opart,
                                                             const float2 *__restrict__ mpart,
                                                             int Hq, int Hkv, int P,
                                                             __nv_bfloat16 *__restrict__ O,
                                                             float *__restrict__ lse,
                                                             const DecAppend ap)
{
    constexpr int kPer = kDecMaxSplits / 4;   // splits per thread group, at most
    grid_dep_sync();
    __shared__ float wgt[kDecMaxSplits];
    __shared__ float red[4 * D / 32], part[4][D];
    __shared__ float Msh, Lsh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == gridDim.x - 1) {       // the last block appends
        for (int bb = tid; bb < ap.B; bb += blockDim.x)
            decode_append(ap.ids, bb, ap.Lmax, ap.L, ap.K, ap.topk, ap.cap, ap.glen, ap.gpos,
                          ap.status);
        return;
    }
    const int bh = blockIdx.x;               // b * Hq + hq
    const int b = bh / Hq, hq = bh - b * Hq;
    const int gqa = Hq / Hkv, h = hq / gqa, q = hq - h * gqa;
    const int64_t base = ((int64_t)b * Hkv + h) * P;
    const int gq = tid / D, c = tid - gq * D;
    float ov[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pp = gq + 4 * k;
        ov[k] = pp < P ? opart[((base + pp) * gqa + q) * D + c] : 0.f;
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
        for (int w = 0; w < 4 * D / 32; ++w) M = fmaxf(M, red[w]);
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
        for (int w = 0; w < 4 * D / 32; ++w) Lt += red[w];
        Lsh = Lt;
    }
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pp = gq + 4 * k;
        if (pp < P) acc += wgt[pp] * ov[k];
    }
    part[gq][c] = acc;
    __syncthreads();
    if (tid < D) {
        const float lsum = Lsh;
        const float tot = part[0][tid] + part[1][tid] + part[2][tid] + part[3][tid];
        O[(int64_t)bh * D + tid] = __float2bfloat16_rn(lsum > 0.f ? tot / lsum : 0.f);
        if (lse && tid == 0)
            lse[bh] = lsum > 0.f ? (M + log2f(lsum)) * 0.69314718055994531f : -CUDART_INF_F;
    }
}

}  // namespace

int decode_splits(int B, int Hkv)
{
    // about kDecCtasPerSm CTAs per SM of 152 over all (batch, kv head) pairs
    const int want = (kDecCtasPerSm * 152 + B * Hkv - 1) / (B * Hkv);
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
    a.scale_log2 = p.scale_log2;
    a.opart = reinterpret_cast<float *>(ws);
    a.mpart = reinterpret_cast<float2 *>(ws + ((rows * p.d * 4 + 255) & ~(size_t)255));
    a.status = p.status;
    const dim3 grid((unsigned)P, (unsigned)p.Hkv, (unsigned)p.B);
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
    if (p.d == 64)
        e = launch_pdl(decode_merge_kernel<64>, dim3((unsigned)(p.B * p.Hq + 1)), dim3(256), 0, s,
                       a.opart, a.mpart, p.Hq, p.Hkv, P, p.O, p.lse, ap);
    else
        e = launch_pdl(decode_merge_kernel<128>, dim3((unsigned)(p.B * p.Hq + 1)), dim3(512), 0, s,
                       a.opart, a.mpart, p.Hq, p.Hkv, P, p.O, p.lse, ap);
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
