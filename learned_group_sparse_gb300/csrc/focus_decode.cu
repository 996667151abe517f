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

constexpr int kDecC = 64;           // kept keys per chunk of K/V rows
constexpr int kDecSC = 256;         // virtual keys per super-chunk (two per thread)
constexpr int kDecMaxSplits = 128;  // splits per (batch, kv head), at most one per merge thread
constexpr int kDecThreads = 128;
constexpr int kDecMaxGqa = 8;       // query heads per kv head
constexpr int kDecMaxTopk = 8;
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

// The new token i = L - 1 of every sequence joins the lists of its k groups.
__global__ void decode_append_kernel(const int32_t *__restrict__ ids, int B, int Lmax, int L,
                                     int K, int topk, int cap, int32_t *__restrict__ glen,
                                     int32_t *__restrict__ gpos, int *status)
{
    grid_dep_sync();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= B * topk) return;
    const int b = t / topk, s = t - b * topk;
    const int g = ids[((int64_t)b * Lmax + (L - 1)) * topk + s];
    if ((unsigned)g >= (unsigned)K) return;    // an id outside [0, K) joins no list
    const int idx = glen[b * K + g];
    if (idx < cap) {
        gpos[((int64_t)b * K + g) * cap + idx] = L - 1;
        glen[b * K + g] = idx + 1;
    } else {
        atomicExch(status, kErrCapacity);
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
};

// Shared memory of a decode CTA for head size D: two buffers of K and V rows
// for a chunk of kept keys (16 bytes of padding per row keep a thread's
// own-row loads free of bank conflicts), the queries in fp32, the chunk's
// scores, and the positions of a super-chunk's kept keys.
template <int D>
struct DecSmem {
    static constexpr int kRow = D * 2 + 16;                     // bytes per cached row
    static constexpr int kBuf = 2 * kDecC * kRow;               // K rows, then V rows
    static constexpr int kQ = 2 * kBuf;                         // float [gqa][D]
    static constexpr int kS = kQ + kDecMaxGqa * D * 4;          // float [gqa][kDecC]
    static constexpr int kPos = kS + kDecMaxGqa * kDecC * 4;    // int [kDecSC]
    static constexpr int kBytes = kPos + kDecSC * 4;
};

// The position of virtual key vk if this split scores it, else -1: window
// keys always; a key from the list of g if it lies before the window and g is
// the lowest group it shares with the new token.
__device__ __forceinline__ int decode_key(const DecArgs &a, int b, int i, int vk, int nw, int nvirt,
                                          const int *gi, const int *seg)
{
    if (vk < nw) return i - vk;
    if (vk >= nvirt) return -1;
    int s = 0;
    while (s + 1 < a.topk && vk >= seg[s + 1]) ++s;
    const int g = gi[s];
    const int jj = a.gpos[((int64_t)b * a.K + g) * a.cap + (vk - seg[s])];
    if ((unsigned)jj > (unsigned)i || i - jj < a.window) return -1;
    // the list of the new token's lowest group owns every shared key in it
    bool lowest = true;
    for (int y = 0; y < a.topk; ++y) lowest = lowest && gi[y] >= g;
    if (lowest) return jj;
    const int32_t *gj = a.ids + ((int64_t)b * a.Lmax + jj) * a.topk;
    int own = 0x7fffffff;
    for (int x = 0; x < a.topk; ++x) {
        const int gx = gj[x];
        for (int y = 0; y < a.topk; ++y)
            if (gi[y] == gx && gx < own) own = gx;
    }
    return own == g ? jj : -1;
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 3) decode_attn_kernel(const DecArgs a)
{
    grid_dep_sync();
    using L = DecSmem<D>;
    extern __shared__ __align__(16) uint8_t dsm[];
    float *qf = reinterpret_cast<float *>(dsm + L::kQ);
    float *S = reinterpret_cast<float *>(dsm + L::kS);
    int *spos = reinterpret_cast<int *>(dsm + L::kPos);
    __shared__ int gi[kDecMaxTopk];
    __shared__ int seg[kDecMaxTopk + 1];   // virtual-key bounds: window, then each list
    __shared__ float mrun[kDecMaxGqa], lrun[kDecMaxGqa], alpha[kDecMaxGqa];
    __shared__ int wcnt[2 * (kDecThreads / 32)];

    const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gqa = a.Hq / a.Hkv;
    const int i = a.L - 1;
    const int topk = a.topk;
    constexpr int kUnits = D / 8;   // 16-byte units per row

    if (tid < topk) gi[tid] = a.ids[((int64_t)b * a.Lmax + i) * topk + tid];
    if (tid < kDecMaxGqa) {
        mrun[tid] = -CUDART_INF_F;
        lrun[tid] = 0.f;
    }
    for (int e = tid; e < gqa * D; e += kDecThreads) {
        const int hq = h * gqa + e / D;
        qf[e] = __bfloat162float(a.q[((int64_t)b * a.Hq + hq) * D + (e % D)]) * a.scale_log2;
    }
    __syncthreads();
    if (tid == 0) {
        seg[0] = min(a.window, i + 1);
        for (int s = 0; s < topk; ++s) {
            const int g = gi[s];
            const int len = (unsigned)g < (unsigned)a.K ? a.glen[b * a.K + g] : 0;
            seg[s + 1] = seg[s] + min(max(len, 0), a.cap);
        }
    }
    __syncthreads();
    const int nvirt = seg[topk];
    const int nw = seg[0];

    float o[kDecMaxGqa];
#pragma unroll
    for (int q = 0; q < kDecMaxGqa; ++q) o[q] = 0.f;

    // K and V rows of kept keys [c0, c0 + cnt) into buffer bf (16-byte copies)
    auto issue = [&](int bf, int c0, int cnt) {
        uint8_t *kb = dsm + bf * L::kBuf;
        uint8_t *vb = kb + kDecC * L::kRow;
        for (int x = tid; x < cnt * kUnits; x += kDecThreads) {
            const int u = x / kUnits, q8 = x - u * kUnits;
            const int64_t row = ((int64_t)b * a.Lmax + spos[c0 + u]) * a.Hkv + h;
            cp_async16(kb + u * L::kRow + q8 * 16, a.k + row * D + q8 * 8, 16);
            cp_async16(vb + u * L::kRow + q8 * 16, a.v + row * D + q8 * 8, 16);
        }
        cp_async_commit();
    };

    for (int sc = p; sc * kDecSC < nvirt; sc += a.P) {
        // ---- the super-chunk's virtual keys (two per thread: both load
        // chains in flight), compacted into spos[0 .. nv)
        const int v0 = sc * kDecSC + tid;
        const int j0 = decode_key(a, b, i, v0, nw, nvirt, gi, seg);
        const int j1 = decode_key(a, b, i, v0 + kDecThreads, nw, nvirt, gi, seg);
        const unsigned b0 = __ballot_sync(0xffffffffu, j0 >= 0);
        const unsigned b1 = __ballot_sync(0xffffffffu, j1 >= 0);
        if (lane == 0) {
            wcnt[warp] = __popc(b0);
            wcnt[kDecThreads / 32 + warp] = __popc(b1);
        }
        __syncthreads();
        int before0 = 0, before1 = 0, nv = 0;
#pragma unroll
        for (int w = 0; w < 2 * (kDecThreads / 32); ++w) {
            if (w < warp) before0 += wcnt[w];
            if (w < kDecThreads / 32 + warp) before1 += wcnt[w];
            nv += wcnt[w];
        }
        const unsigned below = (1u << lane) - 1u;
        if (j0 >= 0) spos[before0 + __popc(b0 & below)] = j0;
        if (j1 >= 0) spos[before1 + __popc(b1 & below)] = j1;
        __syncthreads();
        // ---- chunks of kDecC kept keys, the next chunk's copies in flight
        const int nch = (nv + kDecC - 1) / kDecC;
        if (nch > 0) issue(0, 0, min(kDecC, nv));
        for (int k = 0; k < nch; ++k) {
            const int c0 = k * kDecC, cnt = min(kDecC, nv - c0);
            if (k + 1 < nch) {
                issue((k + 1) & 1, c0 + kDecC, min(kDecC, nv - c0 - kDecC));
                cp_async_wait_group1();
            } else {
                cp_async_wait_all();
            }
            __syncthreads();
            const uint8_t *kb = dsm + (k & 1) * L::kBuf;
            const uint8_t *vb = kb + kDecC * L::kRow;
            // scores of key u for every query head (base 2, scale folded into q)
            if (tid < cnt) {
                const uint4 *kr = reinterpret_cast<const uint4 *>(kb + tid * L::kRow);
                float acc[kDecMaxGqa];
#pragma unroll
                for (int q = 0; q < kDecMaxGqa; ++q) acc[q] = 0.f;
#pragma unroll 4
                for (int q8 = 0; q8 < kUnits; ++q8) {
                    const uint4 raw = kr[q8];
                    const __nv_bfloat162 *kp = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                    float kv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(kp[e]);
                        kv[2 * e] = f.x;
                        kv[2 * e + 1] = f.y;
                    }
#pragma unroll
                    for (int q = 0; q < kDecMaxGqa; ++q) {
                        if (q < gqa) {
                            const float4 qa =
                                *reinterpret_cast<const float4 *>(qf + q * D + q8 * 8);
                            const float4 qb =
                                *reinterpret_cast<const float4 *>(qf + q * D + q8 * 8 + 4);
                            acc[q] = fmaf(qa.x, kv[0], acc[q]);
                            acc[q] = fmaf(qa.y, kv[1], acc[q]);
                            acc[q] = fmaf(qa.z, kv[2], acc[q]);
                            acc[q] = fmaf(qa.w, kv[3], acc[q]);
                            acc[q] = fmaf(qb.x, kv[4], acc[q]);
                            acc[q] = fmaf(qb.y, kv[5], acc[q]);
                            acc[q] = fmaf(qb.z, kv[6], acc[q]);
                            acc[q] = fmaf(qb.w, kv[7], acc[q]);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < kDecMaxGqa; ++q)
                    if (q < gqa) S[q * kDecC + tid] = acc[q];
            }
            __syncthreads();
            // online softmax per query head: warp w takes heads w, w + 4, ...
            for (int q = warp; q < gqa; q += kDecThreads / 32) {
                float mx = -CUDART_INF_F;
                for (int u = lane; u < cnt; u += 32) mx = fmaxf(mx, S[q * kDecC + u]);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float mold = mrun[q];
                const float mnew = fmaxf(mold, mx);
                float sum = 0.f;
                for (int u = lane; u < cnt; u += 32) {
                    const float pr = exp2f(S[q * kDecC + u] - mnew);
                    S[q * kDecC + u] = pr;
                    sum += pr;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    sum += __shfl_xor_sync(0xffffffffu, sum, off);
                __syncwarp();
                if (lane == 0) {
                    const float al = (mold == -CUDART_INF_F) ? 0.f : exp2f(mold - mnew);
                    alpha[q] = al;
                    lrun[q] = lrun[q] * al + sum;
                    mrun[q] = mnew;
                }
            }
            __syncthreads();
            // O += P V: thread t owns column t of every head's output
            if (tid < D) {
                float acc[kDecMaxGqa];
#pragma unroll
                for (int q = 0; q < kDecMaxGqa; ++q) acc[q] = (q < gqa) ? o[q] * alpha[q] : 0.f;
                for (int u = 0; u < cnt; ++u) {
                    const float vv = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(vb + u * L::kRow + tid * 2));
#pragma unroll
                    for (int q = 0; q < kDecMaxGqa; ++q)
                        if (q < gqa) acc[q] = fmaf(S[q * kDecC + u], vv, acc[q]);
                }
#pragma unroll
                for (int q = 0; q < kDecMaxGqa; ++q) o[q] = acc[q];
            }
            __syncthreads();   // buffer k & 1 and the scores are free again
        }
    }
    // ---- this split's unnormalised result and its {max, sum}
    const int64_t base = (((int64_t)b * a.Hkv + h) * a.P + p) * gqa;
    if (tid < D) {
#pragma unroll
        for (int q = 0; q < kDecMaxGqa; ++q)
            if (q < gqa) a.opart[(base + q) * D + tid] = o[q];
    }
    if (tid < gqa) a.mpart[base + tid] = make_float2(mrun[tid], lrun[tid]);
}

// O = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p for every query head.
// The splits' {max, sum} are read in parallel; four groups of D threads then
// take a quarter of the splits' partial outputs each.
template <int D>
__global__ void __launch_bounds__(4 * D) decode_merge_kernel(const float *__restrict__ opart,
                                                             const float2 *__restrict__ mpart,
                                                             int Hq, int Hkv, int P,
                                                             __nv_bfloat16 *__restrict__ O,
                                                             float *__restrict__ lse)
{
    grid_dep_sync();
    __shared__ float wgt[kDecMaxSplits];
    __shared__ float red[4 * D / 32], part[4][D];
    __shared__ float Msh, Lsh;
    const int bh = blockIdx.x;               // b * Hq + hq
    const int b = bh / Hq, hq = bh - b * Hq;
    const int gqa = Hq / Hkv, h = hq / gqa, q = hq - h * gqa;
    const int64_t base = ((int64_t)b * Hkv + h) * P;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
    // partial outputs: group gq takes splits gq, gq + 4, ...; thread column c
    const int gq = tid / D, c = tid - gq * D;
    float acc = 0.f;
#pragma unroll 4
    for (int pp = gq; pp < P; pp += 4) {
        const float w = wgt[pp];
        if (w != 0.f) acc += w * opart[((base + pp) * gqa + q) * D + c];
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
    // about three CTAs per SM of 152 over all (batch, kv head) pairs
    const int want = (3 * 152 + B * Hkv - 1) / (B * Hkv);
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
    prof_begin("decode_append", s);
    e = launch_pdl(decode_append_kernel, dim3((unsigned)((p.B * p.topk + 127) / 128)), dim3(128),
                   0, s, p.ids, p.B, p.Lmax, p.L, p.K, p.topk, p.cap, p.glen, p.gpos, p.status);
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
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
    prof_begin("decode_merge", s);
    if (p.d == 64)
        e = launch_pdl(decode_merge_kernel<64>, dim3((unsigned)(p.B * p.Hq)), dim3(256), 0, s,
                       a.opart, a.mpart, p.Hq, p.Hkv, P, p.O, p.lse);
    else
        e = launch_pdl(decode_merge_kernel<128>, dim3((unsigned)(p.B * p.Hq)), dim3(512), 0, s,
                       a.opart, a.mpart, p.Hq, p.Hkv, P, p.O, p.lse);
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
