// Backward of soft-gated training attention on the 5th-generation tensor
// cores (Focus, gist.science/zh technical summary 2.1.2 "gated attention":
// s_ij = q_i . k_j * scale * gate_ij, gate_ij = 1 inside the local window
// (i - j < w) and sigma(lambda g_i . g_j) elsewhere, causal softmax over
// every pair while training).
//
// With dP_ij = dO_i . v_j, D_i = dO_i . O_i and dS_ij = P_ij (dP_ij - D_i):
//   dT_ij = dS_ij scale gate_ij:   dQ_i = sum_j dT_ij k_j,   dK_j = sum_i dT_ij q_i
//   dV_j = sum_i P_ij dO_i
//   for a gated pair, with t_ij = scale q_i . k_j and a_ij = g_i . g_j:
//   da_ij = dS_ij t_ij lambda sigma (1 - sigma):   dG_i gets sum_j da_ij g_j + sum_j da_ji g_j
//   d lambda = sum over gated pairs of dS_ij t_ij a_ij sigma (1 - sigma)
// Two kernels, one per side, each recomputing P from the forward's
// log-sum-exp, so that every sum is owned by one CTA (no atomics, a fixed
// order, bit-identical repeats):
//   query side (CTA: 128 queries x a chunk of 4 heads): dQ per head, the
//     chunk's sum_j da_ij g_j (one partial per chunk) and d lambda;
//   key side (CTA: 128 keys x a kv head, over its query heads): dK, dV and
//     sum_i da_ij g_i (one partial per kv head).
// A CTA's own rows are the TMEM lanes; it streams the other side's tiles.
// Per tile one thread issues three products into TMEM,
//   S = R1 C1^T (q . k, bf16),  A = RG CG^T (g . g, fp16; skipped when every
//   pair of the tile is local),  dP = R2 C2^T (dO . v, bf16)
// with R1, R2, RG the CTA's Q, dO, G_q (query side) or K, V, G_k (key side)
// and C1, C2, CG the streamed tile's K, V, G_k or Q, dO, G_q.  Four
// warpgroups, one per quarter of the tile's columns (a thread per row), read
// them with one TMEM load, release S for the next tile's products, and write
// P, dT and da as bf16 / fp16 operands (the query side into TMEM, the key
// side as 128-byte-swizzled tiles in shared memory); the thread then issues
// the gradient products into TMEM accumulators:
//   query side: dQ += dT C1,  dG_q += da CG
//   key side:   dV += P^T C2,  dK += dT^T C1,  dG_k += da^T CG
// The streamed tiles serve K-major (as the B operand of S, A, dP) and
// MN-major (as the B operand of the gradient products).  Every wait is
// bounded; a CTA that gives up drains its copies and MMAs before it releases
// shared memory and TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "focus_internal.h"
#include "focus_ptx.cuh"

namespace focus {

namespace {

enum { kSideQ = 0, kSideK = 1 };
constexpr int kBR = 128;            // the CTA's own rows (TMEM lanes)
constexpr int kEwGroups = 4;        // elementwise warpgroups: a quarter of a tile's columns each
constexpr int kEwWarps = 4 * kEwGroups;
constexpr int kBwThreads = 32 * kEwWarps + 128;   // + the producer, the MMA thread, 2 idle
constexpr int kBwProducer = kEwWarps;
constexpr int kBwMma = kEwWarps + 1;
// Registers per thread after the split: elementwise warpgroups / the last
// one.  32 kEwWarps * kBwRegsEw + 128 * kBwRegsOther must not exceed the
// launch's kBwThreads * (registers per thread at launch), which the
// preflight checks.
constexpr int kBwRegsEw = 96;
constexpr int kBwRegsOther = 88;
constexpr float kLog2e = 1.4426950408889634f;

enum {
    W_ROWFULL = 0, W_ROWEMPTY = 1, W_CFULL = 2, W_CEMPTY = 6, W_SFULL = 10, W_SFREE = 11,
    W_PFULL = 12, W_PEMPTY = 13, W_ACCDONE = 14, W_ACCFREE = 15, W_DRAIN = 16, kWBars = 17
};

// Shared memory and TMEM columns of one CTA.  BC: rows of a streamed tile
// (64; 32 on the key side for d 128 with K_g > 64, whose accumulators dV, dK
// and dG_k take 2 d + 64 KPC TMEM columns; a 32-row tile halves the work of
// each MMA against the same reads of the CTA's own 128-row operands, so the
// 64-row tile is kept wherever TMEM allows).  The operands P, dT and da sit in
// TMEM (bf16 / fp16 pairs, BC / 2 columns each) where the columns allow,
// else as 128-byte-swizzled tiles in shared memory (key side with d 128 and
// K_g > 64); the streamed tiles pass through as many stages (up to four) as
// shared memory holds.
template <int SIDE, int D, int KPC, int BC>
struct BwLayout {
    static constexpr uint32_t kRowT = kBR * D * 2;        // R1 or R2: D/64 chunks of 16 KB
    static constexpr uint32_t kRowG = kBR * KPC * 128;    // RG: KPC chunks of 16 KB
    static constexpr uint32_t kColT = BC * D * 2;         // C1 or C2: chunks of BC * 128 bytes
    static constexpr uint32_t kColG = BC * KPC * 128;     // CG
    // key side: -lse2 and -D of the tile's queries (2 BC floats, in 1 KB)
    static constexpr uint32_t kVecB = SIDE == kSideK ? 1024 : 0;
    static constexpr uint32_t kStage = 2 * kColT + kColG + kVecB;
    // TMEM columns: S, A, dP, the accumulators, then the operands
    static constexpr uint32_t kColS = 0, kColA = BC, kColP = 2 * BC, kAcc = 3 * BC;
    static constexpr uint32_t kAccG = kAcc + (SIDE == kSideK ? 2 * D : D);
    static constexpr int kNOpd = SIDE == kSideK ? 3 : 2;   // [P,] dT, da
    static constexpr uint32_t kOutM = kAccG + 64 * KPC;
    static constexpr bool kTmemOut = kOutM + kNOpd * (BC / 2) <= 512;
    // Otherwise (key side with d 128): P and dT over the columns of A, which
    // the elementwise pass has read by then (the next tile's A product is
    // issued after this tile's gradient products), da in shared memory.
    static constexpr bool kAOut = !kTmemOut;
    static constexpr uint32_t kOutPm = kTmemOut ? kOutM : kColA;                     // key side: P
    static constexpr uint32_t kOutTm =
        kTmemOut ? kOutM + (SIDE == kSideK ? BC / 2 : 0) : kColA + BC / 2;          // dT
    static constexpr uint32_t kOutAm = kOutTm + BC / 2;                              // da (TMEM)
    // shared memory
    static constexpr uint32_t kOutT = kBR * 128;          // an operand tile: 128 rows of 128 bytes
    static constexpr int kNOut = kTmemOut ? 0 : 1;        // operand tiles in shared memory: da
    static constexpr uint32_t kFixed = 2 * kRowT + kRowG + kNOut * kOutT + 2048;
    static constexpr int NS = kFixed + 4 * kStage <= 232448   ? 4
                              : kFixed + 3 * kStage <= 232448 ? 3
                                                              : 2;
    static constexpr uint32_t kR1 = 0;
    static constexpr uint32_t kR2 = kR1 + kRowT;
    static constexpr uint32_t kRG = kR2 + kRowT;
    static constexpr uint32_t kOut = kRG + kRowG;
    static constexpr uint32_t kC = kOut + kNOut * kOutT;  // stages: C1, C2, CG[, vec]
    static constexpr uint32_t kBar = kC + NS * kStage;
    static constexpr uint32_t kMisc = kBar + kWBars * 8;    // TMEM base, abort flag
    static constexpr uint32_t kRed = kMisc + 16;            // a float per elementwise warp
    static constexpr uint32_t kBytes = kRed + 4 * kEwWarps + 1024;   // + alignment slack
    static_assert(kOutM <= 512 && (kTmemOut || SIDE == kSideK), "TMEM columns");
    static_assert(kBytes <= 232448, "shared memory per CTA");
    static_assert(kStage % 1024 == 0, "stage alignment");
};

struct BwArgs {
    int B, n, Hq, Hkv, nks, Kg, window, hc, nhc, nqt;   // nqt: 128-row query tiles
    float scale;         // softmax scale
    float half_scale;    // scale / 2
    float half_lambda;   // lambda / 2
    float lambda;
    const float *nl2;    // [B, Hq, npad] -lse log2(e), -inf past n
    const float *nD;     // [B, Hq, npad] -dO . O, 0 past n
    int npad;
    float *dq;           // [B, n, Hq, D]
    float *dk, *dv;      // [B, n, Hkv, D]
    float *dg_part;      // [nhc + Hkv][B, n, Kg]
    float *dlam_part;    // [B, nhc, nqt]
    int *status;
    long long *trace;    // nullable: [CTA][kBwTrace] SM cycles (CTAs below trace_ctas)
    int trace_ctas;
};

// Per-CTA trace slots (SM cycles): the producer's waits, the MMA thread's
// waits, the first elementwise thread's waits and phases.
enum {
    BT_P_ROWEMPTY = 0, BT_P_CEMPTY = 1, BT_P_TOTAL = 3,
    BT_M_ROWFULL = 8, BT_M_CFULL = 9, BT_M_SFREE = 10, BT_M_PFULL = 11, BT_M_ACCFREE = 12,
    BT_M_TOTAL = 14,
    BT_E_SFULL = 16, BT_E_TMEM = 17, BT_E_MATH = 18, BT_E_PEMPTY = 19, BT_E_STORE = 20,
    BT_E_ACCDONE = 21, BT_E_TOTAL = 23, BT_E_TILES = 24, kBwTrace = 32
};

// A streamed tile against the CTA's rows: its first column row c0; whether
// some pair of it is gated (i - j >= w), every pair is, and whether some
// pair has j > i.  r0 = the CTA's first row, rend = one past its last valid
// row (query side).
struct BwTile {
    int c0;
    bool gated, allg, causal;
};

template <int SIDE, int BC>
__device__ __forceinline__ BwTile bw_tile(int v, int r0, int rend, int n, int w)
{
    BwTile x;
    if (SIDE == kSideQ) {   // rows = queries [r0, rend), columns = keys [c0, c0 + 64)
        x.c0 = 64 * v;
        x.gated = rend - 1 - x.c0 >= w;
        x.allg = r0 - (x.c0 + 63) >= w;
        x.causal = x.c0 + 63 > r0;
    } else {                // rows = keys [r0, r0 + 128), columns = queries [c0, c0 + BC)
        x.c0 = r0 + BC * v;
        const int ce = min(x.c0 + BC, n);
        x.gated = ce - 1 - r0 >= w;
        x.allg = x.c0 - (r0 + 127) >= w;
        x.causal = r0 + 127 > x.c0;
    }
    return x;
}

// Instruction descriptor of kind::f16 with fp16 A (K-major) and fp16 B
// (MN-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32_bmn(int M, int N)
{
    return idesc_f16_f32(M, N) | (1u << 16);
}

// Loads 16 consecutive fp32 columns of this thread's TMEM lane at each of
// 3 addresses (one wait for all): v[16 * l + c] = column c at a_l.
__device__ __forceinline__ void tmem_ld3x16(uint32_t a0, uint32_t a1, uint32_t a2, float *v)
{
    uint32_t r[48];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
#pragma unroll
    for (int i = 0; i < 48; ++i) v[i] = __uint_as_float(r[i]);
}

// The same with 8 columns at each address: v[8 * l + c].
__device__ __forceinline__ void tmem_ld3x8(uint32_t a0, uint32_t a1, uint32_t a2, float *v)
{
    uint32_t r[24];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
#pragma unroll
    for (int i = 0; i < 24; ++i) v[i] = __uint_as_float(r[i]);
}

// Loads NC (a multiple of 16) consecutive fp32 columns of this thread's TMEM
// lane and waits.
template <int NC>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float *v)
{
    if constexpr (NC % 32 == 0) {
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) tmem_ld32(taddr + 32 * c, v + 32 * c);
    } else {
#pragma unroll
        for (int c = 0; c < NC / 16; ++c) tmem_ld16(taddr + 16 * c, v + 16 * c);
    }
}

// Stores 4 consecutive 32-bit columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_st4u(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}

// Stores 8 consecutive 32-bit columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}

// tanh with the hardware approximation (relative error about 2^-11)
__device__ __forceinline__ float bw_tanh(float x)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
    return t;
}

__device__ __forceinline__ float bw_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes per instruction: a * b + c, a * b, a + b.
__device__ __forceinline__ float2 fma2v(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 mul2v(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 add2v(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// The elementwise constants, as lane pairs.
struct EwConst {
    float2 sc2;   // scale log2(e)
    float2 sc;    // scale
    float2 hs2;   // scale log2(e) / 2
    float2 hs;    // scale / 2
    float2 hl;    // lambda / 2
    float2 q1;    // -scale / 4
    float2 q0;    // scale / 4
    float2 lam;   // lambda
};

// One elementwise pass over this row's HC columns of a tile: from S, A, dP
// (f[0..HC), f[HC..2HC), f[2HC..3HC)) and the columns' or the row's
// -lse2 and -D (nl, nd), the packed P, dT and (GATED) da.  Column c of the
// tile is causal iff c <= lim (query side) / c >= lim (key side), tested
// when CAUSAL (a tile across the diagonal), and gated iff c <= loc /
// c >= loc, tested when EDGE (a gated tile across the window's edge).
template <int SIDE, int HC, bool GATED, bool EDGE, bool CAUSAL>
__device__ __forceinline__ void ew_tile(const float *f, const float *vl, int BC, float2 nl_r,
                                        float2 nd_r, const EwConst &k, int cb, int lim, int loc,
                                        uint32_t *pkP, uint32_t *pkT, uint32_t *pkA, float2 &dl2)
{
#pragma unroll
    for (int e = 0; e < HC; e += 2) {
        const float2 sv = make_float2(f[e], f[e + 1]);
        const float2 dpv = make_float2(f[2 * HC + e], f[2 * HC + e + 1]);
        float2 nl = nl_r, nd = nd_r;
        if (SIDE == kSideK) {
            nl = *reinterpret_cast<const float2 *>(vl + e);
            nd = *reinterpret_cast<const float2 *>(vl + BC + e);
        }
        float2 g2 = k.sc2, g1 = k.sc, sps = make_float2(0.f, 0.f), av = sps;
        if constexpr (GATED) {
            av = make_float2(f[HC + e], f[HC + e + 1]);
            const float2 z = mul2v(av, k.hl);
            const float2 th = make_float2(bw_tanh(z.x), bw_tanh(z.y));
            g2 = fma2v(th, k.hs2, k.hs2);                 // scale log2(e) sigma
            g1 = fma2v(th, k.hs, k.hs);                   // scale sigma
            sps = fma2v(mul2v(th, k.q1), th, k.q0);       // scale sigma (1 - sigma)
            if constexpr (EDGE) {   // a tile across the window's edge: local pairs keep gate 1
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int c = cb + e + q;
                    const bool gp = SIDE == kSideQ ? c <= loc : c >= loc;
                    if (!gp) {
                        (q ? g2.y : g2.x) = k.sc2.x;
                        (q ? g1.y : g1.x) = k.sc.x;
                        (q ? sps.y : sps.x) = 0.f;
                    }
                }
            }
        }
        const float2 xx = fma2v(sv, g2, nl);
        float2 p = make_float2(bw_ex2(xx.x), bw_ex2(xx.y));
        if constexpr (CAUSAL) {
            const int c = cb + e;
            if (!(SIDE == kSideQ ? c <= lim : c >= lim)) p.x = 0.f;
            if (!(SIDE == kSideQ ? c + 1 <= lim : c + 1 >= lim)) p.y = 0.f;
        }
        const float2 ds = mul2v(p, add2v(dpv, nd));
        const float2 dt = mul2v(ds, g1);
        pkP[e / 2] = pack_bf16x2(p.x, p.y);
        pkT[e / 2] = pack_bf16x2(dt.x, dt.y);
        if constexpr (GATED) {
            const float2 u = mul2v(mul2v(ds, sv), sps);   // d gate sigma (1 - sigma)
            const float2 da = mul2v(u, k.lam);
            if (SIDE == kSideQ) dl2 = fma2v(u, av, dl2);
            pkA[e / 2] = pack_f16x2(da.x, da.y);
        }
    }
}

// D[tmem] (+)= A[smem] B[smem] with fp16 A and B: the same instruction as
// the bf16 form, the operand type is in the instruction descriptor.
template <uint32_t AHI, uint32_t BHI>
__device__ __forceinline__ void bw_mma(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                       uint32_t idesc, uint32_t accumulate)
{
    tc_mma_bf16_lo<AHI, BHI>(d_tmem, a_lo, b_lo, idesc, accumulate);
}

template <int SIDE, int D, int KPC, int BC>
__global__ void __launch_bounds__(kBwThreads, 1)
    gated_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmR1,
                        const __grid_constant__ CUtensorMap tmR2,
                        const __grid_constant__ CUtensorMap tmRG,
                        const __grid_constant__ CUtensorMap tmC1,
                        const __grid_constant__ CUtensorMap tmC2,
                        const __grid_constant__ CUtensorMap tmCG, const BwArgs a)
{
    using L = BwLayout<SIDE, D, KPC, BC>;
    constexpr int kChunks = D / 64;
    constexpr int HC = BC / kEwGroups;  // columns per elementwise warpgroup
    constexpr int NS = L::NS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kMisc + 4);
    float *red = reinterpret_cast<float *>(sm + L::kRed);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.z;
    const int kvq = a.Hq / a.Hkv;
    const int64_t cta = ((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    long long *tr = (a.trace && cta < a.trace_ctas) ? a.trace + cta * kBwTrace : nullptr;
    const long long t_start = clock64();
    // the CTA's rows, heads and streamed tiles
    int r0, rend, h0, nh, ncol, kvh0;
    if (SIDE == kSideQ) {
        const int qt = gridDim.x - 1 - blockIdx.x;   // the longest rows first
        r0 = kBR * qt;
        rend = min(r0 + kBR, a.n);
        h0 = blockIdx.y * a.hc;
        nh = min(a.hc, a.Hq - h0);
        ncol = (rend + 63) / 64;                    // key tiles [0, rend)
        kvh0 = 0;
    } else {
        r0 = kBR * blockIdx.x;
        rend = min(r0 + kBR, a.n);
        kvh0 = blockIdx.y;
        h0 = kvh0 * kvq;
        nh = kvq;
        ncol = (a.n - r0 + BC - 1) / BC;            // query tiles [r0, n)
    }

    if (threadIdx.x == 0) {
        mbar_init(&bars[W_ROWFULL], 1);
        mbar_init(&bars[W_ROWEMPTY], 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars[W_CFULL + s], 1);
            mbar_init(&bars[W_CEMPTY + s], 1);
        }
        mbar_init(&bars[W_SFULL], 1);
        mbar_init(&bars[W_SFREE], kEwWarps);
        mbar_init(&bars[W_PFULL], kEwWarps);
        mbar_init(&bars[W_PEMPTY], 1);
        mbar_init(&bars[W_ACCDONE], 1);
        mbar_init(&bars[W_ACCFREE], kEwWarps);
        mbar_init(&bars[W_DRAIN], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kBwMma) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kBwProducer && lane == 0) {
        tma_prefetch_desc(&tmR1);
        tma_prefetch_desc(&tmR2);
        tma_prefetch_desc(&tmRG);
        tma_prefetch_desc(&tmC1);
        tma_prefetch_desc(&tmC2);
        tma_prefetch_desc(&tmCG);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // (set-up above touches no global memory; launched with launch_pdl)
    grid_dep_sync();

    if (warp >= kEwWarps) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBwRegsOther));
        if (warp == kBwProducer) {
            // --------------------------------------------------------- producer
            int t = 0;
            int nrow = 0;   // row-operand loads issued
            bool ok = true;
            long long ptr_[4] = {0, 0, 0, 0};   // producer slots
            for (int hi = 0; ok && hi < nh; ++hi) {
                const int h = h0 + hi;
                if (SIDE == kSideQ || hi == 0) {
                    if (hi > 0 && lane == 0)
                        ok = mbar_wait_t(&bars[W_ROWEMPTY], (hi - 1) & 1, abort_flag, a.status,
                                     tr != nullptr, ptr_[BT_P_ROWEMPTY]);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t *d1 = sm + L::kR1, *d2 = sm + L::kR2, *dg = sm + L::kRG;
                        const uint32_t bytes = 2 * L::kRowT + (hi == 0 ? L::kRowG : 0u);
                        mbar_arrive_expect_tx(&bars[W_ROWFULL], bytes);
                        const int rh = SIDE == kSideQ ? h : kvh0;   // head of R1 / R2
                        for (int c = 0; c < kChunks; ++c) {
                            tma_load_4d(d1 + c * 16384, &tmR1, &bars[W_ROWFULL], c * 64, rh, r0, b);
                            tma_load_4d(d2 + c * 16384, &tmR2, &bars[W_ROWFULL], c * 64, rh, r0, b);
                        }
                        if (hi == 0)
                            for (int c = 0; c < KPC; ++c)
                                tma_load_4d(dg + c * 16384, &tmRG, &bars[W_ROWFULL], c * 64, 0,
                                            r0, b);
                    }
                    ++nrow;
                }
                for (int v = 0; ok && v < ncol; ++v, ++t) {
                    const int st = t % NS;
                    if (t >= NS && lane == 0)
                        ok = mbar_wait_t(&bars[W_CEMPTY + st], ((t / NS) - 1) & 1, abort_flag,
                                         a.status, tr != nullptr, ptr_[BT_P_CEMPTY]);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        ok = false;
                        break;
                    }
                    const int c0 = SIDE == kSideQ ? 64 * v : r0 + BC * v;
                    if (lane == 0) {
                        uint8_t *sc = sm + L::kC + st * L::kStage;
                        mbar_arrive_expect_tx(&bars[W_CFULL + st],
                                              L::kStage - L::kVecB + (SIDE == kSideK ? 8 * BC : 0));
                        if (SIDE == kSideK) {
                            // the tile's queries: minus the base-2 log-sum-exp (-inf
                            // past n: P = 0) and minus D, from rows padded past n
                            const int64_t x = ((int64_t)b * a.Hq + h) * a.npad + c0;
                            uint8_t *vd = sc + 2 * L::kColT + L::kColG;
                            bulk_load(vd, a.nl2 + x, 4 * BC, &bars[W_CFULL + st]);
                            bulk_load(vd + 4 * BC, a.nD + x, 4 * BC, &bars[W_CFULL + st]);
                        }
                        const int ch = SIDE == kSideQ ? h / kvq : h;   // head of C1 / C2
                        for (int c = 0; c < kChunks; ++c) {
                            tma_load_4d(sc + c * (BC * 128), &tmC1, &bars[W_CFULL + st], c * 64,
                                        ch, c0, b);
                            tma_load_4d(sc + L::kColT + c * (BC * 128), &tmC2, &bars[W_CFULL + st],
                                        c * 64, ch, c0, b);
                        }
                        for (int c = 0; c < KPC; ++c)
                            tma_load_4d(sc + 2 * L::kColT + c * (BC * 128), &tmCG,
                                        &bars[W_CFULL + st], c * 64, 0, c0, b);
                    }
                    __syncwarp();
                }
            }
            if (tr && lane == 0) {
                ptr_[BT_P_TOTAL] = clock64() - t_start;
                for (int i = 0; i < 4; ++i) tr[i] = ptr_[i];
            }
            // A CTA that gave up lets the copies already issued land before
            // shared memory is released.
            if (*abort_flag && lane == 0) {
                const uint64_t t0 = global_timer_ns();
                if (nrow > 0)
                    while (!mbar_try_wait(&bars[W_ROWFULL], (nrow - 1) & 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                for (int tt = max(0, t - NS); tt <= t; ++tt)
                    while (!mbar_try_wait(&bars[W_CFULL + tt % NS], (tt / NS) & 1) &&
                           global_timer_ns() - t0 < 300000000ull) {
                    }
            }
        } else if (warp == kBwMma) {
            // ----------------------------------------------------- MMA issuer
            if (lane == 0) {
                constexpr uint32_t kIdS = idesc_bf16_f32(kBR, BC, false, false);
                constexpr uint32_t kIdA = idesc_f16_f32(kBR, BC);
                constexpr uint32_t kIdAcc = idesc_bf16_f32(kBR, D, false, true);
                constexpr uint32_t kIdG = idesc_f16_f32_bmn(kBR, 64 * KPC);
                constexpr uint32_t kHi = sdesc_hi(1024);
                const uint32_t r1 = sdesc_lo(smem_u32(sm + L::kR1), 16);
                const uint32_t r2 = sdesc_lo(smem_u32(sm + L::kR2), 16);
                const uint32_t rg = sdesc_lo(smem_u32(sm + L::kRG), 16);
                // streamed tiles: the leading offset is the MN-major chunk stride
                // (unused by the K-major products)
                const uint32_t cb = sdesc_lo(smem_u32(sm + L::kC), BC * 128);
                const uint32_t outA = sdesc_lo(smem_u32(sm + L::kOut), 16);   // da (kAOut)
                int t = 0;
                bool ok = true, dg_started = false;
                const bool trc = tr != nullptr;
                long long mtr[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // slots 8..15
                int pt = -1, p_hi = 0;                 // the tile whose gradient products are next
                bool p_gated = false, p_first = false, p_last = false;
                // the gradient products of tile tt: dQ, or dV and dK, first ...
                auto grads_main = [&](int tt, bool first, int hi) -> bool {
                    if (!mbar_wait_t(&bars[W_PFULL], tt & 1, abort_flag, a.status, trc,
                                     mtr[BT_M_PFULL - 8]))
                        return false;
                    if (SIDE == kSideQ && first && hi > 0 &&
                        !mbar_wait_t(&bars[W_ACCFREE], (hi - 1) & 1, abort_flag, a.status, trc,
                                     mtr[BT_M_ACCFREE - 8]))
                        return false;
                    tc_fence_after();
                    const uint32_t c1 = cb + (tt % NS) * (L::kStage >> 4);
                    const uint32_t c2 = c1 + (L::kColT >> 4);
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk) {
                        // operands in TMEM: 16 rows of the streamed tile = 8 columns
                        // per step; B: 16 rows of 128 bytes further
                        const uint32_t bo = kk * 128;
                        if (SIDE == kSideQ) {
                            const uint32_t acc = (kk > 0 || !first) ? 1u : 0u;
                            tc_mma_bf16_ts_lo<kHi>(tmem + L::kAcc, tmem + L::kOutTm + kk * 8,
                                                   c1 + bo, kIdAcc, acc);
                        } else {
                            const uint32_t acc = (kk > 0 || tt > 0) ? 1u : 0u;
                            tc_mma_bf16_ts_lo<kHi>(tmem + L::kAcc, tmem + L::kOutPm + kk * 8,
                                                   c2 + bo, kIdAcc, acc);
                            tc_mma_bf16_ts_lo<kHi>(tmem + L::kAcc + D, tmem + L::kOutTm + kk * 8,
                                                   c1 + bo, kIdAcc, acc);
                        }
                    }
                    return true;
                };
                // ... then dG and the releases
                auto grads_tail = [&](int tt, bool gtd, bool last) {
                    const uint32_t cg = cb + (tt % NS) * (L::kStage >> 4) + 2 * (L::kColT >> 4);
                    if (gtd) {
#pragma unroll
                        for (int kk = 0; kk < BC / 16; ++kk) {
                            const uint32_t acc = (kk > 0 || dg_started) ? 1u : 0u;
                            if (L::kTmemOut)
                                tc_mma_bf16_ts_lo<kHi>(tmem + L::kAccG, tmem + L::kOutAm + kk * 8,
                                                       cg + kk * 128, kIdG, acc);
                            else
                                bw_mma<kHi, kHi>(tmem + L::kAccG, outA + kk * 2, cg + kk * 128,
                                                 kIdG, acc);
                        }
                        dg_started = true;
                    }
                    tc_commit(&bars[W_PEMPTY]);
                    tc_commit(&bars[W_CEMPTY + tt % NS]);
                    if (SIDE == kSideQ && last) tc_commit(&bars[W_ACCDONE]);
                };
                auto grads = [&](int tt, bool gtd, bool first, bool last, int hi) -> bool {
                    if (!grads_main(tt, first, hi)) return false;
                    grads_tail(tt, gtd, last);
                    return true;
                };
                for (int hi = 0; ok && hi < nh; ++hi) {
                    if (SIDE == kSideQ || hi == 0) {
                        ok = mbar_wait_t(&bars[W_ROWFULL], hi & 1, abort_flag, a.status, trc,
                                     mtr[BT_M_ROWFULL - 8]);
                        if (!ok) break;
                    }
                    for (int v = 0; ok && v < ncol; ++v, ++t) {
                        const BwTile x = bw_tile<SIDE, BC>(v, r0, rend, a.n, a.window);
                        const int st = t % NS;
                        ok = mbar_wait_t(&bars[W_CFULL + st], (t / NS) & 1, abort_flag, a.status,
                                         trc, mtr[BT_M_CFULL - 8]);
                        if (ok && t > 0)
                            ok = mbar_wait_t(&bars[W_SFREE], (t - 1) & 1, abort_flag, a.status,
                                             trc, mtr[BT_M_SFREE - 8]);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t c1 = cb + st * (L::kStage >> 4);
                        const uint32_t c2 = c1 + (L::kColT >> 4), cg = c2 + (L::kColT >> 4);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t ro = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                            const uint32_t co = ((kk >> 2) * (BC * 128) + (kk & 3) * 32) >> 4;
                            const uint32_t acc = kk > 0 ? 1u : 0u;
                            bw_mma<kHi, kHi>(tmem + L::kColS, r1 + ro, c1 + co, kIdS, acc);
                            bw_mma<kHi, kHi>(tmem + L::kColP, r2 + ro, c2 + co, kIdS, acc);
                        }
                        auto issue_a = [&]() {
                            if (!x.gated) return;
#pragma unroll
                            for (int ks = 0; ks < 4 * KPC; ++ks) {
                                if (ks >= a.nks) break;
                                const uint32_t ro = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                                const uint32_t co = ((ks >> 2) * (BC * 128) + (ks & 3) * 32) >> 4;
                                bw_mma<kHi, kHi>(tmem + L::kColA, rg + ro, cg + co, kIdA,
                                                 ks > 0 ? 1u : 0u);
                            }
                        };
                        if constexpr (L::kAOut) {
                            // A's columns hold the previous tile's P and dT until its
                            // dV and dK products are issued (the tensor pipe runs in
                            // issue order); its dG product, on da in shared memory,
                            // follows the signal
                            if (pt >= 0) ok = grads_main(pt, p_first, p_hi);
                            if (!ok) break;
                            issue_a();
                            tc_commit(&bars[W_SFULL]);
                            if (pt >= 0) grads_tail(pt, p_gated, p_last);
                        } else {
                            issue_a();
                            tc_commit(&bars[W_SFULL]);
                            if (SIDE == kSideQ && v == ncol - 1) tc_commit(&bars[W_ROWEMPTY]);
                            if (pt >= 0) ok = grads(pt, p_gated, p_first, p_last, p_hi);
                        }
                        pt = t;
                        p_gated = x.gated;
                        p_first = v == 0;
                        p_last = v == ncol - 1;
                        p_hi = hi;
                    }
                }
                if (ok && pt >= 0) ok = grads(pt, p_gated, p_first, p_last, p_hi);
                if (ok && SIDE == kSideK) tc_commit(&bars[W_ACCDONE]);
                if (trc) {
                    mtr[BT_M_TOTAL - 8] = clock64() - t_start;
                    for (int i = 0; i < 8; ++i) tr[8 + i] = mtr[i];
                }
                // every MMA issued completes before TMEM is released
                tc_commit(&bars[W_DRAIN]);
                mbar_wait_until(&bars[W_DRAIN], 0, global_timer_ns() + 500000000ull);
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBwRegsEw));
        // ------------------------------------- elementwise (warps 0-7)
        const int wg = warp >> 2;                 // quarter of the tile's columns
        const int r = (warp & 3) * 32 + lane;     // own row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int row = r0 + r;                   // query (query side) or key (key side)
        EwConst kc;
        kc.sc2 = make_float2(a.scale * kLog2e, a.scale * kLog2e);
        kc.sc = make_float2(a.scale, a.scale);
        kc.hs2 = make_float2(a.half_scale * kLog2e, a.half_scale * kLog2e);
        kc.hs = make_float2(a.half_scale, a.half_scale);
        kc.hl = make_float2(a.half_lambda, a.half_lambda);
        kc.q1 = make_float2(-0.5f * a.half_scale, -0.5f * a.half_scale);
        kc.q0 = make_float2(0.5f * a.half_scale, 0.5f * a.half_scale);
        kc.lam = make_float2(a.lambda, a.lambda);
        float2 dl2 = make_float2(0.f, 0.f);
        const bool etr = tr != nullptr && threadIdx.x == 0;
        long long etr_[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};   // slots 16..31
        bool ok = true;
        int t = 0;
        uint8_t *oA = sm + L::kOut;   // da (kAOut)
        for (int hi = 0; ok && hi < nh; ++hi) {
            const int h = h0 + hi;
            // query side: minus this row's base-2 log-sum-exp (-inf past n) and D
            float2 nl_r = make_float2(-CUDART_INF_F, -CUDART_INF_F), nd_r = make_float2(0.f, 0.f);
            if (SIDE == kSideQ) {   // rows below npad: -inf and 0 past n
                const int64_t x = ((int64_t)b * a.Hq + h) * a.npad + row;
                const float l2 = a.nl2[x], dd = a.nD[x];
                nl_r = make_float2(l2, l2);
                nd_r = make_float2(dd, dd);
            }
            for (int v = 0; ok && v < ncol; ++v, ++t) {
                const BwTile x = bw_tile<SIDE, BC>(v, r0, rend, a.n, a.window);
                ok = mbar_wait_t(&bars[W_SFULL], t & 1, abort_flag, a.status, etr,
                                 etr_[BT_E_SFULL - 16]);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                long long te = etr ? clock64() : 0;
                float f[3 * HC];   // S, A, dP of this row's HC columns
                const uint32_t cc = wg * HC;
                if constexpr (HC == 16)
                    tmem_ld3x16(trow + L::kColS + cc, trow + L::kColA + cc, trow + L::kColP + cc,
                                f);
                else
                    tmem_ld3x8(trow + L::kColS + cc, trow + L::kColA + cc, trow + L::kColP + cc, f);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[W_SFREE]);   // S, A, dP may be overwritten
                if (etr) {
                    const long long t2 = clock64();
                    etr_[BT_E_TMEM - 16] += t2 - te;
                    te = t2;
                }
                // key side: the stage's -lse2 and -D, from this warpgroup's columns
                const float *vl = reinterpret_cast<const float *>(
                                      sm + L::kC + (t % NS) * L::kStage + 2 * L::kColT + L::kColG) +
                                  wg * HC;
                uint32_t pkP[HC / 2], pkT[HC / 2], pkA[HC / 2];
                const int dlt = row - x.c0;   // the row against the tile's first column
                const int loc = SIDE == kSideQ ? dlt - a.window : dlt + a.window;
                // the tile's kind (uniform over the CTA): gated or not, across
                // the window's edge, across the diagonal
#define FOCUS_EW(G, E, C)                                                                       \
    ew_tile<SIDE, HC, G, E, C>(f, vl, BC, nl_r, nd_r, kc, wg * HC, dlt, loc, pkP, pkT, pkA, dl2)
                if (!x.gated) {
                    if (x.causal) FOCUS_EW(false, false, true);
                    else FOCUS_EW(false, false, false);
                } else if (x.allg) {
                    if (x.causal) FOCUS_EW(true, false, true);
                    else FOCUS_EW(true, false, false);
                } else {
                    if (x.causal) FOCUS_EW(true, true, true);
                    else FOCUS_EW(true, true, false);
                }
#undef FOCUS_EW
                // the operand tiles are free once the previous tile's gradient
                // products are done
                if (etr) {
                    const long long t2 = clock64();
                    etr_[BT_E_MATH - 16] += t2 - te;
                    te = t2;
                }
                if (t > 0)
                    ok = mbar_wait_t(&bars[W_PEMPTY], (t - 1) & 1, abort_flag, a.status, etr,
                                     etr_[BT_E_PEMPTY - 16]);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if constexpr (L::kTmemOut) {
                    // [P,] dT and da into TMEM: this row's HC columns as HC / 2 pairs
                    static_assert(HC == 8 || HC == 16, "4 or 8 TMEM columns per operand");
                    const uint32_t tc = trow + wg * (HC / 2);
                    if constexpr (HC == 16) {
                        if (SIDE == kSideK) tmem_st8u(tc + L::kOutPm, pkP);
                        tmem_st8u(tc + L::kOutTm, pkT);
                        if (x.gated) tmem_st8u(tc + L::kOutAm, pkA);
                    } else {
                        if (SIDE == kSideK) tmem_st4u(tc + L::kOutPm, pkP);
                        tmem_st4u(tc + L::kOutTm, pkT);
                        if (x.gated) tmem_st4u(tc + L::kOutAm, pkA);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                } else {
                    // P and dT over A's columns (read above), da as a tile in shared
                    // memory: row r, columns [wg HC, wg HC + HC) as 16-byte units u
                    // of the 128-byte row at (u xor (r mod 8))
                    const uint32_t tc = trow + wg * (HC / 2);
                    if constexpr (HC == 16) {
                        tmem_st8u(tc + L::kOutPm, pkP);
                        tmem_st8u(tc + L::kOutTm, pkT);
                    } else {
                        tmem_st4u(tc + L::kOutPm, pkP);
                        tmem_st4u(tc + L::kOutTm, pkT);
                    }
                    if (x.gated) {   // the dG product runs on gated tiles only
                        const uint32_t rowoff = (uint32_t)r * 128u;
#pragma unroll
                        for (int q = 0; q < HC / 8; ++q) {
                            const uint32_t u = (uint32_t)(wg * (HC / 8) + q);
                            const uint32_t off = rowoff + ((u ^ (uint32_t)(r & 7)) << 4);
                            st_shared_v4(smem_u32(oA + off), pkA[4 * q], pkA[4 * q + 1],
                                         pkA[4 * q + 2], pkA[4 * q + 3]);
                        }
                        fence_proxy_async_smem();   // the MMA reads the tile through the async proxy
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[W_PFULL]);
                if (etr) {
                    etr_[BT_E_STORE - 16] += clock64() - te;
                    etr_[BT_E_TILES - 16] += 1;
                }
                if (SIDE == kSideQ && v == ncol - 1) {
                    // dQ of head h is complete: this row's quarter of its columns
                    ok = mbar_wait_t(&bars[W_ACCDONE], hi & 1, abort_flag, a.status, etr,
                                     etr_[BT_E_ACCDONE - 16]);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    constexpr int QC = D / kEwGroups;
                    float o[QC];
                    tmem_ldn<QC>(trow + L::kAcc + wg * QC, o);
                    float4 *dst = reinterpret_cast<float4 *>(
                        a.dq + (((int64_t)b * a.n + row) * a.Hq + h) * D + wg * QC);
                    if (row < a.n)
#pragma unroll
                        for (int q = 0; q < QC / 4; ++q)
                            dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[W_ACCFREE]);
                }
            }
        }
        // ---- the CTA's accumulators
        if (ok && SIDE == kSideK) {
            ok = mbar_wait_t(&bars[W_ACCDONE], 0, abort_flag, a.status, etr,
                             etr_[BT_E_ACCDONE - 16]);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const bool valid = row < a.n;
            if (SIDE == kSideK) {
                // dV and dK: this row's quarter of the D columns of each
                constexpr int QC = D / kEwGroups;
                const int64_t base = (((int64_t)b * a.n + row) * a.Hkv + kvh0) * D + wg * QC;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    float o[QC];
                    tmem_ldn<QC>(trow + L::kAcc + m * D + wg * QC, o);
                    float4 *dst = reinterpret_cast<float4 *>((m == 0 ? a.dv : a.dk) + base);
                    if (valid)
#pragma unroll
                        for (int q = 0; q < QC / 4; ++q)
                            dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                }
            }
            // the dG partial: this row's quarter of the 64 KPC columns (zero
            // when no pair of the CTA is gated)
            const bool any_gated = SIDE == kSideQ ? (rend - 1 >= a.window)
                                                  : (a.n - 1 - r0 >= a.window);
            const int part = SIDE == kSideQ ? blockIdx.y : a.nhc + kvh0;
            float *dst = a.dg_part + ((int64_t)part * a.B * a.n + (int64_t)b * a.n + row) * a.Kg;
            constexpr int GC = 64 * KPC / kEwGroups;
            float o[GC];
            if (any_gated) {
                tmem_ldn<GC>(trow + L::kAccG + wg * GC, o);
            } else {
#pragma unroll
                for (int q = 0; q < GC; ++q) o[q] = 0.f;
            }
            if (valid)
#pragma unroll
                for (int q = 0; q < GC; ++q)
                    if (wg * GC + q < a.Kg) dst[wg * GC + q] = o[q];
        }
        if (etr) {
            etr_[BT_E_TOTAL - 16] = clock64() - t_start;
            for (int i = 0; i < 16; ++i) tr[16 + i] = etr_[i];
        }
        if (SIDE == kSideQ) {
            // d lambda: this CTA's partial, the EW warps' sums in a fixed order
            float dlam = dl2.x + dl2.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, off);
            if (lane == 0) red[warp] = dlam;
            named_bar_sync(1, 32 * kEwWarps);
            if (threadIdx.x == 0 && !*abort_flag) {
                float s = 0.f;
                for (int w = 0; w < kEwWarps; ++w) s += red[w];
                const int qt = gridDim.x - 1 - blockIdx.x;
                a.dlam_part[((int64_t)b * a.nhc + blockIdx.y) * a.nqt + qt] = s;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBwMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int SIDE, int D, int KPC, int BC>
cudaError_t bw_preflight_t()
{
    auto kern = gated_bwd_tc_kernel<SIDE, D, KPC, BC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)BwLayout<SIDE, D, KPC, BC>::kBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    // the warpgroups' shares after setmaxnreg must fit in the launch's registers
    if ((int64_t)fa.numRegs * kBwThreads < 32 * kEwWarps * kBwRegsEw + 128 * kBwRegsOther)
        return cudaErrorInvalidConfiguration;
    return cudaSuccess;
}

template <int SIDE, int D, int KPC, int BC>
cudaError_t bw_launch_t(const GatedBwTcPlan &plan, const BwArgs &a, cudaStream_t s)
{
    const int m = SIDE == kSideQ ? 0 : 6;
    const dim3 grid = SIDE == kSideQ ? dim3((unsigned)a.nqt, (unsigned)a.nhc, (unsigned)a.B)
                                     : dim3((unsigned)((a.n + kBR - 1) / kBR), (unsigned)a.Hkv,
                                            (unsigned)a.B);
    return launch_pdl(gated_bwd_tc_kernel<SIDE, D, KPC, BC>, grid, dim3(kBwThreads),
                      (size_t)BwLayout<SIDE, D, KPC, BC>::kBytes, s, plan.map[m], plan.map[m + 1],
                      plan.map[m + 2], plan.map[m + 3], plan.map[m + 4], plan.map[m + 5], a);
}

// The key side's streamed tile: 64 query rows, 32 for d 128 with K_g > 64
// (TMEM columns for the accumulators).
inline int bw_key_bc(int d, int Kg) { return (d == 128 && Kg > 64) ? 32 : 64; }

}  // namespace

cudaError_t gated_bwd_tc_preflight(int d, int Kg)
{
    cudaError_t e;
    if (d == 64) {
        if (Kg > 64) {
            if ((e = bw_preflight_t<kSideQ, 64, 2, 64>()) != cudaSuccess) return e;
            return bw_preflight_t<kSideK, 64, 2, 64>();
        }
        if ((e = bw_preflight_t<kSideQ, 64, 1, 64>()) != cudaSuccess) return e;
        return bw_preflight_t<kSideK, 64, 1, 64>();
    }
    if (Kg > 64) {
        if ((e = bw_preflight_t<kSideQ, 128, 2, 64>()) != cudaSuccess) return e;
        return bw_preflight_t<kSideK, 128, 2, 32>();
    }
    if ((e = bw_preflight_t<kSideQ, 128, 1, 64>()) != cudaSuccess) return e;
    return bw_preflight_t<kSideK, 128, 1, 64>();
}

cudaError_t gated_bwd_tc_prepare(const GatedLaunch &p, const __half *g16, int kp,
                                 GatedBwTcPlan *plan)
{
    cudaError_t e = gated_bwd_tc_preflight(p.d, p.Kg);
    if (e != cudaSuccess) return e;
    plan->p = p;
    plan->kp = kp;
    const uint32_t kbc = (uint32_t)bw_key_bc(p.d, p.Kg);
    // query side: rows Q, dO, G_q (128); streamed K, V, G_k (64)
    // key side: rows K, V, G_k (128); streamed Q, dO, G_q (64, or 32)
    if (!make_map_4d(&plan->map[0], p.q, false, p.B, p.n, p.Hq, p.d, 128) ||
        !make_map_4d(&plan->map[1], p.dO, false, p.B, p.n, p.Hq, p.d, 128) ||
        !make_map_4d(&plan->map[2], g16, true, p.B, p.n, 1, kp, 128) ||
        !make_map_4d(&plan->map[3], p.k, false, p.B, p.n, p.Hkv, p.d, 64) ||
        !make_map_4d(&plan->map[4], p.v, false, p.B, p.n, p.Hkv, p.d, 64) ||
        !make_map_4d(&plan->map[5], g16, true, p.B, p.n, 1, kp, 64) ||
        !make_map_4d(&plan->map[6], p.k, false, p.B, p.n, p.Hkv, p.d, 128) ||
        !make_map_4d(&plan->map[7], p.v, false, p.B, p.n, p.Hkv, p.d, 128) ||
        !make_map_4d(&plan->map[8], g16, true, p.B, p.n, 1, kp, 128) ||
        !make_map_4d(&plan->map[9], p.q, false, p.B, p.n, p.Hq, p.d, kbc) ||
        !make_map_4d(&plan->map[10], p.dO, false, p.B, p.n, p.Hq, p.d, kbc) ||
        !make_map_4d(&plan->map[11], g16, true, p.B, p.n, 1, kp, kbc))
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t gated_bwd_tc_launch(const GatedBwTcPlan &plan, const float *rowv, int npad,
                                float *dlam_part, float *dg_part, cudaStream_t s, int *launches)
{
    const GatedLaunch &p = plan.p;
    BwArgs a;
    a.B = p.B;
    a.n = p.n;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.nks = plan.kp / 16;
    a.Kg = p.Kg;
    a.window = std::min(p.window, p.n);   // i - j < n for every pair
    a.hc = std::min(kGatedHeadChunk, p.Hq);
    a.nhc = (p.Hq + a.hc - 1) / a.hc;
    a.nqt = (p.n + kBR - 1) / kBR;
    a.scale = p.scale;
    a.half_scale = 0.5f * p.scale;
    a.half_lambda = 0.5f * p.lambda;
    a.lambda = p.lambda;
    a.nl2 = rowv;
    a.nD = rowv + (size_t)p.B * p.Hq * npad;
    a.npad = npad;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.dg_part = dg_part;
    a.dlam_part = dlam_part;
    a.status = p.wc.status;
    a.trace = nullptr;
    a.trace_ctas = 0;
    cudaError_t e;
    const bool two = p.Kg > 64;
    gated_trace_buffer(0, &a.trace, &a.trace_ctas);
    prof_begin("gated_bwd_dq", s);
    if (p.d == 64)
        e = two ? bw_launch_t<kSideQ, 64, 2, 64>(plan, a, s)
                : bw_launch_t<kSideQ, 64, 1, 64>(plan, a, s);
    else
        e = two ? bw_launch_t<kSideQ, 128, 2, 64>(plan, a, s)
                : bw_launch_t<kSideQ, 128, 1, 64>(plan, a, s);
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    gated_trace_buffer(1, &a.trace, &a.trace_ctas);
    prof_begin("gated_bwd_dkv", s);
    if (p.d == 64)
        e = two ? bw_launch_t<kSideK, 64, 2, 64>(plan, a, s)
                : bw_launch_t<kSideK, 64, 1, 64>(plan, a, s);
    else
        e = two ? bw_launch_t<kSideK, 128, 2, 32>(plan, a, s)
                : bw_launch_t<kSideK, 128, 1, 64>(plan, a, s);
    prof_end(s);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

int gated_bwd_tc_dlam_count(int B, int n, int Hq)
{
    const int hc = std::min(kGatedHeadChunk, Hq);
    return B * ((Hq + hc - 1) / hc) * ((n + kBR - 1) / kBR);
}

}  // namespace focus
