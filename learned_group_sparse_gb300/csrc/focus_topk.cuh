// Per-row top-NS selection for the assignment epilogues (Focus, gist.science/zh
// technical summary 2.1.3: at inference a token joins its k highest-scoring
// groups; NS = k + 1 so that the margin to the first group left out is known).
//
// One thread owns one token's score row (its TMEM lane) and keeps the NS best
// (score, id) pairs in registers, in descending order with equal scores going
// to the lower id.  Candidates are offered in increasing id order, so once the
// list holds NS real entries (after the first NS candidates) every kept id is
// lower than the candidate's and a tie never displaces a kept entry: a plain
// "score >" decides.  The insertion is branch-free (NS compares, then each
// slot selects its old value, its upper neighbour or the candidate), so the
// 32 rows of a warp never diverge.
#pragma once

#include <math_constants.h>
#include <stdint.h>

namespace focus {

// (score, id) order: larger score first, equal scores -> lower id first.
__device__ __forceinline__ bool topk_better(float s1, int i1, float s2, int i2)
{
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

template <int NS>
struct TopList {
    float s[NS];
    int i[NS];

    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            s[q] = -CUDART_INF_F;
            i[q] = 0x7fffffff;   // an empty slot loses to every real candidate
        }
    }

    // Slot q takes its upper neighbour if the candidate beats slot q - 1, the
    // candidate if it beats slot q only, else keeps its value.  g[] is
    // computed from the old list; slots are rewritten from the bottom up.
    __device__ __forceinline__ void insert(float cv, int ci, const bool *g)
    {
#pragma unroll
        for (int q = NS - 1; q > 0; --q) {
            s[q] = g[q - 1] ? s[q - 1] : (g[q] ? cv : s[q]);
            i[q] = g[q - 1] ? i[q - 1] : (g[q] ? ci : i[q]);
        }
        s[0] = g[0] ? cv : s[0];
        i[0] = g[0] ? ci : i[0];
    }

    // Any candidate, with the full order (used while empty slots remain).
    // NaN scores rank as -inf.
    __device__ __forceinline__ void offer_first(float cv, int ci)
    {
        if (cv != cv) cv = -CUDART_INF_F;
        bool g[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) g[q] = topk_better(cv, ci, s[q], i[q]);
        insert(cv, ci, g);
    }

    // A candidate whose id is above every kept id, once the list is full.
    __device__ __forceinline__ void offer_next(float cv, int ci)
    {
        if (cv != cv) cv = -CUDART_INF_F;
        bool g[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) g[q] = cv > s[q];
        insert(cv, ci, g);
    }

    // Merges another sorted list into this one (keeps the NS best of both).
    __device__ __forceinline__ void merge(const float *os, const int *oi)
    {
        float ms[NS];
        int mi[NS];
        int a = 0, b = 0;
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            // a + b == q <= NS - 1, so both heads exist
            float sa = -CUDART_INF_F, sb = -CUDART_INF_F;
            int ia = 0x7fffffff, ib = 0x7fffffff;
#pragma unroll
            for (int x = 0; x < NS; ++x) {
                if (x == a) {
                    sa = s[x];
                    ia = i[x];
                }
                if (x == b) {
                    sb = os[x];
                    ib = oi[x];
                }
            }
            const bool ta = topk_better(sa, ia, sb, ib);
            ms[q] = ta ? sa : sb;
            mi[q] = ta ? ia : ib;
            a += ta ? 1 : 0;
            b += ta ? 0 : 1;
        }
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            s[q] = ms[q];
            i[q] = mi[q];
        }
    }

    // Smallest gap between consecutive kept scores among the first nsel.
    __device__ __forceinline__ float gap(int nsel) const
    {
        float g = CUDART_INF_F;
#pragma unroll
        for (int q = 1; q < NS; ++q)
            if (q < nsel) g = fminf(g, s[q - 1] - s[q]);
        return g;
    }
};

}  // namespace focus
