// Host-side launcher shared by the attention translation units.
#pragma once

#include "focus_attn_kernel.cuh"
#include "focus_internal.h"

namespace focus {

template <int MODE, int D>
cudaError_t launch_attn_impl(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    if (p.grid <= 0) return cudaSuccess;
    auto kern = focus_attn_kernel<MODE, D>;
    constexpr uint32_t smem = AttnSmem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    AttnArgs a;
    a.B = p.B;
    a.n = p.n;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.rows = p.rows;
    a.window = p.window;
    a.scale_log2 = p.scale_log2;
    a.K = p.K;
    a.topk = p.topk;
    a.ids = p.ids;
    a.offsets = p.offsets;
    a.pos = p.pos;
    a.tiles = p.tiles;
    a.ntiles = p.ntiles;
    a.out = p.out;
    a.lse = p.lse;
    a.part_out = p.part_out;
    a.part_lse_out = p.part_lse_out;
    a.part_o = p.part_o;
    a.part_lse = p.part_lse;
    a.inv = p.inv;
    a.status = p.status;
    a.pair_count = p.pair_count;
    prof_begin(MODE == kGroup ? "attn_group" : MODE == kWindow ? "attn_window" : "attn_dense", s);
    kern<<<(unsigned)p.grid, kThreads, smem, s>>>(*p.tmQ, *p.tmK, *p.tmV, a);
    prof_end(s);
    *launches += 1;
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_attn_mode(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    if (p.d == 64) return launch_attn_impl<MODE, 64>(p, s, launches);
    return launch_attn_impl<MODE, 128>(p, s, launches);
}

}  // namespace focus
