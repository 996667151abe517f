// Host-side launcher shared by the attention translation units.
#pragma once

#include "focus_attn_kernel.cuh"
#include "focus_internal.h"

namespace focus {

template <int D>
uint32_t attn_smem_bytes(int mode, int K)
{
    return mode == kDense ? AttnSmem<D>::bytes(0) : AttnSmem<D>::bytes(K);
}

// The launch attributes of one kernel instance for K groups: its dynamic
// shared memory, and a check that the warpgroups' register shares after
// setmaxnreg fit in what the block is launched with (otherwise the increase
// would wait forever).  Enqueues nothing.
template <int MODE, int D>
cudaError_t attn_preflight_impl(int K)
{
    auto kern = focus_attn_kernel<MODE, D>;
    const uint32_t smem = attn_smem_bytes<D>(MODE, K);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if ((int64_t)fa.numRegs * kThreads < 256 * kRegsSoftmax + 128 * kRegsOther)
        return cudaErrorInvalidConfiguration;
    return cudaSuccess;
}

template <int MODE>
cudaError_t attn_preflight_mode(int d, int K)
{
    return d == 64 ? attn_preflight_impl<MODE, 64>(K) : attn_preflight_impl<MODE, 128>(K);
}

template <int MODE, int D>
cudaError_t launch_attn_impl(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    if (p.grid <= 0) return cudaSuccess;
    auto kern = focus_attn_kernel<MODE, D>;
    const uint32_t smem = attn_smem_bytes<D>(MODE, p.K);
    cudaError_t e = attn_preflight_impl<MODE, D>(p.K);
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
    a.pair_heads = p.pair_heads;
    a.gids = p.gids;
    a.offsets = p.offsets;
    a.pos = p.pos;
    a.tiles = p.tiles;
    a.ntiles = p.ntiles;
    a.q = p.q;
    a.masks = p.masks;
    a.mask_tiles = p.mask_tiles;
    a.wlo = p.wlo;
    a.work = p.work;
    a.out = p.out;
    a.lse = p.lse;
    a.part_out16 = p.part_out16;
    a.part_meta_out = p.part_meta_out;
    a.win_out16 = p.win_out16;
    a.win_meta_out = p.win_meta_out;
    a.status = p.wc.status;   // the attention kernels' waits use the fixed limit
    a.pair_count = p.pair_count;
    a.trace = trace_buffer(MODE);
    // Persistent: at most one CTA per SM; p.grid bounds the number of work items.
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int64_t grid = p.grid < sms ? p.grid : sms;
    prof_begin(MODE == kGroup ? "attn_group" : MODE == kWindow ? "attn_window" : "attn_dense", s);
    e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, *p.tmQ, *p.tmK, *p.tmV, a);
    prof_end(s);
    *launches += 1;
    return e;
}

template <int MODE>
cudaError_t launch_attn_mode(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    if (p.d == 64) return launch_attn_impl<MODE, 64>(p, s, launches);
    return launch_attn_impl<MODE, 128>(p, s, launches);
}

}  // namespace focus
