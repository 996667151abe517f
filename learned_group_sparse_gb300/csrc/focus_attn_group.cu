// Group-causal attention over each group's gathered members (kGroup mode).
#include "focus_attn_launch.cuh"

namespace focus {

cudaError_t launch_attn_group(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    return launch_attn_mode<kGroup>(p, s, launches);
}

cudaError_t attn_preflight(int d, int K)
{
    cudaError_t e = attn_preflight_mode<kGroup>(d, K);
    return e != cudaSuccess ? e : attn_window_preflight(d, K);
}

size_t attn_smem_needed(int d, int K)
{
    const uint32_t g = d == 64 ? attn_smem_bytes<64>(kGroup, K)
                               : attn_smem_bytes<128>(kGroup, K);
    const uint32_t w = d == 64 ? attn_smem_bytes<64>(kWindow, K)
                               : attn_smem_bytes<128>(kWindow, K);
    return g > w ? g : w;
}

}  // namespace focus
