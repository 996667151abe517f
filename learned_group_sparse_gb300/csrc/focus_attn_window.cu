// Sliding-window attention that skips group-sharing pairs (kWindow mode) and
// plain causal attention (kDense mode, the comparison baseline).
#include "focus_attn_launch.cuh"

namespace focus {

cudaError_t launch_attn_window(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    return launch_attn_mode<kWindow>(p, s, launches);
}

cudaError_t attn_window_preflight(int d, int K)
{
    return attn_preflight_mode<kWindow>(d, K);
}

cudaError_t launch_attn_dense(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    return launch_attn_mode<kDense>(p, s, launches);
}

}  // namespace focus
