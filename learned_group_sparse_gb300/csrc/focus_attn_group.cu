// Group-causal attention over each group's gathered members (kGroup mode).
#include "focus_attn_launch.cuh"

namespace focus {

cudaError_t launch_attn_group(const AttnLaunch &p, cudaStream_t s, int *launches)
{
    return launch_attn_mode<kGroup>(p, s, launches);
}

}  // namespace focus
