// Waits bounded by a launch's run-time limit (focus_set_wait_limit), for the
// kernels whose waits take it: the assignment, merge and decode kernels.
// (The attention kernels keep the constant limit of focus_ptx.cuh.)
#pragma once

#include "focus_ptx.cuh"

namespace focus {

// Non-blocking test of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with the limit of the launch's WaitCtl (focus_set_wait_limit),
// checked after every poll that finds the phase incomplete.  The device
// timer may tick in microseconds and a blocking poll may be suspended for
// longer than that, so a limit under a microsecond makes the wait poll
// without blocking and give up at its second unsuccessful poll: a tiny limit
// makes any wait that has to wait at all run out.  Used by the assignment,
// merge and decode kernels.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          const WaitCtl &w)
{
    if (w.limit_ns < 1000ull) {
        if (mbar_test_wait(bar, parity) || mbar_test_wait(bar, parity)) return true;
        *abort = 1;
        if (w.status) atomicExch(w.status, kDeviceTimeout);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *abort = 1;
            if (w.status) atomicExch(w.status, kDeviceTimeout);
            return false;
        }
        if ((it & 63u) == 0 && *abort) return false;
    }
}

}  // namespace focus
