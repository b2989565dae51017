// common.cuh -- the device error word and the bounded mbarrier wait shared by
// every kernel of the library.
#pragma once
#include "ptx.cuh"

namespace fp8bs {

// Per-device error word (one copy per device that loads the library).
// bit 0: a pipeline wait exceeded its time limit.  Read and cleared by
// fp8bs_last_error().
__device__ unsigned int g_error_word;

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s

// Wait for phase `parity` of barrier `bar`, giving up after `limit_ns` or
// as soon as *abort is set.  On time-out it sets *abort and the error word.
// Returns true when the phase completed.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t *abort,
                                             uint64_t limit_ns = WAIT_LIMIT_NS)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort)
                return false;
            if (ptx::globaltimer_ns() - t0 > limit_ns) {
                *abort = 1u;
                atomicOr(&g_error_word, 1u);
                return false;
            }
        }
    }
}

// Drain wait (no abort flag): used at exit for the kernel's own copies.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(&g_error_word, 1u);
            return;
        }
}

} // namespace fp8bs
