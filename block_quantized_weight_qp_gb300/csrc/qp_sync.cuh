// qp_sync.cuh — bounded waits on mbarriers and the stop protocol shared by
// the warp-specialized kernels (the prefill GEMM, the standalone dequant).
//
// Every wait is bounded by a time limit.  The first role whose wait runs out
// latches an error bit in the device error word and raises the CTA's stop
// flag; the other roles give up at their next poll.  Before shared memory and
// tensor memory are released, each role waits (again with a bound, but
// regardless of the stop flag) for the asynchronous work it issued itself:
// copies into shared memory, MMAs into TMEM.
#pragma once
#include <cstdint>

#include "qp_ptx.cuh"

namespace qp {

// How a CTA's roles stop together: `flag` (in this CTA's shared memory) is
// raised by the first role whose wait runs out, and every other wait gives up
// once it sees it.  In a CTA pair the raise is also stored into the partner's
// flag (`peer`: its shared::cluster address; 0 for a lone CTA), so that the
// partner's roles stop at their next poll rather than at their own limit.
struct Stop {
    volatile uint32_t *flag;
    uint32_t peer;
    __device__ __forceinline__ bool raised() const { return *flag != 0u; }
    __device__ __forceinline__ void raise(uint32_t *err, uint32_t errbit) const {
        *flag = 1u;
        if (peer) st_shared_cluster_u32(peer, 1u);
        atomicOr(err, errbit);
    }
};

// Bounded wait on a barrier phase.  Returns false (and stops every role of
// this CTA) when the limit passes or another role already gave up.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, uint64_t limit_ns, const Stop &stop,
                                           uint32_t *err, uint32_t errbit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0) {
            if (stop.raised()) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                stop.raise(err, errbit);
                return false;
            }
        }
    }
}

// The same for waits that are not on the critical path (the epilogue waiting
// for a whole tile's mainloop, the producer running ahead of the MMA): back
// off with nanosleep between polls so the waiting warp does not take issue
// slots from the decode warps sharing its SM sub-partition.
__device__ __forceinline__ bool wait_phase_sleepy(uint64_t *bar, uint32_t parity, uint32_t max_sleep_ns,
                                                  uint64_t limit_ns, const Stop &stop, uint32_t *err,
                                                  uint32_t errbit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t sleep_ns = 32;
    for (;;) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (stop.raised()) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            stop.raise(err, errbit);
            return false;
        }
        if (sleep_ns < max_sleep_ns) sleep_ns <<= 1;
    }
}

// Warp-uniform form for roles whose every lane reads the guarded data.
__device__ __forceinline__ bool wait_phase_warp(uint64_t *bar, uint32_t parity, uint64_t limit_ns, const Stop &stop,
                                                uint32_t *err, uint32_t errbit) {
    const bool ok = wait_phase(bar, parity, limit_ns, stop, err, errbit);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait for work this thread issued itself (copies into shared
// memory, the tensor cores' MMAs into TMEM) to complete before the memory it
// writes is released.  Unlike wait_phase it does not give up when the CTA
// stops, only at the time limit.
__device__ __forceinline__ bool wait_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(64);
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// After a producer stops: waits until every copy it issued into the n
// stages of a ring has landed.  `armed` = the ring's arms so far, made in ring
// order from stage 0 (each arm is followed by its copy, except arm `skip`,
// whose copy the stall test hook left out).  Stage s was last armed for its
// phase uses - 1, the latest phase its barrier can reach.
__device__ __forceinline__ bool drain_ring(uint64_t *full, int n, int armed, int skip, uint64_t limit_ns) {
    bool ok = true;
    for (int s = 0; s < n && s < armed; ++s) {
        const int uses = armed / n + (s < armed % n ? 1 : 0);
        if (s + (uses - 1) * n == skip) continue;
        if (!wait_drain(&full[s], static_cast<uint32_t>((uses - 1) & 1), limit_ns)) ok = false;
    }
    return ok;
}

// Fallback before shared memory and TMEM are released: a fixed pause, for
// copies whose completion this CTA cannot observe or whose drain ran out.
__device__ __forceinline__ void pause_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

__device__ __forceinline__ void advance(int &stage, uint32_t &phase, int n) {
    if (++stage == n) {
        stage = 0;
        phase ^= 1u;
    }
}

}  // namespace qp
