// Bounded waits on mbarriers shared by the tensor-core kernels, and small
// tensor-memory / store helpers. Every wait gives up after `limit` ns or once
// another role has aborted, so no kernel can spin forever; a role that gives
// up sets the abort flag that the others watch.
#pragma once

#include <cstdint>

#include "tc_common.cuh"

namespace gdn {

constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait

using ptx::globaltimer_ns;
using ptx::mbar_test_wait;
using ptx::mbar_try_wait;
using ptx::mbar_try_wait_cluster;
using ptx::tmem_ld16;
using ptx::tmem_wait_ld;

// Bounded wait: false if another role aborted or the limit passed (then aborts).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                         uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// wait_bar for a barrier completed by other CTAs of the cluster (acquire at
// cluster scope).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity,
                                                 volatile uint32_t *abort, uint64_t limit) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
    return true;
}
// Polling variant for the latency-critical roles: a suspended waiter can take
// hundreds of cycles to resume after the phase completes.
__device__ __forceinline__ bool spin_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                         uint64_t limit) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                *abort = 1;
                return false;
            }
        }
    }
}
// Polling with a pause between polls, for roles of several warps: a tight
// mbarrier poll from every warp of a group takes issue slots and shared-memory
// bandwidth from the warps doing the work (and from the tensor core's operand
// reads); a pause of ~ns bounds the added latency to about that.
__device__ __forceinline__ bool nap_bar(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                        uint64_t limit, uint32_t ns) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(ns);
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit) {
                *abort = 1;
                return false;
            }
        }
    }
}
constexpr uint32_t kNapNs = 32;
// A warp leaves its loop together: the tcgen05 loads that follow a wait are
// warp-collective.
__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }
__device__ __forceinline__ void store_bf16x8_global(void *dst, const float *v) {
    uint4 u = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                         pack_bf16(v[6], v[7]));
    *reinterpret_cast<uint4 *>(dst) = u;
}
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}


}  // namespace gdn
