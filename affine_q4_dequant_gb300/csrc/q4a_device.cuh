// q4a_device.cuh -- PTX wrappers shared by the kernels of libq4a.so: mbarriers, TMA tile
// loads, programmatic dependent launch, and the bounded wait with its device error word.
// Every translation unit that includes this header gets its own error word (the library is
// built without relocatable device code); each unit exposes a host reader for it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "q4a_internal.h"

namespace q4a {
namespace {

// Set to nonzero by a kernel of this translation unit that gave up a bounded wait.
__device__ uint32_t g_device_error;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: a waiting warp sleeps in hardware until the phase
// completes (or the hint elapses) instead of spinning and taking issue slots from the
// warps that compute.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: after kWaitLimitNs the thread records the failure in the device error
// word and in the CTA's abort flag, then carries on. Control flow never depends on
// shared-memory data, so a give-up can only produce garbage values, never a hang, a
// skipped barrier or an out-of-range address. The retry loop is out of line: every launch
// starts with a cold instruction cache, and inlining it at each wait site costs more
// fetch time than the call costs a thread that is waiting anyway.
__device__ __noinline__ void mbar_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 3) == 0) {
            if (*abort_flag) return;
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(&g_device_error, 1u);
                *abort_flag = 1u;
                return;
            }
        }
    }
}

// Waits for a phase that TMA copies complete, whatever the abort flag says: a CTA must not
// exit while its own copies may still write shared memory. Bounded like every other wait.
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 3) == 0 && global_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_device_error, 1u);
            return;
        }
    }
}

__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return;
    mbar_wait_slow(bar, parity, abort_flag);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* map, int x, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2}], [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: the kernel may start while the previous kernel of the
// stream is finishing; grid_dep_wait() returns once that kernel has completed and its
// memory is visible. Nothing a previous kernel may write is touched before it.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

}  // namespace
}  // namespace q4a
