// Inline-PTX wrappers for mbarriers and TMA bulk tensor copies (sm_90+ PTX,
// used here on sm_103a), with bounded waits.
//
// Every wait on an mbarrier is bounded in time.  Past kWaitTimeoutNs, the
// waiting thread ORs APSP_DEVICE_ERR_TIMEOUT into the device error word and
// returns false, and the kernel unwinds.  The host reports that as
// APSP_ETIMEOUT.  A thread that sees the error word already set stops
// waiting too, so one timeout ends the whole grid promptly.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; nothing is linked from libcuda)
#include <cstdint>

namespace apsp {

constexpr int kDeviceErrTimeout = 1;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // default: 2 s; a normal wait takes microseconds

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make the initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (after recording a timeout, unless another thread already recorded an
// error) if that does not happen within timeout_ns.  With watch_err = false
// the error word is not consulted (used while draining).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* err,
                                                  unsigned long long timeout_ns,
                                                  bool watch_err = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (watch_err && *reinterpret_cast<volatile int*>(err) != 0) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                atomicOr(err, kDeviceErrTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes
// on `bar`.  x is the innermost (column) coordinate; callers keep x * 4 a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 2-D tiled bulk tensor reduction shared -> global: every in-bounds element
// of the box becomes min(global, shared), performed in L2, with the element
// type of the tensor map (INT32 maps: signed 32-bit minimum).  Elements of
// the box outside the tensor are not written.  Tracked by the issuing
// thread's bulk async-groups.
__device__ __forceinline__ void tma_reduce_min_2d(const CUtensorMap* tm, int x, int y, uint32_t src) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.min.tile.bulk_group"
        " [%0, {%1, %2}], [%3];" ::"l"(reinterpret_cast<uint64_t>(tm)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// The shared-memory sources of every committed bulk group have been read.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Every committed bulk group has completed (its global writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace apsp
