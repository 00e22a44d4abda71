/*
 * libapsp test hooks.  These exist only to exercise failure detection; a
 * production caller never needs them.
 */
#ifndef APSP_DEBUG_H
#define APSP_DEBUG_H

#include "apsp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * apsp_debug_inject_phase3_timeout -- arm a one-shot fault for the next
 * solve that runs a persistent TMA kernel: the persistent phase 3 of the
 * three-kernel schedule, or the round-fused kernel.  In the first such launch
 * with k-slabs (the first phase-3 launch, or round 0's fused launch), CTA 0's
 * producer skips issuing its first k-slab.  The consumers' bounded
 * wait for that slab then runs out after `timeout_ns`: they record a timeout
 * in the device error word and leave, and the producer waits (also bounded)
 * for its copies still in flight before it leaves.  No fault, trap or
 * unbounded wait is involved.  The next apsp_stream_check() returns
 * APSP_ETIMEOUT and clears the word.  The matrix content after such a solve
 * is undefined.
 *   timeout_ns  1 .. 2e9 nanoseconds, the bound on each wait in that launch.
 * Returns APSP_EINVAL for an out-of-range timeout.
 */
apsp_status_t apsp_debug_inject_phase3_timeout(unsigned long long timeout_ns);

/*
 * apsp_debug_inject_grid_timeout -- arm a one-shot fault for the next
 * grid-wide search (apsp_sssp_i32 or apsp_sssp_graph_search): CTA 0 leaves
 * the cooperative launch before it reaches the first grid barrier.  The other
 * CTAs' bounded waits at that barrier run out after `timeout_ns`; they record
 * the timeout and leave, and the call returns APSP_ETIMEOUT.  dist is then
 * undefined.  No fault, trap or unbounded wait is involved, and the next
 * search on the same context is unaffected.
 *   timeout_ns  1 .. 2e9 nanoseconds.
 * Returns APSP_EINVAL for an out-of-range timeout.
 */
apsp_status_t apsp_debug_inject_grid_timeout(unsigned long long timeout_ns);

/*
 * apsp_debug_fail_next_allocations -- make the next `count` device buffer
 * allocations of the dense entry points (workspace and staging buffers) fail
 * on the host, as cudaMalloc does when the device is full: no memory is
 * requested, and the call that needed the buffer returns APSP_ENOMEM with
 * apsp_last_cuda_error() = cudaErrorMemoryAllocation.  Nothing is enqueued
 * for that call, and the next call allocates normally.
 *   count  0 .. 1000 (0 disarms the hook).
 * Returns APSP_EINVAL for an out-of-range count.
 */
apsp_status_t apsp_debug_fail_next_allocations(int count);

/*
 * apsp_debug_small_cluster_size -- the number of CTAs in the thread-block
 * cluster that solves small matrices (n <= 512) on the current device: 16,
 * or 8 where the device cannot place a 16-CTA cluster, or 0 where it can
 * place neither (those solves then take the round schedules).  For tests
 * and benchmarks.
 *   is_float  0: the int32 kernel, 1: the fp32 kernel.
 * Returns the size, or -1 if the device is unsupported or a CUDA call failed.
 */
int apsp_debug_small_cluster_size(int is_float);

#ifdef __cplusplus
}
#endif

#endif
