/*
 * libapsp_peak -- microbenchmark of the relaxation step's issue rate on the
 * current GPU, which gives the compute roofline for the min-plus update
 * (phase 3 of blocked Floyd-Warshall).  No page prints this number; the
 * library measures it.
 *
 * A relaxation is one update acc = min(acc, a + b).  Each variant runs
 * `iters` iterations of an 8 x 8 register block of independent relaxations
 * per thread (the same shape as the phase-3 inner loop, but without shared
 * memory traffic), on `blocks` x `threads` threads.
 *
 *   variant 0: int32, fused add-min intrinsic (__viaddmin_s32)
 *   variant 1: int32, add then two-input min written separately
 *   variant 2: int32, two relaxations per three-input min (__vimin3_s32)
 *   variant 3: fp32, fminf(acc, a + b)
 *   variant 4: fp32, fminf(acc, fminf(a0 + b0, a1 + b1)), two per step
 *
 * Outputs (host pointers, any may be NULL):
 *   relax_per_clk_sm  relaxations per SM clock cycle per SM.  Cycles come
 *                     from clock64 inside the kernel, so the value does not
 *                     depend on the clock frequency.
 *   ms                kernel time from CUDA events.
 *   relax_total       relaxations performed.
 * Returns 0 on success, -1 on a bad argument, -2 when `blocks` exceeds what
 * the GPU can keep resident at once, or a cudaError_t value (> 0).
 * Synchronises the device.
 */
#ifndef APSP_PEAK_H
#define APSP_PEAK_H

#ifdef __cplusplus
extern "C" {
#endif

int apsp_peak_addmin(int variant, int blocks, int threads, int iters, double* relax_per_clk_sm,
                     double* ms, long long* relax_total);

/* Number of variants understood by apsp_peak_addmin. */
int apsp_peak_variants(void);

#ifdef __cplusplus
}
#endif

#endif
