/*
 * MEASUREMENT TOOLING, not part of libapsp's solving interface: a separate
 * library (libapsp_peak.so) that the benchmark loads for its roofline
 * denominators.  No solve entry point depends on it.
 *
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
 *   variant 5: int32, adds as multiply-add by an opaque 1, three-input
 *              integer min
 *   variant 6: int32 adds, fp32 three-input min over the (non-negative)
 *              bit patterns
 *   variant 7: int32 adds as multiply-add, fp32 three-input min over the
 *              bit patterns
 * Variants 0-7 keep their operands in registers.  The compiler may treat
 * those operands as loop-invariant and move the additions out of the loop.
 * Variants 1 and 3-7 then measure the minimum alone, and only variant 0
 * (fused add-min) measures the whole step.
 * Variants 8-13 run the library's own tile-product inner loop (mm_core.cuh)
 * on a 32-deep slab resident in shared memory, so they measure the real
 * step, loads included ( `threads` is ignored: 256 per block):
 *   variant 8 / 11:  int32 / fp32 fused core (one k per step)
 *   variant 9 / 12:  int32 / fp32 min3 core (two adds + three-input min)
 *   variant 10 / 13: int32 / fp32 packed core (one packed add + three-input
 *                    min, k-pair interleaved operands)
 *   variant 14 / 15: the int32 fused / fp32 packed core compiled for two
 *                    resident blocks per SM (at most 128 registers)
 *   variant 16 / 17: int32 mixed core, 2 / 3 of 8 accumulator rows on the
 *                    fused add-min, the rest on adds + three-input min
 *   variant 18 / 19 / 20: the same with 2 / 3 / 4 fused rows, the adds
 *                    written as multiply-adds by an opaque 1 (FMA pipe)
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

/*
 * apsp_peak_l2_read -- read bandwidth of the L2 cache: a buffer of `bytes`
 * (16 B .. 256 MiB; choose it well inside the L2) is read once to bring it
 * into L2, then `passes` more times with 16-byte loads that bypass L1, by
 * `blocks` x `threads` threads in a grid-stride loop.  This is the
 * denominator of the sparse searches' roofline, whose arc stream is served
 * from L2.
 *   gbs  bytes read per second / 1e9 over the timed passes (CUDA events).
 *   ms   time of the timed passes.
 * Returns 0, -1 on a bad argument, or a cudaError_t value (> 0).
 * Allocates and frees its buffer; synchronises the device.
 */
int apsp_peak_l2_read(long long bytes, int blocks, int threads, int passes, double* gbs, double* ms);

#ifdef __cplusplus
}
#endif

#endif
