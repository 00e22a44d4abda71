/*
 * libapsp out-of-core entry points -- blocked Floyd-Warshall on a matrix
 * that stays in host memory, for n whose n x n matrix does not fit (or is not
 * meant to be kept) in device memory.
 *
 * The operation is the one of apsp.h (same layout, INF encoding, value
 * rules and preconditions); only where the matrix lives differs.  The thesis
 * page (1library.co excerpt, section 4.7) names such a modification for
 * graphs of any size but its text is not on the page; the method here is
 * blocked Floyd-Warshall one level up.  Super-blocks of K x K (K a multiple
 * of 128), one super-round per diagonal super-block R:
 *   1. D[R,R] is closed on the GPU by the in-core solver;
 *   2. the row panel D[R,:] and the column panel D[:,R] become min-plus
 *      products with the closed block (kept on the device for the round);
 *   3. every other super-block D[I,J] <- min(D[I,J], D[I,R] (x) D[R,J]) is
 *      copied in, updated and copied back, through a ring of three device
 *      buffers so that copies overlap the products.
 * int32 results are identical to apsp_solve; fp32 results agree within the
 * same rounding tolerance (sums may associate differently).
 *
 * apsp_solve_ooc_i32 / _f32
 *   host          the matrix, row-major, leading dimension ld >= n.  Pinned
 *                 (page-locked) memory lets the copies overlap the products;
 *                 pageable memory works but serialises them.  Overwritten
 *                 with the distances.
 *   device_bytes  device memory the call may allocate for its buffers:
 *                 5 K^2 + 2 K npad elements (npad = n rounded up to K).
 *                 0: 70% of the currently free device memory.
 *   block         K; 0 picks the largest multiple of 128 up to 16384 (and
 *                 up to n rounded to 128) that fits device_bytes.  Otherwise a
 *                 positive multiple of 128.  With K >= n the whole matrix is
 *                 one super-block: one copy in, the in-core solve, one out.
 *   stream        work is issued on this stream and on two private streams;
 *                 the call returns when it is done (blocking).
 * Returns APSP_OK; APSP_EINVAL for bad arguments, a block that is not a
 * multiple of 128, or a budget too small for K = 128; APSP_ENOMEM when the
 * buffers cannot be allocated; APSP_ECUDA / APSP_ETIMEOUT as apsp_solve.
 *
 * apsp_ooc_block -- the K that apsp_solve_ooc_* would pick for n, a budget
 * in bytes and an element size (4); 0 if even K = 128 does not fit.  Host
 * arithmetic only.
 */
#ifndef APSP_OOC_H
#define APSP_OOC_H

#include <stdint.h>

#include "apsp.h"

#ifdef __cplusplus
extern "C" {
#endif

apsp_status_t apsp_solve_ooc_i32(int32_t* host, int n, int ld, unsigned long long device_bytes, int block,
                                 apsp_stream_t stream);
apsp_status_t apsp_solve_ooc_f32(float* host, int n, int ld, unsigned long long device_bytes, int block,
                                 apsp_stream_t stream);
int apsp_ooc_block(int n, unsigned long long device_bytes, int elem_bytes);

#ifdef __cplusplus
}
#endif

#endif /* APSP_OOC_H */
