/*
 * libapsp sparse entry points -- Johnson's all-pairs shortest paths with
 * Delta-stepping single-source searches, on one GPU (GB300, sm_103a).
 *
 * The operations:
 *   Delta-stepping SSSP (Delta-stepping page, CEUR Vol-1662 comp2, the
 *   algorithm and its parallel description).  Vertices wait in buckets of
 *   width Delta by tentative distance.  The lowest non-empty bucket is
 *   emptied by relaxing the light arcs (w <= Delta) of its vertices again and
 *   again.  After that the heavy arcs (w > Delta) of every vertex removed
 *   from it are relaxed once.  Needs weights >= 0.  Any Delta > 0 gives the
 *   same distances; Delta only changes the amount of work.
 *
 *   Johnson's APSP (Johnson/Dijkstra page, CEUR Vol-1631, the extendGraph,
 *   BellmanFord, UpdateWeights and to() steps).  A virtual vertex s gets a
 *   0-weight arc to every vertex.  Bellman-Ford from s gives potentials h,
 *   or finds a negative cycle.  The weights become
 *   w'(u,v) = w(u,v) + h(u) - h(v) >= 0.  One SSSP runs from every vertex on
 *   w' (here Delta-stepping; the page uses Dijkstra, and the distances are
 *   the same).  The results map back as D(i,j) = D'(i,j) + h(j) - h(i).
 *   When no weight is negative, h = 0 and the Bellman-Ford step is skipped.
 *
 * Both compute the same matrix as apsp_solve (apsp.h) wherever both apply:
 * D[i][j] is the least total weight of a directed path i ~> j, INF
 * (APSP_INF_I32) when j cannot be reached from i, and 0 on the diagonal.
 * Unlike apsp_solve, arc weights may be negative here, provided there is no
 * negative cycle.
 *
 * Graph format, CSR in device memory:
 *   row_ptr  int64[n + 1], row_ptr[0] = 0, non-decreasing; the arcs leaving
 *            vertex u are row_ptr[u] .. row_ptr[u+1]-1.
 *   col_idx  int32[m], heads of the arcs, each in [0, n).
 *   w        int32[m], arc weights in (-INF, INF).
 * Self-loops and parallel arcs are allowed.  A self-loop never shortens a
 * path; a negative one is a negative cycle.
 *
 * A dense int32 matrix is read the same way as apsp_solve reads it.  Entry
 * (u, v) with u != v and a value < INF is an arc; a value >= INF means no
 * arc.  The diagonal is ignored.
 *
 * Value range (checked): every arc weight lies in (-INF, INF).  Every true
 * distance must lie above -INF; a graph that breaks this returns
 * APSP_EINVAL.  A distance at or above INF reads as INF, as in apsp_solve.
 *
 * Blocking: unlike apsp_solve, these calls wait for `stream` before they
 * return.  They read the arc count, and Bellman-Ford's round flags, on the
 * host.  Kernel faults therefore show up in the return value.
 *
 * Workspace: per-device buffers, grown on demand and freed by
 * apsp_sparse_release().  They hold the CSR built from a dense matrix, h,
 * w', and the arcs partitioned light-first against Delta.  The caller owns
 * every pointer passed in.
 *
 * Limits: n <= APSP_SPARSE_MAX_N.  Each search CTA keeps one source's
 * distances, a bitmap of queued vertices and the least queued distance per
 * bitmap word in shared memory, 4.25 bytes per vertex.
 *
 * Thread safety: any host thread may call these.  Sparse calls on one
 * process are serialised by a lock.
 */
#ifndef APSP_SPARSE_H
#define APSP_SPARSE_H

#include <stdint.h>

#include "apsp.h"

#ifdef __cplusplus
extern "C" {
#endif

#define APSP_SPARSE_MAX_N 32768

/*
 * apsp_solve_sparse_i32 -- in-place APSP on a dense int32 device matrix by
 * Johnson's method.  The same contract as apsp_solve (layout, ld, INF), but
 * weights may be negative.
 *   dist   device pointer, n x ld row-major, overwritten with the distances.
 *   delta  bucket width for the Delta-stepping searches; <= 0 picks one from
 *          the largest (reweighted) arc weight and the mean out-degree.
 * Returns APSP_OK, or:
 *   APSP_EINVAL       bad arguments, n > APSP_SPARSE_MAX_N, or the value
 *                     range is broken;
 *   APSP_ENEGCYCLE    a negative cycle, and dist is left unchanged;
 *   APSP_ENOMEM       the workspace could not be allocated;
 *   APSP_ECUDA        a CUDA error; see apsp_last_cuda_error();
 *   APSP_EUNSUPPORTED the device is not sm_103.
 */
apsp_status_t apsp_solve_sparse_i32(int32_t* dist, int n, int ld, int32_t delta,
                                    apsp_stream_t stream);

/*
 * apsp_johnson_csr_i32 -- Johnson's APSP on a CSR graph (format above).
 *   out    device pointer, n x ld row-major (ld >= n), written in full.
 * Status codes as for apsp_solve_sparse_i32.
 */
apsp_status_t apsp_johnson_csr_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w,
                                   int n, int32_t delta, int32_t* out, int ld, apsp_stream_t stream);

/*
 * apsp_sssp_delta_i32 -- Delta-stepping from each of nsrc sources on a CSR
 * graph with weights >= 0.  A negative weight returns APSP_EINVAL.
 *   sources  device int32[nsrc], each in [0, n).
 *   out      device pointer, nsrc x ldo row-major (ldo >= n).  Row q holds
 *            the distances from sources[q] (INF for unreachable).
 *   delta    as for apsp_solve_sparse_i32.
 */
apsp_status_t apsp_sssp_delta_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w,
                                  int n, const int32_t* sources, int nsrc, int32_t delta,
                                  int32_t* out, int ldo, apsp_stream_t stream);

/*
 * apsp_sssp_i32 -- one Delta-stepping search from `source` using the whole
 * GPU, for graphs of any size the device memory holds (the Delta-stepping
 * page's single-source setting; no shared-memory limit on n).  CSR as above,
 * weights >= 0 (a negative weight returns APSP_EINVAL), fewer than 2^31 arcs.
 *   dist   device int32[n], 16-byte aligned: the distances from source, INF
 *          for unreachable.  It also serves as the search's working array.
 *   delta  bucket width; <= 0 picks w_max / (2 * mean out-degree).  Past
 *          the search's peak (a bucket that selected n / 64 vertices or
 *          more) each bucket is twice as wide as the one before, up to about
 *          2 * w_max.  Neither delta nor the widening changes the distances.
 * The search is one cooperative launch whose CTAs meet at grid barriers.
 * Every barrier wait is bounded (2 s); one that runs out returns
 * APSP_ETIMEOUT, and dist is then undefined.  Workspace: about 8 bytes per
 * arc plus 5.25 bytes per vertex, kept per device like the rest.
 */
apsp_status_t apsp_sssp_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n, int source,
                            int32_t delta, int32_t* dist, apsp_stream_t stream);

/*
 * Prepared graphs for repeated single-source searches.  apsp_sssp_i32
 * checks and partitions the arcs (light first, against delta) on every call;
 * a prepared graph does that once, like building the CSR, and each search
 * then runs on it alone.
 *
 * apsp_sssp_graph_create -- check the CSR graph (as apsp_sssp_i32), choose
 *   delta (<= 0: the library's default), and build the graph's own device
 *   copy: row_ptr, the partitioned arcs and the search state.  The caller's
 *   arrays may be freed afterwards.  Blocks on `stream`.  *out receives the
 *   handle (NULL on failure).  Status codes as for apsp_sssp_i32.
 * apsp_sssp_graph_search -- one search from `source` into dist (device
 *   int32[n], 16-byte aligned), on the device the graph was created on (else
 *   APSP_EINVAL).  Blocks on `stream`.  Searches on one graph run one at a
 *   time.
 * apsp_sssp_graph_info -- n, m and the delta in use (any pointer may be NULL).
 * apsp_sssp_graph_destroy -- free the graph (NULL is a no-op).
 */
typedef struct apsp_sssp_graph* apsp_sssp_graph_t;

apsp_status_t apsp_sssp_graph_create(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n,
                                     int32_t delta, apsp_stream_t stream, apsp_sssp_graph_t* out);
apsp_status_t apsp_sssp_graph_search(apsp_sssp_graph_t graph, int source, int32_t* dist, apsp_stream_t stream);
apsp_status_t apsp_sssp_graph_info(apsp_sssp_graph_t graph, int* n, long long* m, int32_t* delta);
apsp_status_t apsp_sssp_graph_destroy(apsp_sssp_graph_t graph);

/*
 * apsp_csr_count_i32 / apsp_csr_fill_i32 -- build the CSR of a dense int32
 * device matrix, with the arcs as defined above.
 * count: writes row_ptr (device, int64[n + 1]), and the arc count m to
 *   *m_out (host).  Blocks on `stream`.
 * fill:  writes col_idx and w (device, m entries each), in increasing column
 *   order within a row, given the row_ptr from count.  Asynchronous on
 *   `stream`.
 */
apsp_status_t apsp_csr_count_i32(const int32_t* dist, int n, int ld, int64_t* row_ptr, long long* m_out,
                                 apsp_stream_t stream);
apsp_status_t apsp_csr_fill_i32(const int32_t* dist, int n, int ld, const int64_t* row_ptr,
                                int32_t* col_idx, int32_t* w, apsp_stream_t stream);

/* Free the sparse workspace on every device that has one. */
apsp_status_t apsp_sparse_release(void);

/*
 * apsp_sparse_timing_enable / _read -- measurement hooks for the bench.
 * While enabled, each search launch is bracketed by CUDA events on its
 * stream.  _read returns, and resets, the summed search-kernel time in ms,
 * the number of search launches, and the number of kernels the sparse entry
 * points launched (counted whether or not timing is enabled).  Any pointer
 * may be NULL.
 */
apsp_status_t apsp_sparse_timing_enable(int enable);
apsp_status_t apsp_sparse_timing_read(double* search_ms, long long* searches, long long* kernels);

#ifdef __cplusplus
}
#endif

#endif /* APSP_SPARSE_H */
