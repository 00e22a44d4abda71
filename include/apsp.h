/*
 * libapsp -- all-pairs shortest paths by blocked Floyd-Warshall on one GPU
 * (GB300, sm_103a).
 *
 * The operation (thesis page on Katz & Kider's blocked Floyd-Warshall,
 * 1library.co excerpt, section 4.6 and Algorithms 16-18): the input is a
 * weighted directed graph stored as a dense n x n distance matrix D.
 * D[i][j] holds the weight of arc i->j, INF means "no arc", and the diagonal
 * is 0.  The matrix is cut into B x B tiles and processed in n/B rounds.  In
 * round r the primary tile is K = [rB, (r+1)B):
 *   phase 1 closes the primary tile: D[K,K] gets its own Floyd-Warshall
 *           closure;
 *   phase 2 updates the row panel D[K,J] and the column panel D[I,K] of that
 *           tile (J, I != K);
 *   phase 3 applies D[i][j] = min(D[i][j], D[i][k] + D[k][j]) for k in K to
 *           every remaining tile (I,J), I != K and J != K.
 * Phase 3 carries the O(n^3) work.  After the last round D[i][j] is the
 * least total weight of a directed path from i to j, or INF if j cannot be
 * reached from i.  Tiling and reordering change no value (the "Loops into
 * zones" page, closing paragraph), so int32 results are exact.
 *
 * Layout: D is row-major with leading dimension ld >= n (elements).  Entry
 * (i, j) lives at dist[i * ld + j].  Columns n .. ld-1 are never read or
 * written.
 *
 * Value encoding:
 *   int32: INF = APSP_INF_I32 = 0x3FFFFFFF.  An input entry >= INF is read
 *          as INF.  A path whose length reaches INF cannot be represented and
 *          reads as INF.  Because INF + INF < 2^31, no sum overflows.
 *   fp32:  INF = +infinity; additions are IEEE round-to-nearest.
 *
 * Preconditions (not checked by apsp_solve*, see apsp_validate_*):
 *   D[i][i] = 0 and every weight >= 0; for fp32 also no NaN.  Negative
 *   weights are outside this library's contract.
 *
 * Ownership: the caller allocates and frees `dist`.  The library keeps a
 * small per-device workspace (two B x n panels plus two B x B tiles, where
 * B = 128) that it allocates on first use, grows when a larger n arrives, and
 * frees in apsp_release().
 *
 * Asynchrony: apsp_solve* enqueue kernels on `stream` and return without
 * waiting.  An argument error returns at once.  A launch error returns
 * APSP_ECUDA at once.  A fault during execution shows up on the next call
 * that synchronises, such as apsp_stream_check().  Solves on one device are
 * ordered one after another on the GPU, because they share the workspace.
 *
 * Thread safety: every entry point may be called from any host thread.
 */
#ifndef APSP_H
#define APSP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* apsp_stream_t;

typedef enum {
    APSP_OK = 0,
    APSP_EINVAL = 1,        /* bad argument: NULL with n > 0, n < 0, ld < n, n > APSP_MAX_N */
    APSP_ECUDA = 2,         /* CUDA runtime/launch error; see apsp_last_cuda_error() */
    APSP_ETIMEOUT = 3,      /* a bounded device-side wait ran out */
    APSP_EUNSUPPORTED = 4,  /* current device is not compute capability 10.3 (sm_103a) */
    APSP_ENOMEM = 5,        /* workspace or staging allocation failed */
    APSP_ENEGCYCLE = 6      /* the graph has a negative cycle (sparse entry points, apsp_sparse.h) */
} apsp_status_t;

#define APSP_INF_I32 0x3FFFFFFF
#define APSP_TILE 128       /* B: round block and CTA tile edge */
#define APSP_MAX_N 262144   /* largest n accepted (a 256 GiB int32 matrix) */

/*
 * apsp_solve / apsp_solve_i32 -- in-place APSP on an int32 device matrix.
 *   dist   device pointer to the n x n matrix (row-major, leading dim ld).
 *          16-byte alignment with ld % 4 == 0 takes the vectorised path;
 *          any other alignment still works, but more slowly.
 *   n      number of vertices, 0 <= n <= APSP_MAX_N (n = 0: no-op, APSP_OK).
 *   ld     leading dimension in elements, ld >= max(n, 1).
 *   stream CUDA stream to enqueue on.
 * Returns APSP_OK once the work is enqueued.
 */
apsp_status_t apsp_solve(int32_t* dist, int n, int ld, apsp_stream_t stream);
apsp_status_t apsp_solve_i32(int32_t* dist, int n, int ld, apsp_stream_t stream);

/* apsp_solve_f32 -- the same for an fp32 device matrix (INF = +inf). */
apsp_status_t apsp_solve_f32(float* dist, int n, int ld, apsp_stream_t stream);

/*
 * apsp_solve_host_i32 / _f32 -- the end-to-end call for callers that hold
 * the matrix in HOST memory.  It copies the matrix to the device (into a
 * library-owned staging buffer), solves, copies the result back in place and
 * waits for completion.  Pinned host memory gives full copy bandwidth.  It
 * uses the current device and the given stream.
 *   host   host pointer to the n x n matrix (leading dimension ld).
 * Returns APSP_OK when the result is back in host memory.
 */
apsp_status_t apsp_solve_host_i32(int32_t* host, int n, int ld, apsp_stream_t stream);
apsp_status_t apsp_solve_host_f32(float* host, int n, int ld, apsp_stream_t stream);

/*
 * apsp_solve_host_batch_i32 / _f32 -- `count` independent n x n problems
 * held in HOST memory, solved one after another with their copies
 * overlapped.  Matrix b is uploaded from in[b] into one of two
 * library-owned staging buffers on a library-owned copy stream, solved on
 * `stream`, and its result is downloaded into out[b].  The upload of matrix
 * b + 1 and the download of matrix b - 1 run while matrix b is solved, so
 * with pinned host memory a batch takes about count solves plus one upload
 * and one download.  The call returns when every result is in host memory.
 *   in     host array of `count` pointers to the input matrices (leading
 *          dimension ld).  Pointers may repeat: each input is only read.
 *   out    host array of `count` pointers to the result matrices (leading
 *          dimension ld).  out[b] may equal in[b] (in place).  It must not
 *          overlap any other in[] or out[] matrix.
 *   count  number of problems, >= 0 (0: no-op, APSP_OK).
 *   n, ld  as for apsp_solve; the same for every problem.
 * Ownership: the caller keeps every host buffer; the library keeps the
 * staging buffers, the copy stream and its events until apsp_release().
 * Errors: APSP_EINVAL for count < 0, a bad n or ld, or a NULL pointer among
 * in[0..count) and out[0..count) (checked before any work); APSP_ECUDA for a
 * failed copy or launch; APSP_ENOMEM when a staging buffer cannot be
 * allocated.  After an error no further problem is started, and the call
 * still waits for the work already enqueued.  Device-side wait timeouts are
 * reported by apsp_stream_check(stream), as for apsp_solve.
 */
apsp_status_t apsp_solve_host_batch_i32(const int32_t* const* in, int32_t* const* out, int count, int n,
                                        int ld, apsp_stream_t stream);
apsp_status_t apsp_solve_host_batch_f32(const float* const* in, float* const* out, int count, int n, int ld,
                                        apsp_stream_t stream);

/*
 * apsp_validate_i32 / _f32 -- check the preconditions on the device.
 *   flags_dev  device pointer to one int.  The call ORs bits into it and does
 *              not clear it first:
 *              1 = non-zero diagonal entry, 2 = negative entry,
 *              4 = NaN (fp32 only).
 * Asynchronous on `stream`, like apsp_solve.
 */
apsp_status_t apsp_validate_i32(const int32_t* dist, int n, int ld, apsp_stream_t stream,
                                int* flags_dev);
apsp_status_t apsp_validate_f32(const float* dist, int n, int ld, apsp_stream_t stream,
                                int* flags_dev);

/*
 * apsp_stream_check -- wait for `stream` to finish, then report any CUDA
 * error from the work on it (APSP_ECUDA) or any device-side bounded-wait
 * timeout that a library kernel recorded (APSP_ETIMEOUT).
 */
apsp_status_t apsp_stream_check(apsp_stream_t stream);

/* CUDA error code (cudaError_t) of the last APSP_ECUDA seen by this thread. */
int apsp_last_cuda_error(void);

/* Static, human-readable name of a status code. */
const char* apsp_status_string(apsp_status_t status);

/* Library version as major * 10000 + minor * 100 + patch. */
int apsp_version(void);

/* Free every device's workspace and staging buffers.  The caller must make
 * sure that no solve is still running. */
apsp_status_t apsp_release(void);

/*
 * apsp_solve_noalloc -- the int32 solve of apsp_solve for callers that may
 * not allocate device memory.  The pages have no counterpart to this entry
 * point: it exists for callers whose GPU memory is owned by another
 * allocator (a framework's caching pool, or a process held to a fixed memory
 * budget), or that run where an allocation, which can synchronise the whole
 * device, is not allowed.
 *
 * It allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).  Its workspace is a fixed scratch array of
 * APSP_NOALLOC_SCRATCH_BYTES (about 8.1 MiB) in the library's device image.
 * Every GPU that loads the library holds that array until the process exits.
 *   dist, n, ld, stream  as for apsp_solve, with n <= APSP_NOALLOC_MAX_N.
 *                        A larger n returns APSP_EINVAL before any work.
 *   err_dev              optional device pointer to one int.  After the solve
 *                        (in stream order) it receives the device error
 *                        word: 0, or APSP's timeout flag if a bounded
 *                        device-side wait ran out (the result is then
 *                        undefined).  NULL skips the copy.  This is the only
 *                        way a timeout of this entry point is reported:
 *                        apsp_stream_check reads the default workspace's
 *                        error word, not the scratch array's.
 * Set-up: the first call with n >= 1 on each device does a one-time set-up
 * with that device current.  It looks up the scratch array's device address
 * (cudaGetSymbolAddress) and loads every kernel the call launches, setting
 * their shared-memory limits.  Under lazy module loading this is where the
 * driver maps the library's device image (the scratch array included), and
 * that mapping may allocate: make the first call at initialisation time,
 * with a small n, before memory runs short and before any stream capture.
 * Later calls allocate nothing.
 * Sharing: all calls share the one array, which keeps the last call's
 * contents; each call clears what must start at zero.  Calls whose work
 * overlaps on the GPU (on different streams, or from different host
 * threads without ordering) race on the array and give wrong results.  Order
 * them, e.g. on one stream.
 */
#define APSP_NOALLOC_MAX_N 8192
#define APSP_NOALLOC_SCRATCH_BYTES 8519936 /* 256 + (2*128*8192 + 2*128*128) * 4 */
apsp_status_t apsp_solve_noalloc(int32_t* dist, int n, int ld, apsp_stream_t stream, int* err_dev);

/*
 * Phase timing, for profiling.  While it is enabled, each solve records CUDA
 * events on its stream around every phase launch.  apsp_phase_timing_read
 * waits for those events and returns, per phase (index 0, 1, 2 = phase 1, 2,
 * 3), the total milliseconds and the number of launches since the last read.
 * It then clears the totals.  Events are recorded on the launching stream,
 * so their gaps are exactly the kernels' durations on that stream.
 */
apsp_status_t apsp_phase_timing_enable(int enable);
apsp_status_t apsp_phase_timing_read(double ms_out[3], long long launches_out[3]);

#ifdef __cplusplus
}
#endif

#endif /* APSP_H */
