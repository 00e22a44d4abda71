// Sparse-graph shortest paths on sm_103a: Delta-stepping SSSP and Johnson's
// APSP.  The contract is in include/apsp_sparse.h.
//
// Delta-stepping (Delta-stepping page, CEUR Vol-1662 comp2): one CTA runs
// one source at a time.  Persistent CTAs take sources from a global counter.
// The tentative distances, the "queued" set (vertices waiting in some
// bucket), the set R (vertices removed from the current bucket) and the
// frontier list all live in shared memory.  The bucket of a queued vertex is
// dist / Delta, so no bucket arrays are kept.  The lowest non-empty bucket is
// found by a scan of the queued bitmap.  A phase takes that bucket's queued
// vertices as the frontier and relaxes their light arcs.  Vertices that
// improve are queued again, and phases repeat until the bucket stays empty.
// The heavy arcs of R are then relaxed once.  One warp walks one frontier
// vertex's arc list, so a hub of a scale-free graph spreads over 32 lanes.
// No step waits on another CTA: every loop ends because distances only
// decrease.
//
// Johnson (Johnson/Dijkstra page, CEUR Vol-1631): Bellman-Ford from the
// virtual vertex in int64, one launch per round, Gauss-Seidel style (a
// round may use values updated in the same round, which only speeds
// convergence).  It ends after a round that changes nothing; a change in
// round n + 1 means a negative cycle.  Then the reweighting
// w' = w + h(u) - h(v), the searches on w', and the mapping back in each
// search's epilogue.
//
// Arithmetic: distances in the search are int32 with INT_MAX as
// "unreached".  A relaxation adds in unsigned 32-bit arithmetic (both terms
// are below 2^31, so the sum cannot wrap) and saturates at INT_MAX.  With
// h > -INF, every reweighted distance of a pair whose true distance is below
// INF is below 2 * INF < INT_MAX.  So those come out exact, and the rest map
// to INF.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/apsp.h"
#include "../../include/apsp_debug.h"
#include "../../include/apsp_sparse.h"
#include "tma.cuh"

namespace apsp {
void set_last_cuda_error(int e);  // defined with apsp_last_cuda_error()
}

namespace {

constexpr int32_t kInf = APSP_INF_I32;
constexpr int32_t kUnreached = INT_MAX;
constexpr int kScanThreads = 1024;

apsp_status_t sp_fail(cudaError_t e) {
    apsp::set_last_cuda_error((int)e);
    return APSP_ECUDA;
}

bool sp_supported_device() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3;
}

// ------------------------------------------------------------------ CSR build

// Arcs per row (warp per row); row_ptr[row + 1] = count, row_ptr[0] = 0.
__global__ void csr_count_kernel(const int32_t* __restrict__ d, long long ld, int n,
                                 int64_t* __restrict__ rp) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int row = (int)wid;
    const int32_t* drow = d + (long long)row * ld;
    int cnt = 0;
    for (int j = lane; j < n; j += 32) cnt += (j != row && drow[j] < kInf) ? 1 : 0;
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
        rp[row + 1] = cnt;
        if (row == 0) rp[0] = 0;
    }
}

// In-place inclusive prefix sum of a[1..n] (a[0] = 0) by one CTA: each
// thread sums a contiguous chunk, the chunk sums are scanned in shared
// memory, and each thread rewrites its chunk.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(int64_t* __restrict__ a, int n) {
    __shared__ int64_t part[kScanThreads];
    const int t = threadIdx.x;
    const int chunk = (n + kScanThreads - 1) / kScanThreads;
    const int b = 1 + t * chunk, e = min(n + 1, b + chunk);
    int64_t s = 0;
    for (int i = b; i < e; ++i) s += a[i];
    part[t] = s;
    __syncthreads();
    for (int off = 1; off < kScanThreads; off <<= 1) {
        const int64_t v = t >= off ? part[t - off] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int64_t run = t > 0 ? part[t - 1] : 0;
    for (int i = b; i < e; ++i) {
        run += a[i];
        a[i] = run;
    }
}

// Column indices and weights of each row, in column order (warp per row;
// a ballot gives each arc its slot).
__global__ void csr_fill_kernel(const int32_t* __restrict__ d, long long ld, int n,
                                const int64_t* __restrict__ rp, int32_t* __restrict__ col,
                                int32_t* __restrict__ w) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int row = (int)wid;
    const int32_t* drow = d + (long long)row * ld;
    int64_t pos = rp[row];
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int j = j0 + lane;
        const int32_t v = j < n ? drow[j] : kInf;
        const bool arc = j < n && j != row && v < kInf;
        const unsigned mask = __ballot_sync(0xffffffffu, arc);
        if (arc) {
            const int64_t p = pos + __popc(mask & ((1u << lane) - 1u));
            col[p] = j;
            w[p] = v;
        }
        pos += __popc(mask);
    }
}

// min and max of w[0..m) into range[0], range[1], and whether any head
// col[e] lies outside [0, n) into range[2] (initialised INT_MAX, INT_MIN, 0).
__global__ void weight_range_kernel(const int32_t* __restrict__ w, const int32_t* __restrict__ col,
                                    long long m, int n, int* __restrict__ range) {
    int lo = INT_MAX, hi = INT_MIN;
    unsigned bad = 0;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < m;
         e += (long long)gridDim.x * blockDim.x) {
        lo = min(lo, w[e]);
        hi = max(hi, w[e]);
        if (col) bad |= (unsigned)col[e] >= (unsigned)n ? 1u : 0u;
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if ((threadIdx.x & 31) == 0) {
        atomicMin(range, lo);
        atomicMax(range + 1, hi);
        if (bad) atomicOr(range + 2, 1);
    }
}

// *bad = 1 unless row_ptr[0] = 0 and row_ptr is non-decreasing.
__global__ void rowptr_check_kernel(const int64_t* __restrict__ rp, int n, int* __restrict__ bad) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i > n) return;
    if (i == 0 ? rp[0] != 0 : rp[i] < rp[i - 1]) atomicOr(bad, 1);
}

// ------------------------------------------------------------------ Bellman-Ford

// One round over every arc against the potentials h (warp per tail vertex).
__global__ void bf_round_kernel(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                const int32_t* __restrict__ w, int n, long long* __restrict__ h,
                                int* __restrict__ changed) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int u = (int)wid;
    const long long hu = *reinterpret_cast<volatile long long*>(h + u);
    int any = 0;
    for (int64_t e = rp[u] + lane; e < rp[u + 1]; e += 32) {
        const int v = col[e];
        const long long nv = hu + w[e];
        if (nv < *reinterpret_cast<volatile long long*>(h + v) && nv < atomicMin(h + v, nv)) any = 1;
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) *changed = 1;
}

// w' = w + h(u) - h(v) (>= 0 once Bellman-Ford has converged).  flag gets 1
// when some h(u) <= -INF: a distance below the int32 range.
__global__ void reweight_kernel(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                const int32_t* __restrict__ w, int n, const long long* __restrict__ h,
                                int32_t* __restrict__ wh, int* __restrict__ flag) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int u = (int)wid;
    const long long hu = h[u];
    if (hu <= -(long long)kInf) {
        if (lane == 0) *flag = 1;
        return;
    }
    for (int64_t e = rp[u] + lane; e < rp[u + 1]; e += 32) {
        const long long hv = h[col[e]];
        // hv > -INF (checked by v's own warp), hu <= 0, w < INF: 0 <= w' < 2 * INF
        wh[e] = (int32_t)((long long)w[e] + hu - (hv > -(long long)kInf ? hv : 0));
    }
}

// ------------------------------------------------------------------ Delta-stepping

// Light-first partition of each vertex's arcs against delta, packed as
// (head, weight) pairs: arcs[rp[u] .. rp[u] + nlight[u]) are the light arcs
// (w <= delta) of u and the rest of its range the heavy ones, each part in
// CSR order.  partition_kernel takes a warp per vertex (two ballot passes);
// a vertex with more than kPartBig arcs is put on a list instead, for
// partition_big_kernel, which gives each such vertex a whole CTA.
constexpr int kPartBig = 8192;
constexpr int kPartBigThreads = 1024;

__global__ void partition_kernel(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                 const int32_t* __restrict__ w, int n, int32_t delta, int2* __restrict__ arcs,
                                 int32_t* __restrict__ nlight, int32_t* __restrict__ biglist,
                                 int* __restrict__ bigcount) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int u = (int)wid;
    const int64_t beg = rp[u], end = rp[u + 1];
    if (end - beg > kPartBig) {
        if (lane == 0) biglist[atomicAdd(bigcount, 1)] = u;
        return;
    }
    int nl = 0;
    for (int64_t e = beg + lane; e < end; e += 32) nl += w[e] <= delta ? 1 : 0;
    nl = __reduce_add_sync(0xffffffffu, nl);
    const unsigned lt = (1u << lane) - 1u;
    int64_t lpos = beg, hpos = beg + nl;
    for (int64_t e0 = beg; e0 < end; e0 += 32) {
        const int64_t e = e0 + lane;
        const bool valid = e < end;
        const int32_t c = valid ? col[e] : 0, ww = valid ? w[e] : 0;
        const bool light = valid && ww <= delta, heavy = valid && ww > delta;
        const unsigned ml = __ballot_sync(0xffffffffu, light), mh = __ballot_sync(0xffffffffu, heavy);
        if (light) arcs[lpos + __popc(ml & lt)] = make_int2(c, ww);
        if (heavy) arcs[hpos + __popc(mh & lt)] = make_int2(c, ww);
        lpos += __popc(ml);
        hpos += __popc(mh);
    }
    if (lane == 0) nlight[u] = nl;
}

// One CTA per listed vertex: the same stable light-first partition, the
// arcs taken 1024 at a time with CTA-wide ranks (warp ballots plus a scan of
// the 32 warps' counts).
__global__ void __launch_bounds__(kPartBigThreads)
partition_big_kernel(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                     const int32_t* __restrict__ w, int32_t delta, int2* __restrict__ arcs,
                     int32_t* __restrict__ nlight, const int32_t* __restrict__ biglist) {
    __shared__ int s_light[32], s_heavy[32], s_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = biglist[blockIdx.x];
    const int64_t beg = rp[u], end = rp[u + 1];
    int nl = 0;
    for (int64_t e = beg + tid; e < end; e += kPartBigThreads) nl += w[e] <= delta ? 1 : 0;
    nl = __reduce_add_sync(0xffffffffu, nl);
    if (tid == 0) s_total = 0;
    __syncthreads();
    if (lane == 0) atomicAdd(&s_total, nl);
    __syncthreads();
    const int64_t light_total = s_total;
    const unsigned lt = (1u << lane) - 1u;
    int64_t lpos = beg, hpos = beg + light_total;  // the same in every thread
    for (int64_t e0 = beg; e0 < end; e0 += kPartBigThreads) {
        const int64_t e = e0 + tid;
        const bool valid = e < end;
        const int32_t c = valid ? col[e] : 0, ww = valid ? w[e] : 0;
        const bool light = valid && ww <= delta, heavy = valid && ww > delta;
        const unsigned ml = __ballot_sync(0xffffffffu, light), mh = __ballot_sync(0xffffffffu, heavy);
        if (lane == 0) {
            s_light[warp] = __popc(ml);
            s_heavy[warp] = __popc(mh);
        }
        __syncthreads();
        int lb = 0, hb = 0, lsum = 0, hsum = 0;
        for (int x = 0; x < kPartBigThreads / 32; ++x) {
            if (x < warp) {
                lb += s_light[x];
                hb += s_heavy[x];
            }
            lsum += s_light[x];
            hsum += s_heavy[x];
        }
        if (light) arcs[lpos + lb + __popc(ml & lt)] = make_int2(c, ww);
        if (heavy) arcs[hpos + hb + __popc(mh & lt)] = make_int2(c, ww);
        lpos += lsum;
        hpos += hsum;
        __syncthreads();  // s_light / s_heavy are rewritten next
    }
    if (tid == 0) nlight[u] = (int32_t)light_total;
}

struct SpShared {
    int dmin[2];  // least queued distance, double-buffered by bucket parity
    int item;
};

// Shared memory of a search CTA: dist (int32, n), the queued bitmap, and
// per bitmap word the least distance of its queued vertices (wmin).
__host__ __device__ constexpr size_t sssp_shared_offset(int n) {
    return ((size_t)n * 4 + (size_t)((n + 31) / 32) * 8 + 15) / 16 * 16;
}

size_t sssp_smem_bytes(int n) { return sssp_shared_offset(n) + sizeof(SpShared); }

// Position of the k-th (0-based) set bit of x; x has more than k set bits.
__device__ __forceinline__ int kth_set_bit(uint32_t x, int k) {
    int pos = 0;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
        const int c = __popc(x & ((1u << s) - 1u));
        if (k >= c) {
            k -= c;
            x >>= s;
            pos += s;
        }
    }
    return pos;
}

// Largest lane j with key_j <= t, for keys non-decreasing across the warp
// and key_0 <= t.
__device__ __forceinline__ int last_lane_at_or_below(int key, int t) {
    int pos = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
        const int x = __shfl_sync(0xffffffffu, key, pos + step);
        if (x <= t) pos += step;
    }
    return pos;
}

// Relax the light (kLight) or heavy arcs of the warp's frontier.  Lane j
// holds in `bits` the frontier members of bitmap word j * kWarps + warp.
// A warp scan numbers the members 0 .. T-1 and they are taken 32 at a time,
// so every batch but the last is full: lane k finds the word and the bit of
// member b + k, loads that vertex's arc range, a second warp scan lays the
// ranges of at most 64 arcs end to end, and the lanes walk the concatenation
// in chunks of 32 arcs, up to kUnroll chunks with their loads in flight
// together; a longer range is then walked by the whole warp alone, so that
// no lane binary-searches the scan for its arcs.  Measured (Johnson, all
// sources) against laying every range end to end: BA n = 16384: 17.30 ->
// 17.03 ms; ER n = 2048, degree 100: 1.06 -> 0.87 ms; ER n = 8192, degree
// 4096: 397 -> 222 ms.  Returns this lane's least distance among its
// successful relaxations (INT_MAX if none).
template <bool kLight, int kWarps, int kUnroll>
__device__ __forceinline__ int32_t expand(uint32_t bits, const int64_t* __restrict__ rp,
                                          const int32_t* __restrict__ nlight, const int2* __restrict__ arcs,
                                          int32_t* dist, uint32_t* queued, int32_t* wmin, int warp, int lane) {
    int32_t best = INT_MAX;
    const int c = __popc(bits);
    int wincl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += y;
    }
    const int members = __shfl_sync(0xffffffffu, wincl, 31);
    const int wexcl = wincl - c;
    for (int b0 = 0; b0 < members; b0 += 32) {
        const int g = b0 + lane;
        const int j = last_lane_at_or_below(wexcl, g);
        const uint32_t wbits = __shfl_sync(0xffffffffu, bits, j);
        const int wstart = __shfl_sync(0xffffffffu, wexcl, j);
        int beg = 0, cnt = 0;
        uint32_t dv = 0;
        if (g < members) {
            const int v = (j * kWarps + warp) * 32 + kth_set_bit(wbits, g - wstart);
            const int r0 = (int)rp[v], nl = nlight[v];
            if (kLight) {
                beg = r0;
                cnt = nl;
            } else {
                beg = r0 + nl;
                cnt = (int)rp[v + 1] - r0 - nl;
            }
            dv = (uint32_t)dist[v];
        }
        // Vertices of more than kWarpArcs arcs are walked by the whole warp,
        // one at a time (below); the others' arc ranges are laid end to end.
        constexpr int kWarpArcs = 64;
        const int lcnt = cnt <= kWarpArcs ? cnt : 0;
        int incl = lcnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        const int excl = incl - lcnt;
        for (int base = 0; base < total; base += 32 * kUnroll) {
            int2 a[kUnroll];
            uint32_t d[kUnroll];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int t = base + q * 32 + lane;
                const int pos = last_lane_at_or_below(excl, t);
                const int e = __shfl_sync(0xffffffffu, beg, pos) + t - __shfl_sync(0xffffffffu, excl, pos);
                d[q] = __shfl_sync(0xffffffffu, dv, pos);
                a[q] = t < total ? arcs[e] : make_int2(0, -1);
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                if (a[q].y < 0) continue;  // past the end (weights here are >= 0)
                const uint32_t s = d[q] + (uint32_t)a[q].y;  // < 2^32: both terms < 2^31
                const int32_t nd = s >= (uint32_t)kUnreached ? kUnreached : (int32_t)s;
                const int u = a[q].x;
                if (nd < dist[u] && nd < atomicMin(dist + u, nd)) {
                    atomicOr(queued + (u >> 5), 1u << (u & 31));
                    atomicMin(wmin + (u >> 5), nd);
                    best = min(best, nd);
                }
            }
        }
        for (uint32_t hm = __ballot_sync(0xffffffffu, cnt > kWarpArcs); hm; hm &= hm - 1) {
            const int src = __ffs(hm) - 1;
            const int hb = __shfl_sync(0xffffffffu, beg, src);
            const int hc = __shfl_sync(0xffffffffu, cnt, src);
            const uint32_t hd = __shfl_sync(0xffffffffu, dv, src);
            for (int t0 = 0; t0 < hc; t0 += 32 * kUnroll) {
                int2 a[kUnroll];
#pragma unroll
                for (int q = 0; q < kUnroll; ++q) {
                    const int t = t0 + q * 32 + lane;
                    a[q] = t < hc ? arcs[hb + t] : make_int2(0, -1);
                }
#pragma unroll
                for (int q = 0; q < kUnroll; ++q) {
                    if (a[q].y < 0) continue;
                    const uint32_t sum = hd + (uint32_t)a[q].y;
                    const int32_t nd = sum >= (uint32_t)kUnreached ? kUnreached : (int32_t)sum;
                    const int u = a[q].x;
                    if (nd < dist[u] && nd < atomicMin(dist + u, nd)) {
                        atomicOr(queued + (u >> 5), 1u << (u & 31));
                        atomicMin(wmin + (u >> 5), nd);
                        best = min(best, nd);
                    }
                }
            }
        }
    }
    return best;
}

// Row `item` of out gets the distances from source sources[item] (or item
// when sources is null).  With h non-null the search ran on reweighted arcs
// and the epilogue maps back: out = dist + h[v] - h[src].  A source outside
// [0, n) sets bit 0 of *err and its row is skipped.
//
// Lane j of warp w owns bitmap word j * kWarps + w (n <= 1024 * kWarps):
// it selects that word's queued vertices into its frontier register F and
// accumulates R (removed from the current bucket) in another register.  The
// word's least queued distance (wmin, kept current by the relaxations with
// an atomic min) lets a selection skip every word with nothing in the
// bucket without reading its distances.
// Per bucket: light phases (select the queued vertices below the bucket's
// upper end hi, relax their light arcs) until a selection comes back empty;
// that last selection also yields the least queued distance at or above hi.
// Then the heavy arcs of R; their successful relaxations, with that least
// distance, give the next bucket.
template <int kThreads, int kMinBlocks = 1536 / kThreads>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
sssp_delta_kernel(const int64_t* __restrict__ rp, const int32_t* __restrict__ nlight,
                  const int2* __restrict__ arcs, int n, const int32_t* __restrict__ sources, int nsrc,
                  int32_t delta, const long long* __restrict__ h, int32_t* __restrict__ out, long long ldo,
                  int* __restrict__ counter, int* __restrict__ err) {
    constexpr int kWarps = kThreads / 32;
    constexpr int kUnroll = 4;
    extern __shared__ __align__(16) unsigned char sp_smem[];
    const int nw = (n + 31) / 32;
    int32_t* dist = reinterpret_cast<int32_t*>(sp_smem);
    uint32_t* queued = reinterpret_cast<uint32_t*>(dist + n);    // waiting in some bucket
    int32_t* wmin = reinterpret_cast<int32_t*>(queued + nw);     // least queued distance per word
    SpShared* sh = reinterpret_cast<SpShared*>(sp_smem + sssp_shared_offset(n));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int myword = lane * kWarps + warp;
    const bool owns = myword < nw;

    for (;;) {
        if (tid == 0) sh->item = atomicAdd(counter, 1);
        __syncthreads();
        const int item = sh->item;
        __syncthreads();  // everyone has read sh->item before thread 0 may rewrite it
        if (item >= nsrc) return;
        const int src = sources ? sources[item] : item;
        if (src < 0 || src >= n) {
            if (tid == 0) atomicOr(err, 1);
            continue;
        }
        for (int v = tid; v < n; v += kThreads) dist[v] = kUnreached;
        for (int i = tid; i < nw; i += kThreads) {
            queued[i] = 0u;
            wmin[i] = INT_MAX;
        }
        if (tid == 0) {
            sh->dmin[0] = INT_MAX;
            sh->dmin[1] = INT_MAX;
        }
        __syncthreads();
        if (tid == 0) {
            dist[src] = 0;
            queued[src >> 5] = 1u << (src & 31);
            wmin[src >> 5] = 0;
        }
        __syncthreads();

        int32_t dmin = 0;  // least queued distance: the current bucket is [.., hi)
        for (int bucket = 0;; ++bucket) {
            const long long hi_ll = ((long long)(dmin / delta) + 1) * delta;
            const int32_t hi = hi_ll >= kUnreached ? kUnreached : (int32_t)hi_ll;
            uint32_t rbits = 0u;  // R, this lane's word
            int32_t beyond;       // least queued distance >= hi seen by the last selection
            for (;;) {
                beyond = INT_MAX;
                uint32_t fbits = 0u;
                if (owns) {
                    const int32_t wm = wmin[myword];
                    if (wm < hi) {  // else nothing of this word is in the bucket: skip its bits
                        uint32_t bits = queued[myword];
                        const uint32_t all = bits;
                        while (bits) {
                            const int b = __ffs(bits) - 1;
                            bits &= bits - 1;
                            const int32_t dd = dist[myword * 32 + b];
                            if (dd < hi)
                                fbits |= 1u << b;
                            else
                                beyond = min(beyond, dd);
                        }
                        queued[myword] = all & ~fbits;
                        wmin[myword] = beyond;
                        rbits |= fbits;
                    } else {
                        beyond = wm;
                    }
                }
                if (!__syncthreads_or(fbits != 0u)) break;
                expand<true, kWarps, kUnroll>(fbits, rp, nlight, arcs, dist, queued, wmin, warp, lane);
                __syncthreads();
            }
            // heavy arcs of R, once; then the next bucket from the least queued distance
            const int32_t hbest =
                expand<false, kWarps, kUnroll>(rbits, rp, nlight, arcs, dist, queued, wmin, warp, lane);
            const int32_t next = __reduce_min_sync(0xffffffffu, min(beyond, hbest));
            const int slot = bucket & 1;
            if (lane == 0 && next != INT_MAX) atomicMin(&sh->dmin[slot], next);
            __syncthreads();
            dmin = sh->dmin[slot];
            if (dmin == INT_MAX) break;
            if (tid == 0) sh->dmin[slot ^ 1] = INT_MAX;  // last read a bucket ago; next written after a barrier
        }

        int32_t* orow = out + (long long)item * ldo;
        const long long hs = h ? h[src] : 0;
        for (int v = tid; v < n; v += kThreads) {
            const int32_t dv = dist[v];
            long long r = dv;
            if (h && dv != kUnreached) r = (long long)dv + h[v] - hs;
            orow[v] = (dv == kUnreached || r >= kInf) ? kInf : (int32_t)r;
        }
        __syncthreads();  // the next source reuses shared memory
    }
}

// ------------------------------------------------------------------ grid-wide Delta-stepping

// One search over the whole GPU, for graphs whose distances do not fit a
// CTA's shared memory (the Delta-stepping page's single-source setting).
// The same buckets, light phases and heavy phase as above, with the state in
// global memory:
//   dist (the caller's output array), queued (the bucket structure, as in the
//   CTA search), wmin (per bitmap word, the least distance of its queued
//   vertices as of the last scan of the word), fresh (per word, the vertices
//   whose distance a relaxation lowered since that scan) and rset (R).
// Lane j of global warp g owns bitmap words (s * G + g) * 32 + j, s = 0, 1,
// ... (G warps in the grid), so a warp's lanes hold 32 adjacent words.
// A light phase selects and relaxes in one sweep, and phases are separated
// by one grid barrier (below) that also reduces an OR (did any warp select a
// vertex?) and a MIN (the next bucket) over all CTAs.  Relaxations of other
// warps run while a warp selects, so only the word's owner writes wmin, and
// relaxations mark the word in fresh instead: a word may be skipped only
// when it has no fresh vertex and its wmin is at least the bucket's end.  State
// that other SMs write is read through L2 (ld.global.cg), never from a stale
// L1 line.  Arc data is read-only and goes through the read-only path.  A
// vertex with more than kGridBig arcs in the phase is not walked by its warp
// alone: its arcs go, in segments of kGridBig, to a grid-wide list (a warp
// claims its lanes' slots with one atomic).  The phase's barrier then says
// (OR) whether the list is empty; if not, the grid's warps share the
// segments out round-robin, and a second barrier closes the phase.  A hub
// of an R-MAT graph (up to 10^5 - 10^6 arcs) is so spread over the whole
// GPU, and so are the many vertices of a few hundred arcs, which a warp
// walking 32 of them at a time would otherwise hold the phase back for.
// Measured on R-MAT scale 22: a threshold of 1024 arcs 3.56 ms per search,
// 256 2.85 ms, 128 2.67 ms, 64 2.97 ms, 32 3.53 ms.

constexpr int kGridThreads = 512;
constexpr int kGridWarps = kGridThreads / 32;
constexpr int kGridBig = 128;  // arcs above which a vertex's arcs go to the grid-wide list (see below)

struct GridCtrl {
    int any[3];          // OR slots, by barrier index mod 3
    int mn[3];           // MIN slots
    unsigned arrive;     // barrier arrivals
    unsigned gen;        // barrier generation
    int err;             // 1: a barrier wait ran out
    int big_count;       // segments on the grid-wide list in this phase
    int cnt[3];          // SUM slots
    int pad[3];
};

struct GridArgs {
    const int64_t* rp;
    const int32_t* nlight;
    const int2* arcs;
    int n, nw;
    int32_t delta;
    int32_t* dist;
    uint32_t* queued;
    int32_t* wmin;
    uint32_t* fresh;
    uint32_t* rset;
    GridCtrl* ctrl;
    int4* big;       // grid-wide list of hub segments: (dv, begin, count, -)
    int big_cap;
    unsigned long long timeout_ns;
    int inject;  // test hook: CTA 0 leaves before the first barrier
    int wide_peak;   // a bucket that selects this many vertices is past the search's peak
    int wide_max;    // the widest bucket, in multiples of delta
};

__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t* p) { return __ldcg(p); }
__device__ __forceinline__ int32_t ld_cg_i32(const int32_t* p) { return __ldcg(p); }

// Grid barrier with a bitwise OR and a MIN reduction; slot k % 3 of the control
// block holds barrier k's reductions, and CTA 0 clears slot (k + 2) % 3 once
// past barrier k (every CTA has read that slot, used by barrier k - 1, and
// none writes it before barrier k + 2).  Waits are bounded: after timeout_ns
// the CTA sets ctrl->err; every waiting CTA sees it and leaves.  With
// reset_list the last CTA to arrive empties the grid-wide hub list while all
// the others wait, so no push of the next phase can precede the reset.
// Returns false when the search must stop.
__device__ bool grid_reduce(const GridArgs& a, int& k, int any_in, int32_t min_in, int& any_out,
                            int32_t& min_out, bool reset_list = false, int sum_in = 0, int* sum_out = nullptr) {
    __shared__ int s_min, s_any, s_err, s_or, s_sum;
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        s_min = INT_MAX;
        s_or = 0;
        s_sum = 0;
    }
    __syncthreads();
    const int wor = __reduce_or_sync(0xffffffffu, any_in);
    const int32_t wm = __reduce_min_sync(0xffffffffu, min_in);
    const int ws = __reduce_add_sync(0xffffffffu, sum_in);
    if (lane == 0 && wor != 0) atomicOr(&s_or, wor);
    if (lane == 0 && wm != INT_MAX) atomicMin(&s_min, wm);
    if (lane == 0 && ws != 0) atomicAdd(&s_sum, ws);
    __syncthreads();
    if (tid == 0) {
        GridCtrl* c = a.ctrl;
        const int slot = k % 3;
        if (s_or) atomicOr(&c->any[slot], s_or);
        if (s_min != INT_MAX) atomicMin(&c->mn[slot], s_min);
        if (s_sum) atomicAdd(&c->cnt[slot], s_sum);
        const unsigned g0 = *reinterpret_cast<volatile unsigned*>(&c->gen);
        __threadfence();
        const unsigned arrived = atomicAdd(&c->arrive, 1u) + 1u;
        if (arrived == gridDim.x) {
            // every other CTA is waiting here, so shared state may be reset
            if (reset_list) c->big_count = 0;
            atomicExch(&c->arrive, 0u);
            __threadfence();
            atomicAdd(&c->gen, 1u);
        } else {
            const unsigned long long t0 = apsp::global_timer_ns();
            unsigned spins = 0;
            while (*reinterpret_cast<volatile unsigned*>(&c->gen) == g0) {
                if (*reinterpret_cast<volatile int*>(&c->err)) break;
                if ((++spins & 255u) == 0u && apsp::global_timer_ns() - t0 > a.timeout_ns) {
                    atomicExch(&c->err, 1);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        s_any = *reinterpret_cast<volatile int*>(&c->any[slot]);
        s_min = *reinterpret_cast<volatile int*>(&c->mn[slot]);
        s_sum = *reinterpret_cast<volatile int*>(&c->cnt[slot]);
        s_err = *reinterpret_cast<volatile int*>(&c->err);
        if (blockIdx.x == 0) {
            const int r = (k + 2) % 3;
            c->any[r] = 0;
            c->mn[r] = INT_MAX;
            c->cnt[r] = 0;
        }
    }
    __syncthreads();
    any_out = s_any;
    min_out = s_min;
    if (sum_out) *sum_out = s_sum;
    const bool ok = s_err == 0;
    __syncthreads();  // s_* are rewritten by the next call
    ++k;
    return ok;
}

// Relax `cnt` arcs from `beg` for a vertex at distance dv, 32 lanes of a warp
// striding over them, up to 4 loads in flight.
__device__ __forceinline__ int32_t relax_run(const int2* __restrict__ arcs, int beg, int cnt, uint32_t dv,
                                             int32_t* dist, uint32_t* queued, uint32_t* fresh, int lane) {
    int32_t best = INT_MAX;
    for (int o = 0; o < cnt; o += 128) {
        int2 x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int t = o + q * 32 + lane;
            x[q] = t < cnt ? __ldg(arcs + beg + t) : make_int2(0, -1);
        }
        // the four targets' distances first, all in flight together: a value
        // read before another relaxation lowers it is only larger (distances
        // only decrease), so the check may try an atomic in vain, never skip a
        // needed one
        int32_t du[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) du[q] = x[q].y < 0 ? 0 : ld_cg_i32(dist + x[q].x);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (x[q].y < 0) continue;
            const uint32_t s = dv + (uint32_t)x[q].y;
            const int32_t nd = s >= (uint32_t)kUnreached ? kUnreached : (int32_t)s;
            const int u = x[q].x;
            if (nd < du[q] && nd < atomicMin(dist + u, nd)) {
                atomicOr(queued + (u >> 5), 1u << (u & 31));
                atomicOr(fresh + (u >> 5), 1u << (u & 31));
                best = min(best, nd);
            }
        }
    }
    return best;
}

// Relax the light (kLight) or heavy arcs of the vertices of 32 bitmap words:
// lane j holds in `bits` the members of word wbase + j (zero past the end),
// and the whole warp takes part.  Batches of 32 vertices as in the CTA
// search; a vertex with more than kGridBig arcs goes to the grid-wide list
// in segments of kGridBig, and `pushed` says whether this lane put any there.
template <bool kLight>
__device__ int32_t expand_words(const GridArgs& a, long long wbase, uint32_t bits, int& pushed) {
    const int lane = threadIdx.x & 31;
    int32_t best = INT_MAX;
    {
        const int c = __popc(bits);
        int wincl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wincl, o);
            if (lane >= o) wincl += y;
        }
        const int members = __shfl_sync(0xffffffffu, wincl, 31);
        const int wexcl = wincl - c;
        for (int b0 = 0; b0 < members; b0 += 32) {
            const int g = b0 + lane;
            const int j = last_lane_at_or_below(wexcl, g);
            const uint32_t wbits = __shfl_sync(0xffffffffu, bits, j);
            const int wstart = __shfl_sync(0xffffffffu, wexcl, j);
            int beg = 0, cnt = 0;
            uint32_t dv = 0;
            if (g < members) {
                const int v = ((int)wbase + j) * 32 + kth_set_bit(wbits, g - wstart);
                const int r0 = (int)__ldg(a.rp + v), nl = __ldg(a.nlight + v);
                if (kLight) {
                    beg = r0;
                    cnt = nl;
                } else {
                    beg = r0 + nl;
                    cnt = (int)__ldg(a.rp + v + 1) - r0 - nl;
                }
                dv = (uint32_t)ld_cg_i32(a.dist + v);
            }
            {
                // vertices with more than kGridBig arcs go to the grid-wide
                // list, one segment per kGridBig arcs; the warp claims its
                // lanes' slots with one atomic
                const int nseg = cnt > kGridBig ? (cnt + kGridBig - 1) / kGridBig : 0;
                int sincl = nseg;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, sincl, o);
                    if (lane >= o) sincl += y;
                }
                const int stotal = __shfl_sync(0xffffffffu, sincl, 31);
                if (stotal > 0) {
                    int sbase = 0;
                    if (lane == 31) sbase = atomicAdd(&a.ctrl->big_count, stotal);
                    sbase = __shfl_sync(0xffffffffu, sbase, 31);
                    const int first = sbase + sincl - nseg;
                    if (sbase + stotal <= a.big_cap) {
                        for (int q = 0; q < nseg; ++q)
                            a.big[first + q] = make_int4((int)dv, beg + q * kGridBig, min(kGridBig, cnt - q * kGridBig), 0);
                        if (nseg > 0) {
                            cnt = 0;
                            pushed = 1;
                        }
                    } else {
                        // Cannot happen: a phase pushes at most the sum of
                        // ceil(arcs / kGridBig) over its vertices, within the
                        // 2 m / kGridBig + 16 slots.  Were it to, the claimed
                        // slots below the cap get empty segments and the warp
                        // walks the arcs itself.
                        for (int q = 0; q < nseg; ++q)
                            if (first + q < a.big_cap) a.big[first + q] = make_int4(0, 0, 0, 0);
                    }
                }
            }
            const uint32_t heavy = __ballot_sync(0xffffffffu, cnt > kGridBig);  // not on the list: walk here
            for (uint32_t hb = heavy; hb; hb &= hb - 1) {
                const int src = __ffs(hb) - 1;
                best = min(best, relax_run(a.arcs, __shfl_sync(0xffffffffu, beg, src),
                                           __shfl_sync(0xffffffffu, cnt, src),
                                           __shfl_sync(0xffffffffu, dv, src), a.dist, a.queued, a.fresh, lane));
            }
            if (cnt > kGridBig) cnt = 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            const int excl = incl - cnt;
            for (int base = 0; base < total; base += 128) {
                int2 x[4];
                uint32_t d[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = base + q * 32 + lane;
                    const int pos = last_lane_at_or_below(excl, t);
                    const int e = __shfl_sync(0xffffffffu, beg, pos) + t - __shfl_sync(0xffffffffu, excl, pos);
                    d[q] = __shfl_sync(0xffffffffu, dv, pos);
                    x[q] = t < total ? __ldg(a.arcs + e) : make_int2(0, -1);
                }
                int32_t du[4];  // all four loads in flight before the atomics (see relax_run)
#pragma unroll
                for (int q = 0; q < 4; ++q) du[q] = x[q].y < 0 ? 0 : ld_cg_i32(a.dist + x[q].x);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (x[q].y < 0) continue;
                    const uint32_t sum = d[q] + (uint32_t)x[q].y;
                    const int32_t nd = sum >= (uint32_t)kUnreached ? kUnreached : (int32_t)sum;
                    const int u = x[q].x;
                    if (nd < du[q] && nd < atomicMin(a.dist + u, nd)) {
                        atomicOr(a.queued + (u >> 5), 1u << (u & 31));
                        atomicOr(a.fresh + (u >> 5), 1u << (u & 31));
                        best = min(best, nd);
                    }
                }
            }
        }
    }
    return best;
}

// The same for every vertex in the bitmap `set` (global), clearing it.
template <bool kLight>
__device__ int32_t expand_grid(const GridArgs& a, uint32_t* set, int& pushed) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kGridWarps + warp, G = gridDim.x * kGridWarps;
    int32_t best = INT_MAX;
    for (int s = 0;; ++s) {
        const long long wbase = ((long long)s * G + gw) * 32;
        if (wbase >= a.nw) break;  // warp-uniform
        const int i = (int)wbase + lane;
        uint32_t bits = 0u;
        if (i < a.nw) {
            bits = ld_cg_u32(set + i);
            if (bits) set[i] = 0u;
        }
        if (__any_sync(0xffffffffu, bits != 0u)) best = min(best, expand_words<kLight>(a, wbase, bits, pushed));
    }
    return best;
}

// After the barrier that ends a phase's batches: every warp takes hub
// segments from the grid-wide list until it is empty (the count is final by
// then).
__device__ int32_t drain_grid_list(const GridArgs& a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kGridWarps + warp, G = gridDim.x * kGridWarps;
    const int count = min(*reinterpret_cast<volatile int*>(&a.ctrl->big_count), a.big_cap);
    int32_t best = INT_MAX;
    // segments are at most kGridBig arcs each: a static round-robin over the
    // grid's warps balances them without a shared cursor (1.5% faster with
    // two segments per warp in flight than with one)
    for (int idx = gw; idx < count; idx += 2 * G) {
        // two segments at a time: eight arcs per lane in flight
        const int4 e0 = __ldcg(a.big + idx);  // written by other CTAs before the barrier
        const int4 e1 = idx + G < count ? __ldcg(a.big + idx + G) : make_int4(0, 0, 0, 0);
        int2 x[8];
        uint32_t d[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int t = q * 32 + lane;
            x[q] = t < e0.z ? __ldg(a.arcs + e0.y + t) : make_int2(0, -1);
            x[4 + q] = t < e1.z ? __ldg(a.arcs + e1.y + t) : make_int2(0, -1);
            d[q] = (uint32_t)e0.x;
            d[4 + q] = (uint32_t)e1.x;
        }
        int32_t du[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) du[q] = x[q].y < 0 ? 0 : ld_cg_i32(a.dist + x[q].x);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (x[q].y < 0) continue;
            const uint32_t sum = d[q] + (uint32_t)x[q].y;
            const int32_t nd = sum >= (uint32_t)kUnreached ? kUnreached : (int32_t)sum;
            const int u = x[q].x;
            if (nd < du[q] && nd < atomicMin(a.dist + u, nd)) {
                atomicOr(a.queued + (u >> 5), 1u << (u & 31));
                atomicOr(a.fresh + (u >> 5), 1u << (u & 31));
                best = min(best, nd);
            }
        }
    }
    return best;
}

// The rest of a phase once its batches are done: the closing barrier, or,
// when some warp put hub segments on the grid-wide list, a barrier, the
// list shared out over the grid, and a second barrier whose last arriver
// empties the list (the next phase may push as soon as it is past).
// in_min: this lane's least successful relaxation; out_min: the MIN over
// the grid.  flag_in / flag_out: one more OR over the grid, taken by the
// same barrier.  Returns false when the search must stop.
__device__ bool close_phase(const GridArgs& a, int& k, int pushed, int32_t in_min, int32_t& out_min,
                            int flag_in = 0, int* flag_out = nullptr, int sum_in = 0, int* sum_out = nullptr) {
    int bits;
    if (!grid_reduce(a, k, (pushed ? 1 : 0) | (flag_in ? 2 : 0), in_min, bits, out_min, false, sum_in, sum_out))
        return false;
    if (flag_out) *flag_out = bits >> 1;
    if (!(bits & 1)) return true;
    const int32_t b = drain_grid_list(a);
    int unused;
    int32_t m2;
    if (!grid_reduce(a, k, 0, b, unused, m2, true)) return false;  // its last arriver empties the list
    out_min = min(out_min, m2);
    return true;
}

__global__ void __launch_bounds__(kGridThreads, 2) sssp_grid_kernel(GridArgs a) {
    if (a.inject && blockIdx.x == 0) return;  // test hook (apsp_debug_inject_grid_timeout)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kGridWarps + warp, G = gridDim.x * kGridWarps;
    int k = 0;  // barrier index, the same in every CTA
    int32_t dmin = 0;
    // Bucket widening.  Past the search's peak (a bucket that selected at
    // least n / 64 vertices) the frontier thins out, and a bucket of width
    // delta costs its grid barriers for few vertices.  From then on each
    // bucket is twice as wide as the one before, up to about 2 * w_max.  A
    // heavy arc may then land inside the bucket it leaves: its head is
    // queued below the bucket's end and the next bucket, which starts at the
    // least queued distance, takes it again, so the distances stay exact (a
    // vertex is settled more than once at worst).  Measured on R-MAT scales
    // 21 / 22 / 23, with delta = w_max / (2 * degree): 1.393 / 1.843 /
    // 3.160 ms per search, against 1.955 / 2.528 / 4.42 ms with fixed
    // buckets and the best fixed delta.
    int width = 1;        // the bucket spans `width` multiples of delta
    bool peaked = false;  // some bucket selected at least wide_peak vertices
    for (;;) {  // buckets
        const long long hi_ll = ((long long)(dmin / a.delta) + width) * a.delta;
        const int32_t hi = hi_ll >= kUnreached ? kUnreached : (int32_t)hi_ll;
        int32_t beyond;
        int32_t lmin = INT_MAX;  // least distance set by the last light phase, over the grid
        int nsel = 0;            // vertices this lane selected in the bucket's light phases
        for (;;) {  // light phases
            // Each warp selects the queued vertices below hi in its bitmap
            // words and relaxes their light arcs in the same sweep (a warp
            // expands only the words it selected).  A word is looked at
            // unless it has no fresh vertex and its wmin (exact as of its
            // last scan) is at least hi; a look takes the fresh bits,
            // computes the exact least distance of the vertices left
            // queued, and clears only the bits it selected.  Anything a
            // concurrent relaxation changes meanwhile is marked fresh again,
            // for the next phase.
            //   The bucket's light work is done once a phase sets no
            // distance below hi: every vertex below hi queued before it was
            // selected in it.  The next bucket then starts at the least of
            // what the sweep left queued (`beyond`, per lane), what the
            // phase's relaxations set (lmin; a relaxation after a word's
            // look shows up there) and what the heavy phase sets: a lower
            // bound on every queued distance, so nothing is left behind.
            beyond = INT_MAX;
            int any = 0, pushed = 0;
            int32_t best = INT_MAX;
            for (int s = 0;; ++s) {
                const long long wbase = ((long long)s * G + gw) * 32;
                if (wbase >= a.nw) break;  // warp-uniform
                const int i = (int)wbase + lane;
                uint32_t sel = 0u;
                if (i < a.nw) {
                    uint32_t fr = ld_cg_u32(a.fresh + i);
                    if (fr) fr = atomicExch(a.fresh + i, 0u);
                    const int32_t wm = ld_cg_i32(a.wmin + i);
                    if (fr == 0u && wm >= hi) {
                        beyond = min(beyond, wm);
                    } else {
                        // a relaxation sets the queued bit, then the fresh bit, and the
                        // two may become visible in either order: a fresh bit taken
                        // counts as queued (its distance is already in place, as the
                        // relaxation's returning atomicMin on it came first)
                        const uint32_t all = ld_cg_u32(a.queued + i) | fr;
                        int32_t rem = INT_MAX;
                        const int vb = i * 32;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {  // the word's distances, 4 at a time where any is queued
                            const uint32_t nib = (all >> (q * 4)) & 0xFu;
                            if (nib == 0u) continue;
                            int32_t d4[4];
                            if (vb + q * 4 + 3 < a.n) {
                                const int4 v4 = __ldcg(reinterpret_cast<const int4*>(a.dist + vb + q * 4));
                                d4[0] = v4.x;
                                d4[1] = v4.y;
                                d4[2] = v4.z;
                                d4[3] = v4.w;
                            } else {  // the ragged end of the array
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    d4[c] = vb + q * 4 + c < a.n ? ld_cg_i32(a.dist + vb + q * 4 + c) : INT_MAX;
                            }
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                if (!((nib >> c) & 1u)) continue;
                                if (d4[c] < hi)
                                    sel |= 1u << (q * 4 + c);
                                else
                                    rem = min(rem, d4[c]);
                            }
                        }
                        if (sel) atomicAnd(a.queued + i, ~sel);
                        if (rem != wm) a.wmin[i] = rem;  // only this lane writes word i's wmin
                        beyond = min(beyond, rem);
                        if (sel) {
                            a.rset[i] = ld_cg_u32(a.rset + i) | sel;
                            any = 1;
                            nsel += __popc(sel);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, sel != 0u))
                    best = min(best, expand_words<true>(a, wbase, sel, pushed));
            }
            int any_g;
            if (!close_phase(a, k, pushed, best, lmin, any, &any_g)) return;
            if (!any_g || lmin >= hi) break;
        }
        int pushed = 0;
        const int32_t hbest = expand_grid<false>(a, a.rset, pushed);
        int32_t next;
        int selected = 0;  // over the grid: the same in every CTA, and so is the next width
        if (!close_phase(a, k, pushed, min(min(beyond, hbest), lmin), next, 0, nullptr, nsel, &selected)) return;
        if (next == INT_MAX) break;
        dmin = next;
        if (selected >= a.wide_peak) peaked = true;
        if (peaked) width = min(2 * width, a.wide_max);
    }
}

// dist <- kUnreached everywhere but the source, the bitmaps cleared, the
// control block reset.
__global__ void grid_init_kernel(GridArgs a, int src) {
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long v = t; v < a.n; v += stride) a.dist[v] = v == src ? 0 : kUnreached;
    for (long long i = t; i < a.nw; i += stride) {
        a.queued[i] = i == (src >> 5) ? 1u << (src & 31) : 0u;
        a.wmin[i] = i == (src >> 5) ? 0 : INT_MAX;
        a.fresh[i] = 0u;
        a.rset[i] = 0u;
    }
    if (t == 0) {
        GridCtrl* c = a.ctrl;
        for (int s = 0; s < 3; ++s) {
            c->any[s] = 0;
            c->mn[s] = INT_MAX;
        }
        c->arrive = 0u;
        c->gen = 0u;
        c->err = 0;
        c->big_count = 0;
        for (int s = 0; s < 3; ++s) c->cnt[s] = 0;
    }
}

// Unreached and saturated distances read INF.
__global__ void grid_finish_kernel(int32_t* dist, int n) {
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += (long long)gridDim.x * blockDim.x)
        if (dist[v] >= kInf) dist[v] = kInf;
}

// ------------------------------------------------------------------ host side

struct DevBuf {
    void* p = nullptr;
    size_t bytes = 0;
};

struct SparseState {
    DevBuf rp, body, work, grid;
};

std::mutex g_sp_mu;
std::vector<SparseState> g_sp;

// Optional timing of the search kernel (apsp_sparse_timing_*), under g_sp_mu.
struct SparseTiming {
    bool enabled = false;
    double search_ms = 0.0;
    long long searches = 0;
    long long kernels = 0;  // every kernel launched by the sparse entry points
};
SparseTiming g_sp_timing;

// Kernel launches of the sparse entry points are counted for the timing API
// (callers hold g_sp_mu).
inline void count_kernel(int k = 1) { g_sp_timing.kernels += k; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

apsp_status_t grow(DevBuf& b, size_t need) {
    if (b.bytes >= need) return APSP_OK;
    if (b.p) {
        cudaDeviceSynchronize();
        cudaFree(b.p);
        b.p = nullptr;
        b.bytes = 0;
    }
    const cudaError_t e = cudaMalloc(&b.p, need);
    if (e != cudaSuccess) {
        cudaGetLastError();
        b.p = nullptr;
        apsp::set_last_cuda_error((int)e);
        return APSP_ENOMEM;
    }
    b.bytes = need;
    return APSP_OK;
}

SparseState* sp_state() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if ((int)g_sp.size() <= dev) g_sp.resize(dev + 1);
    return &g_sp[dev];
}

int blocks_for_warps(long long warps) { return (int)((warps * 32 + 255) / 256); }

// Work buffer: [0, 256) small counters, then h (int64, n), w' (int32, m),
// the partitioned arcs (int2, m) and the light-arc counts (int32, n).
struct Work {
    int* range;    // [0] min, [1] max, [2] bad head
    int* counter;  // source counter of the search
    int* changed;  // Bellman-Ford round flag, then the reweighting range flag
    int* err;      // search error bits
    long long* h;
    int32_t* wh;
    int2* arcs;
    int32_t* nlight;
    int32_t* biglist;  // vertices with more than kPartBig arcs
    int* bigcount;
};

size_t work_bytes(int n, long long m) {
    const size_t mm = (size_t)(m > 0 ? m : 1);
    return 256 + align256((size_t)n * 8) + align256(mm * 4) + align256(mm * 8) + 2 * align256((size_t)n * 4);
}

Work work_layout(void* base, int n, long long m) {
    const size_t mm = (size_t)(m > 0 ? m : 1);
    char* b = static_cast<char*>(base);
    Work wk;
    wk.range = reinterpret_cast<int*>(b);
    wk.counter = wk.range + 4;
    wk.changed = wk.range + 5;
    wk.err = wk.range + 6;
    size_t off = 256;
    wk.h = reinterpret_cast<long long*>(b + off);
    off += align256((size_t)n * 8);
    wk.wh = reinterpret_cast<int32_t*>(b + off);
    off += align256(mm * 4);
    wk.arcs = reinterpret_cast<int2*>(b + off);
    off += align256(mm * 8);
    wk.nlight = reinterpret_cast<int32_t*>(b + off);
    off += align256((size_t)n * 4);
    wk.biglist = reinterpret_cast<int32_t*>(b + off);
    wk.bigcount = wk.range + 7;
    return wk;
}

apsp_status_t read_int(const int* dev, int* host, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(host, dev, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? APSP_OK : sp_fail(e);
}

apsp_status_t read_m(const int64_t* rp, int n, long long* m, cudaStream_t s) {
    int64_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, rp + n, sizeof(int64_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return sp_fail(e);
    *m = (long long)v;
    return APSP_OK;
}

// Weight range (and head check when col is given) of m arcs.
apsp_status_t weight_range(const int32_t* w, const int32_t* col, long long m, int n, int* range,
                           cudaStream_t s, int* lo, int* hi, int* bad) {
    const int init[3] = {INT_MAX, INT_MIN, 0};
    cudaError_t e = cudaMemcpyAsync(range, init, sizeof(init), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return sp_fail(e);
    if (m > 0) {
        long long blocks = (m + 255) / 256;
        if (blocks > 4096) blocks = 4096;
        weight_range_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, col, m, n, range);
        count_kernel();
        e = cudaGetLastError();
        if (e != cudaSuccess) return sp_fail(e);
    }
    int r[3];
    e = cudaMemcpyAsync(r, range, sizeof(r), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return sp_fail(e);
    *lo = r[0];
    *hi = r[1];
    if (bad) *bad = r[2];
    return APSP_OK;
}

// A caller's row_ptr: row_ptr[0] = 0 and non-decreasing (so every arc
// index a search forms lies in [0, row_ptr[n])).
apsp_status_t check_row_ptr(const int64_t* rp, int n, int* flag, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), s);
    if (e != cudaSuccess) return sp_fail(e);
    rowptr_check_kernel<<<(n + 1 + 255) / 256, 256, 0, s>>>(rp, n, flag);
    count_kernel();
    e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    int bad = 0;
    apsp_status_t rc = read_int(flag, &bad, s);
    if (rc != APSP_OK) return rc;
    return bad ? APSP_EINVAL : APSP_OK;
}

// The light-first partition of all arcs (partition_kernel, then
// partition_big_kernel for the listed high-degree vertices).  Blocks on s.
apsp_status_t partition_arcs(const int64_t* rp, const int32_t* col, const int32_t* w, int n, int32_t delta,
                             int2* arcs, int32_t* nlight, int32_t* biglist, int* bigcount, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(bigcount, 0, sizeof(int), s);
    if (e != cudaSuccess) return sp_fail(e);
    partition_kernel<<<blocks_for_warps(n), 256, 0, s>>>(rp, col, w, n, delta, arcs, nlight, biglist, bigcount);
    count_kernel();
    e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    int big = 0;
    apsp_status_t rc = read_int(bigcount, &big, s);
    if (rc != APSP_OK) return rc;
    if (big > 0) {
        partition_big_kernel<<<big, kPartBigThreads, 0, s>>>(rp, col, w, delta, arcs, nlight, biglist);
        count_kernel();
        e = cudaGetLastError();
        if (e != cudaSuccess) return sp_fail(e);
    }
    return APSP_OK;
}

// Bucket width when the caller gives none.  The Delta-stepping page tunes
// Delta by measurement (section 4.4); these rules are fitted to sweeps here:
//   per-CTA searches (Johnson): 0.8 * w_max / sqrt(mean out-degree).  Within
//     a few percent of the best of 4-6 widths on er256, er2048, er8192 and
//     ba16384, whose degrees run from 16 to 4096.
//   grid-wide search: w_max / (2 * mean out-degree), with buckets widened
//     after the search's peak (the bucket loop of sssp_grid_kernel).  Of
//     1/4, 3/8, 1/2, 3/4, 1 and 3/2 times w_max / degree with widening, 1/4
//     to 1/2 ran R-MAT scales 20-23 fastest; without widening the best was
//     2 * w_max / degree.
enum class DeltaRule { kCta, kGrid };
int32_t default_delta(int n, long long m, int wmax, DeltaRule rule = DeltaRule::kCta) {
    if (m <= 0 || wmax <= 0) return 1;
    double avg_deg = (double)m / (double)(n > 0 ? n : 1);
    if (avg_deg < 1.0) avg_deg = 1.0;
    double d = rule == DeltaRule::kGrid ? 0.5 * (double)wmax / avg_deg : 0.8 * (double)wmax / sqrt(avg_deg);
    if (d < 1.0) d = 1.0;
    if (d > (double)kInf) d = (double)kInf;
    return (int32_t)d;
}

template <int kThreads, int kMinBlocks = 1536 / kThreads>
apsp_status_t launch_search(const int64_t* rp, const Work& wk, int n, const int32_t* sources, int nsrc,
                            int32_t delta, const long long* h, int32_t* out, long long ldo, size_t smem, int grid,
                            cudaStream_t s) {
    sssp_delta_kernel<kThreads, kMinBlocks><<<grid, kThreads, smem, s>>>(rp, wk.nlight, wk.arcs, n, sources, nsrc, delta, h,
                                                             out, ldo, wk.counter, wk.err);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? APSP_OK : sp_fail(e);
}

// Partition the arcs against delta, then one persistent search CTA per
// resident slot.  512 threads a CTA while at least two CTAs fit an SM (n up
// to about 24K), else 1024 threads in one CTA.  Graphs of at most 8192
// vertices with a mean out-degree of at most 512 take 256-thread CTAs when
// there are sources enough to fill them: twice as many searches share an
// SM, and such a search's phases seldom keep 512 threads busy.  Measured
// (Johnson, all sources): ER n = 2048, degree 100: 1.185 -> 1.064 ms;
// n = 8192, degree 4096: 393.8 -> 402.1 ms; n = 256 (256 sources, fewer
// than the slots): 0.150 -> 0.155 ms.  Where shared memory leaves room for
// four 512-thread CTAs on an SM, a copy of the kernel compiled for 32
// registers a thread (four CTAs) runs instead of the one for 40 (three):
// ER n = 8192, degree 4096: 222 -> 184 ms (20 bytes of spill; with two
// chunks in flight instead of four, no better spill and 249 ms).  Forced
// on BA n = 16384, whose 68 KB of shared memory a CTA hold three an SM
// anyway, the 32-register copy only costs: 17.05 -> 17.91 ms.
apsp_status_t launch_sssp(const int64_t* rp, const int32_t* col, const int32_t* w, int n, long long m,
                          const int32_t* sources, int nsrc, int32_t delta, const long long* h, int32_t* out,
                          long long ldo, const Work& wk, cudaStream_t s) {
    apsp_status_t prc = partition_arcs(rp, col, w, n, delta, wk.arcs, wk.nlight, wk.biglist, wk.bigcount, s);
    if (prc != APSP_OK) return prc;
    cudaError_t e;
    const size_t smem = sssp_smem_bytes(n);
    // Kernel attributes and occupancies for this shared-memory size, kept
    // from the last call on this device (the callers hold g_sp_mu).
    struct LaunchShape {
        int dev = -1, sms = 0, per_sm[4] = {0, 0, 0, 0};  // 256, 512, 1024 threads; 512 at 32 registers
        size_t smem = 0;
    };
    static LaunchShape shape;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return sp_fail(e);
    if (shape.dev != dev || shape.smem != smem) {
        LaunchShape x;
        e = cudaDeviceGetAttribute(&x.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sssp_delta_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sssp_delta_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sssp_delta_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.per_sm[0], sssp_delta_kernel<256>, 256, smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.per_sm[1], sssp_delta_kernel<512>, 512, smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.per_sm[2], sssp_delta_kernel<1024>, 1024, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sssp_delta_kernel<512, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.per_sm[3], sssp_delta_kernel<512, 4>, 512, smem);
        if (e != cudaSuccess) return sp_fail(e);
        x.dev = dev;
        x.smem = smem;
        shape = x;
    }
    const int sms = shape.sms;
    const bool wide = n > 1024 * (512 / 32) || shape.per_sm[1] < 2;  // the 512-thread CTA covers n <= 16384
    const bool narrow = !wide && n <= 1024 * (256 / 32) && m <= 512LL * n &&
                        (long long)nsrc >= (long long)sms * shape.per_sm[0];
    const bool four = !wide && !narrow && shape.per_sm[3] >= 4;  // shared memory leaves room for four
    const int per_sm = shape.per_sm[wide ? 2 : narrow ? 0 : four ? 3 : 1];
    if (per_sm < 1) return APSP_EUNSUPPORTED;
    long long grid = (long long)sms * per_sm;
    if (grid > nsrc) grid = nsrc;
    e = cudaMemsetAsync(wk.counter, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(wk.err, 0, sizeof(int), s);
    if (e != cudaSuccess) return sp_fail(e);
    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (g_sp_timing.enabled) {
        e = cudaEventCreate(&ev[0]);
        if (e == cudaSuccess) e = cudaEventCreate(&ev[1]);
        if (e == cudaSuccess) e = cudaEventRecord(ev[0], s);
        if (e != cudaSuccess) {
            for (cudaEvent_t x : ev)
                if (x) cudaEventDestroy(x);
            return sp_fail(e);
        }
    }
    apsp_status_t rc =
        wide     ? launch_search<1024>(rp, wk, n, sources, nsrc, delta, h, out, ldo, smem, (int)grid, s)
        : narrow ? launch_search<256>(rp, wk, n, sources, nsrc, delta, h, out, ldo, smem, (int)grid, s)
        : four   ? launch_search<512, 4>(rp, wk, n, sources, nsrc, delta, h, out, ldo, smem, (int)grid, s)
                 : launch_search<512>(rp, wk, n, sources, nsrc, delta, h, out, ldo, smem, (int)grid, s);
    count_kernel();  // the search
    if (rc == APSP_OK && ev[1]) {
        e = cudaEventRecord(ev[1], s);
        if (e != cudaSuccess) rc = sp_fail(e);
    }
    int err = 0;
    if (rc == APSP_OK) rc = read_int(wk.err, &err, s);  // waits for the search
    if (rc == APSP_OK && ev[1]) {
        float t = 0.f;
        e = cudaEventElapsedTime(&t, ev[0], ev[1]);
        if (e != cudaSuccess) {
            rc = sp_fail(e);
        } else {
            g_sp_timing.search_ms += t;
            g_sp_timing.searches += 1;
        }
    }
    for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
    if (rc != APSP_OK) return rc;
    return err ? APSP_EINVAL : APSP_OK;
}

// Johnson's APSP on a device CSR with m arcs into out (n x ld).
apsp_status_t johnson(const int64_t* rp, const int32_t* col, const int32_t* w, int n, long long m, int32_t delta,
                      int32_t* out, int ld, const Work& wk, bool check_heads, cudaStream_t s) {
    int lo = 0, hi = 0, bad = 0;
    apsp_status_t rc = weight_range(w, check_heads ? col : nullptr, m, n, wk.range, s, &lo, &hi, &bad);
    if (rc != APSP_OK) return rc;
    if (bad || (m > 0 && (lo <= -kInf || hi >= kInf))) return APSP_EINVAL;
    const int32_t* wuse = w;
    const long long* huse = nullptr;
    cudaError_t e;
    if (m > 0 && lo < 0) {
        // Bellman-Ford from the virtual vertex s: its 0-weight arcs give h = 0.
        e = cudaMemsetAsync(wk.h, 0, (size_t)n * 8, s);
        if (e != cudaSuccess) return sp_fail(e);
        bool converged = false;
        for (int round = 0; round <= n; ++round) {  // n = |V'| - 1 rounds, then one more as the check
            e = cudaMemsetAsync(wk.changed, 0, sizeof(int), s);
            if (e != cudaSuccess) return sp_fail(e);
            bf_round_kernel<<<blocks_for_warps(n), 256, 0, s>>>(rp, col, w, n, wk.h, wk.changed);
            count_kernel();
            e = cudaGetLastError();
            if (e != cudaSuccess) return sp_fail(e);
            int changed = 0;
            rc = read_int(wk.changed, &changed, s);
            if (rc != APSP_OK) return rc;
            if (!changed) {
                converged = true;
                break;
            }
        }
        if (!converged) return APSP_ENEGCYCLE;
        e = cudaMemsetAsync(wk.changed, 0, sizeof(int), s);
        if (e != cudaSuccess) return sp_fail(e);
        reweight_kernel<<<blocks_for_warps(n), 256, 0, s>>>(rp, col, w, n, wk.h, wk.wh, wk.changed);
        count_kernel();
        e = cudaGetLastError();
        if (e != cudaSuccess) return sp_fail(e);
        int range_bad = 0;
        rc = read_int(wk.changed, &range_bad, s);
        if (rc != APSP_OK) return rc;
        if (range_bad) return APSP_EINVAL;
        wuse = wk.wh;
        huse = wk.h;
        rc = weight_range(wk.wh, nullptr, m, n, wk.range, s, &lo, &hi, nullptr);
        if (rc != APSP_OK) return rc;
    }
    if (delta <= 0) delta = default_delta(n, m, hi);
    return launch_sssp(rp, col, wuse, n, m, nullptr, n, delta, huse, out, ld, wk, s);
}

// CSR of a dense matrix into st.rp / st.body; returns m.
apsp_status_t build_csr(const int32_t* dist, int n, int ld, SparseState& st, long long* m_out, cudaStream_t s) {
    apsp_status_t rc = grow(st.rp, align256((size_t)(n + 1) * 8));
    if (rc != APSP_OK) return rc;
    int64_t* rp = static_cast<int64_t*>(st.rp.p);
    csr_count_kernel<<<blocks_for_warps(n), 256, 0, s>>>(dist, ld, n, rp);
    scan_kernel<<<1, kScanThreads, 0, s>>>(rp, n);
    count_kernel(2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    long long m = 0;
    rc = read_m(rp, n, &m, s);
    if (rc != APSP_OK) return rc;
    const size_t colb = align256((size_t)(m > 0 ? m : 1) * 4);
    rc = grow(st.body, 2 * colb);
    if (rc != APSP_OK) return rc;
    int32_t* col = static_cast<int32_t*>(st.body.p);
    int32_t* w = reinterpret_cast<int32_t*>(static_cast<char*>(st.body.p) + colb);
    csr_fill_kernel<<<blocks_for_warps(n), 256, 0, s>>>(dist, ld, n, rp, col, w);
    count_kernel();
    e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    *m_out = m;
    return APSP_OK;
}

// Grid-search buffer: [ctrl 256 B | flags 256 B | (row_ptr copy) | nlight |
// queued | wmin | fresh | rset | arcs | partition's big-vertex list | hub
// segment list], each section 256-byte aligned.  flags: [0..2] weight range,
// [4] row_ptr check, [6] big-vertex count.  The segment list holds at most
// one phase's hub segments: fewer than m / kGridBig full ones plus one
// partial one per hub, itself more than kGridBig arcs, so 2 m / kGridBig + 16
// entries suffice.
int grid_seg_cap(long long m) { return (int)(2 * (m / kGridBig) + 16); }

size_t grid_bytes(int n, long long m, bool own_rp) {
    const size_t nw = (size_t)(n + 31) / 32;
    return 512 + (own_rp ? align256((size_t)(n + 1) * 8) : 0) + 2 * align256((size_t)n * 4) +
           4 * align256(nw * 4) + align256((size_t)(m > 0 ? m : 1) * 8) +
           align256((size_t)grid_seg_cap(m) * sizeof(int4));
}

// Check the graph, choose delta, lay out `buf` and partition the arcs into
// it.  With own_rp the buffer also keeps a copy of row_ptr, so that the
// caller's arrays are not needed afterwards.  Blocks on s.
apsp_status_t grid_prepare(const int64_t* rp, const int32_t* col, const int32_t* w, int n, long long m, int32_t delta,
                           char* buf, bool own_rp, GridArgs& a, cudaStream_t s) {
    const size_t nw = (size_t)(n + 31) / 32;
    a.ctrl = reinterpret_cast<GridCtrl*>(buf);
    int* flags = reinterpret_cast<int*>(buf + 256);
    size_t off = 512;
    int64_t* rp_copy = nullptr;
    if (own_rp) {
        rp_copy = reinterpret_cast<int64_t*>(buf + off);
        off += align256((size_t)(n + 1) * 8);
    }
    int32_t* nlight = reinterpret_cast<int32_t*>(buf + off);
    off += align256((size_t)n * 4);
    a.queued = reinterpret_cast<uint32_t*>(buf + off);
    off += align256(nw * 4);
    a.wmin = reinterpret_cast<int32_t*>(buf + off);
    off += align256(nw * 4);
    a.fresh = reinterpret_cast<uint32_t*>(buf + off);
    off += align256(nw * 4);
    a.rset = reinterpret_cast<uint32_t*>(buf + off);
    off += align256(nw * 4);
    int2* arcs = reinterpret_cast<int2*>(buf + off);
    off += align256((size_t)(m > 0 ? m : 1) * 8);
    int32_t* biglist = reinterpret_cast<int32_t*>(buf + off);
    off += align256((size_t)n * 4);
    a.big = reinterpret_cast<int4*>(buf + off);
    a.big_cap = grid_seg_cap(m);
    a.nlight = nlight;
    a.arcs = arcs;
    a.n = n;
    a.nw = (int)nw;
    a.dist = nullptr;
    a.timeout_ns = 2000000000ull;
    a.inject = 0;

    apsp_status_t rc = check_row_ptr(rp, n, flags + 4, s);
    if (rc != APSP_OK) return rc;
    int lo = 0, hi = 0, bad = 0;
    rc = weight_range(w, col, m, n, flags, s, &lo, &hi, &bad);
    if (rc != APSP_OK) return rc;
    if (bad || (m > 0 && (lo < 0 || hi >= kInf))) return APSP_EINVAL;
    if (delta <= 0) delta = default_delta(n, m, hi, DeltaRule::kGrid);
    a.delta = delta;
    a.wide_peak = n / 64 > 1 ? n / 64 : 1;
    a.wide_max = 1;  // buckets up to about 2 * w_max wide
    while (a.wide_max < (1 << 20) && (long long)a.wide_max * 2 * delta <= 2LL * (hi > 0 ? hi : 1)) a.wide_max *= 2;
    if (own_rp) {
        const cudaError_t e = cudaMemcpyAsync(rp_copy, rp, (size_t)(n + 1) * 8, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return sp_fail(e);
        a.rp = rp_copy;
    } else {
        a.rp = rp;
    }
    return partition_arcs(rp, col, w, n, delta, arcs, nlight, biglist, flags + 6, s);
}

// CTAs of the cooperative search launch: 2 per SM (all resident at once).
apsp_status_t grid_size(int* grid) {
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sssp_grid_kernel, kGridThreads, 0);
    if (e != cudaSuccess) return sp_fail(e);
    if (!coop || per_sm < 1) return APSP_EUNSUPPORTED;
    *grid = sms * min(per_sm, 2);
    return APSP_OK;
}

// Test hook state (apsp_debug_inject_grid_timeout), under g_sp_mu.
bool g_grid_inject = false;
unsigned long long g_grid_inject_ns = 0;

// One search from src on a prepared graph into dist.  Blocks on s.
apsp_status_t grid_run(const GridArgs& prepared, int src, int32_t* dist, cudaStream_t s) {
    GridArgs a = prepared;
    a.dist = dist;
    if (g_grid_inject) {
        a.inject = 1;
        a.timeout_ns = g_grid_inject_ns;
        g_grid_inject = false;
    }
    int grid = 0;
    apsp_status_t rc = grid_size(&grid);
    if (rc != APSP_OK) return rc;
    grid_init_kernel<<<grid * 2, 256, 0, s>>>(a, src);
    count_kernel();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (g_sp_timing.enabled) {
        e = cudaEventCreate(&ev[0]);
        if (e == cudaSuccess) e = cudaEventCreate(&ev[1]);
        if (e == cudaSuccess) e = cudaEventRecord(ev[0], s);
        if (e != cudaSuccess) {
            for (cudaEvent_t x : ev)
                if (x) cudaEventDestroy(x);
            return sp_fail(e);
        }
    }
    void* params[] = {&a};
    e = cudaLaunchCooperativeKernel((const void*)sssp_grid_kernel, dim3(grid), dim3(kGridThreads), params, 0, s);
    count_kernel();
    if (e == cudaSuccess && ev[1]) e = cudaEventRecord(ev[1], s);
    if (e == cudaSuccess) {
        grid_finish_kernel<<<grid * 2, 256, 0, s>>>(dist, a.n);
        count_kernel();
        e = cudaGetLastError();
    }
    int err = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&err, &a.ctrl->err, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && ev[1]) {
        float t = 0.f;
        e = cudaEventElapsedTime(&t, ev[0], ev[1]);
        if (e == cudaSuccess) {
            g_sp_timing.search_ms += t;
            g_sp_timing.searches += 1;
        }
    }
    for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
    if (e != cudaSuccess) return sp_fail(e);
    return err ? APSP_ETIMEOUT : APSP_OK;
}

}  // namespace

extern "C" {

apsp_status_t apsp_sssp_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n, int source,
                            int32_t delta, int32_t* dist, apsp_stream_t stream) {
    if (n < 0 || (n > 0 && (row_ptr == nullptr || dist == nullptr)) || (n > 0 && (source < 0 || source >= n)))
        return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    if (reinterpret_cast<uintptr_t>(dist) % 16 != 0) return APSP_EINVAL;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    cudaStream_t s = (cudaStream_t)stream;
    SparseState* st = sp_state();
    if (!st) return APSP_ECUDA;
    long long m = 0;
    apsp_status_t rc = read_m(row_ptr, n, &m, s);
    if (rc != APSP_OK) return rc;
    if (m < 0 || m >= (long long)INT_MAX || (m > 0 && (col_idx == nullptr || w == nullptr))) return APSP_EINVAL;
    rc = grow(st->grid, grid_bytes(n, m, false));
    if (rc != APSP_OK) return rc;
    GridArgs a;
    rc = grid_prepare(row_ptr, col_idx, w, n, m, delta, static_cast<char*>(st->grid.p), false, a, s);
    if (rc != APSP_OK) return rc;
    return grid_run(a, source, dist, s);
}

}  // extern "C"

struct apsp_sssp_graph {
    int device = 0;
    long long m = 0;
    void* buf = nullptr;
    GridArgs a;
};

extern "C" {

apsp_status_t apsp_sssp_graph_create(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n,
                                     int32_t delta, apsp_stream_t stream, apsp_sssp_graph_t* out) {
    if (out == nullptr) return APSP_EINVAL;
    *out = nullptr;
    if (n <= 0 || row_ptr == nullptr) return APSP_EINVAL;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    cudaStream_t s = (cudaStream_t)stream;
    long long m = 0;
    apsp_status_t rc = read_m(row_ptr, n, &m, s);
    if (rc != APSP_OK) return rc;
    if (m < 0 || m >= (long long)INT_MAX || (m > 0 && (col_idx == nullptr || w == nullptr))) return APSP_EINVAL;
    apsp_sssp_graph* g = new (std::nothrow) apsp_sssp_graph;
    if (!g) return APSP_ENOMEM;
    cudaGetDevice(&g->device);
    g->m = m;
    const cudaError_t e = cudaMalloc(&g->buf, grid_bytes(n, m, true));
    if (e != cudaSuccess) {
        cudaGetLastError();
        apsp::set_last_cuda_error((int)e);
        delete g;
        return APSP_ENOMEM;
    }
    rc = grid_prepare(row_ptr, col_idx, w, n, m, delta, static_cast<char*>(g->buf), true, g->a, s);
    if (rc != APSP_OK) {
        cudaStreamSynchronize(s);
        cudaFree(g->buf);
        delete g;
        return rc;
    }
    *out = g;
    return APSP_OK;
}

apsp_status_t apsp_sssp_graph_search(apsp_sssp_graph_t g, int source, int32_t* dist, apsp_stream_t stream) {
    if (g == nullptr || dist == nullptr || source < 0 || source >= g->a.n) return APSP_EINVAL;
    if (reinterpret_cast<uintptr_t>(dist) % 16 != 0) return APSP_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != g->device) return APSP_EINVAL;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    return grid_run(g->a, source, dist, (cudaStream_t)stream);
}

apsp_status_t apsp_sssp_graph_info(apsp_sssp_graph_t g, int* n, long long* m, int32_t* delta) {
    if (g == nullptr) return APSP_EINVAL;
    if (n) *n = g->a.n;
    if (m) *m = g->m;
    if (delta) *delta = g->a.delta;
    return APSP_OK;
}

apsp_status_t apsp_sssp_graph_destroy(apsp_sssp_graph_t g) {
    if (g == nullptr) return APSP_OK;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != g->device) cudaSetDevice(g->device);
    cudaDeviceSynchronize();
    cudaFree(g->buf);
    if (cur != g->device) cudaSetDevice(cur);
    delete g;
    return APSP_OK;
}

apsp_status_t apsp_csr_count_i32(const int32_t* dist, int n, int ld, int64_t* row_ptr, long long* m_out,
                                 apsp_stream_t stream) {
    if (n < 0 || n > APSP_MAX_N || ld < n || row_ptr == nullptr || m_out == nullptr || (n > 0 && dist == nullptr))
        return APSP_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    if (n == 0) {
        const cudaError_t e = cudaMemsetAsync(row_ptr, 0, sizeof(int64_t), s);
        if (e != cudaSuccess) return sp_fail(e);
        *m_out = 0;
        return APSP_OK;
    }
    csr_count_kernel<<<blocks_for_warps(n), 256, 0, s>>>(dist, ld, n, row_ptr);
    scan_kernel<<<1, kScanThreads, 0, s>>>(row_ptr, n);
    {
        std::lock_guard<std::mutex> lock(g_sp_mu);
        count_kernel(2);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    return read_m(row_ptr, n, m_out, s);
}

apsp_status_t apsp_csr_fill_i32(const int32_t* dist, int n, int ld, const int64_t* row_ptr, int32_t* col_idx,
                                int32_t* w, apsp_stream_t stream) {
    if (n < 0 || n > APSP_MAX_N || ld < n ||
        (n > 0 && (dist == nullptr || row_ptr == nullptr || col_idx == nullptr || w == nullptr)))
        return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    csr_fill_kernel<<<blocks_for_warps(n), 256, 0, (cudaStream_t)stream>>>(dist, ld, n, row_ptr, col_idx, w);
    {
        std::lock_guard<std::mutex> lock(g_sp_mu);
        count_kernel();
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sp_fail(e);
    return APSP_OK;
}

apsp_status_t apsp_sssp_delta_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n,
                                  const int32_t* sources, int nsrc, int32_t delta, int32_t* out, int ldo,
                                  apsp_stream_t stream) {
    if (n < 0 || n > APSP_SPARSE_MAX_N || nsrc < 0 || ldo < n) return APSP_EINVAL;
    if (n > 0 && nsrc > 0 && (row_ptr == nullptr || sources == nullptr || out == nullptr)) return APSP_EINVAL;
    if (n == 0 || nsrc == 0) return APSP_OK;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    cudaStream_t s = (cudaStream_t)stream;
    SparseState* st = sp_state();
    if (!st) return APSP_ECUDA;
    long long m = 0;
    apsp_status_t rc = read_m(row_ptr, n, &m, s);
    if (rc != APSP_OK) return rc;
    if (m < 0 || (m > 0 && (col_idx == nullptr || w == nullptr))) return APSP_EINVAL;
    if (m >= (long long)INT_MAX) return APSP_EINVAL;  // arc indices are int32 in the search
    rc = grow(st->work, work_bytes(n, m));
    if (rc != APSP_OK) return rc;
    const Work wk = work_layout(st->work.p, n, m);
    rc = check_row_ptr(row_ptr, n, wk.err, s);
    if (rc != APSP_OK) return rc;
    int lo = 0, hi = 0, bad = 0;
    rc = weight_range(w, col_idx, m, n, wk.range, s, &lo, &hi, &bad);
    if (rc != APSP_OK) return rc;
    if (bad || (m > 0 && (lo < 0 || hi >= kInf))) return APSP_EINVAL;
    if (delta <= 0) delta = default_delta(n, m, hi);
    return launch_sssp(row_ptr, col_idx, w, n, m, sources, nsrc, delta, nullptr, out, ldo, wk, s);
}

apsp_status_t apsp_johnson_csr_i32(const int64_t* row_ptr, const int32_t* col_idx, const int32_t* w, int n,
                                   int32_t delta, int32_t* out, int ld, apsp_stream_t stream) {
    if (n < 0 || n > APSP_SPARSE_MAX_N || ld < n || (n > 0 && (row_ptr == nullptr || out == nullptr)))
        return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    cudaStream_t s = (cudaStream_t)stream;
    SparseState* st = sp_state();
    if (!st) return APSP_ECUDA;
    long long m = 0;
    apsp_status_t rc = read_m(row_ptr, n, &m, s);
    if (rc != APSP_OK) return rc;
    if (m < 0 || (m > 0 && (col_idx == nullptr || w == nullptr))) return APSP_EINVAL;
    if (m >= (long long)INT_MAX) return APSP_EINVAL;  // arc indices are int32 in the search
    rc = grow(st->work, work_bytes(n, m));
    if (rc != APSP_OK) return rc;
    const Work wk = work_layout(st->work.p, n, m);
    rc = check_row_ptr(row_ptr, n, wk.err, s);
    if (rc != APSP_OK) return rc;
    return johnson(row_ptr, col_idx, w, n, m, delta, out, ld, wk, true, s);
}

apsp_status_t apsp_solve_sparse_i32(int32_t* dist, int n, int ld, int32_t delta, apsp_stream_t stream) {
    if (n < 0 || n > APSP_SPARSE_MAX_N || ld < n || (n > 0 && dist == nullptr)) return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    if (!sp_supported_device()) return APSP_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    cudaStream_t s = (cudaStream_t)stream;
    SparseState* st = sp_state();
    if (!st) return APSP_ECUDA;
    long long m = 0;
    apsp_status_t rc = build_csr(dist, n, ld, *st, &m, s);
    if (rc != APSP_OK) return rc;
    rc = grow(st->work, work_bytes(n, m));
    if (rc != APSP_OK) return rc;
    const size_t colb = align256((size_t)(m > 0 ? m : 1) * 4);
    const int64_t* rp = static_cast<const int64_t*>(st->rp.p);
    const int32_t* col = static_cast<const int32_t*>(st->body.p);
    const int32_t* w = reinterpret_cast<const int32_t*>(static_cast<const char*>(st->body.p) + colb);
    // The searches read only the CSR, so they may overwrite dist as they go.
    return johnson(rp, col, w, n, m, delta, dist, ld, work_layout(st->work.p, n, m), false, s);
}

apsp_status_t apsp_debug_inject_grid_timeout(unsigned long long timeout_ns) {
    if (timeout_ns == 0 || timeout_ns > 2000000000ull) return APSP_EINVAL;
    std::lock_guard<std::mutex> lock(g_sp_mu);
    g_grid_inject = true;
    g_grid_inject_ns = timeout_ns;
    return APSP_OK;
}

apsp_status_t apsp_sparse_timing_enable(int enable) {
    std::lock_guard<std::mutex> lock(g_sp_mu);
    g_sp_timing.enabled = enable != 0;
    return APSP_OK;
}

apsp_status_t apsp_sparse_timing_read(double* search_ms, long long* searches, long long* kernels) {
    std::lock_guard<std::mutex> lock(g_sp_mu);
    if (search_ms) *search_ms = g_sp_timing.search_ms;
    if (searches) *searches = g_sp_timing.searches;
    if (kernels) *kernels = g_sp_timing.kernels;
    g_sp_timing.search_ms = 0.0;
    g_sp_timing.searches = 0;
    g_sp_timing.kernels = 0;
    return APSP_OK;
}

apsp_status_t apsp_sparse_release(void) {
    std::lock_guard<std::mutex> lock(g_sp_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    apsp_status_t rc = APSP_OK;
    for (size_t dev = 0; dev < g_sp.size(); ++dev) {
        SparseState& st = g_sp[dev];
        if (!st.rp.p && !st.body.p && !st.work.p && !st.grid.p) continue;
        if (cudaSetDevice((int)dev) != cudaSuccess) {
            rc = APSP_ECUDA;
            continue;
        }
        cudaDeviceSynchronize();
        for (DevBuf* b : {&st.rp, &st.body, &st.work, &st.grid}) {
            if (b->p) cudaFree(b->p);
            b->p = nullptr;
            b->bytes = 0;
        }
    }
    cudaSetDevice(cur);
    return rc;
}

}  // extern "C"
