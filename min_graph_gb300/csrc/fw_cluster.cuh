// Blocked Floyd-Warshall for small matrices inside one thread-block cluster,
// sm_103a.
//
// Same method as the other schedules (thesis page, 1library.co excerpt,
// section 4.6, Algorithms 16-18): rounds over the diagonal blocks, each with
// phase 1 (closure of the primary block), phase 2 (its row and column
// panels) and phase 3 (every other block).  What changes is the scale.  For
// n <= SC_MAX_N the whole matrix (at most 1 MiB) stays in L2, the blocks are
// 32 x 32 instead of 128 x 128, and one cluster of SC_CLUSTER CTAs runs all
// rounds in a single launch.  Its phases meet at hardware cluster barriers
// (barrier.cluster with release/acquire semantics), so no round waits for a
// kernel launch or a flag in memory, and a phase-1 closure costs 32 short
// steps instead of 128.
//
// Lookahead: in phase 3 of round r, CTA 0 first updates block (r+1, r+1)
// and closes it (phase 1 of round r+1) straight from its registers, then
// takes its share of the remaining phase-3 blocks.  A round is thus one
// barrier after phase 2 and one after phase 3.
//
// Data: D is read and written in place in global memory.  Every read of a
// block that another CTA may have written goes to L2 (ld.global.cg), after
// the cluster barrier that orders the write before it.  Entries outside the
// n x n matrix are INF in registers and shared memory and are never stored;
// inputs above INF are clamped on every load.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fw_kernels.cuh"

namespace apsp {

constexpr int SB = 32;            // block edge
constexpr int SC_MAX_N = 512;     // largest n this path takes
constexpr int SC_THREADS = 256;   // 32 rows x 8 groups of 4 columns
constexpr int SC_ASTRIDE = SB + 1;  // padded row of the transposed A block (no bank conflicts)
// Aligned matrices: the CTA works as SC_GROUPS independent groups of SC_GT
// threads, each on its own block product at a time (8 x 8 threads, 4 x 4
// outputs each), with its own cp.async ring of SC_GSTAGES stages and its
// own named barrier.  A stage holds A as copied (row-major, rows padded to
// SC_ARS), B and C; A is then transposed into one of two per-group buffers
// (rows padded to SC_ATS) so that the product reads four rows of a column
// in one 16-byte load.
constexpr int SC_GROUPS = 4;
constexpr int SC_GT = SC_THREADS / SC_GROUPS;  // 64
constexpr int SC_GSTAGES = 3;
constexpr int SC_ARS = SB + 4;
constexpr int SC_ATS = SB + 4;
constexpr int SC_GSTAGE_ELEMS = SB * SC_ARS + 2 * SB * SB;
constexpr int SC_GROUP_ELEMS = 2 * SB * SC_ATS + SC_GSTAGES * SC_GSTAGE_ELEMS;
template <typename T>
constexpr size_t sc_smem_bytes() { return (size_t)SC_GROUPS * SC_GROUP_ELEMS * sizeof(T); }

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

template <typename T> struct SmallBits;
template <> struct SmallBits<int32_t> {
    __device__ static __forceinline__ int32_t from(int x) { return x; }
};
template <> struct SmallBits<float> {
    __device__ static __forceinline__ float from(int x) { return __int_as_float(x); }
};

// Four entries D[row][col..col+3] read from L2 (ld.global.cg), clamped to INF;
// INF outside the n x n matrix.  vec: D 16-byte aligned and ld % 4 == 0.
template <typename T>
__device__ __forceinline__ void sc_load4(const T* __restrict__ D, long long ld, int n, int row, int col,
                                         bool vec, T* o) {
    if (row < n && vec && col + 4 <= n) {
        const int4 v = __ldcg(reinterpret_cast<const int4*>(D + (long long)row * ld + col));
        o[0] = Sem<T>::clamp(SmallBits<T>::from(v.x));
        o[1] = Sem<T>::clamp(SmallBits<T>::from(v.y));
        o[2] = Sem<T>::clamp(SmallBits<T>::from(v.z));
        o[3] = Sem<T>::clamp(SmallBits<T>::from(v.w));
    } else {
        const int* p = reinterpret_cast<const int*>(D + (long long)row * ld);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = (row < n && col + q < n) ? Sem<T>::clamp(SmallBits<T>::from(__ldcg(p + col + q)))
                                            : Sem<T>::inf();
    }
}

// One 32 x 32 block product on the CTA: c (this thread's row i, columns
// j0..j0+3) = min(c, A (x) B) with A transposed in At[k][i] (row stride
// SC_ASTRIDE) and B row-major in Bs[k][j].
template <typename T>
__device__ __forceinline__ void sc_product(T (&c)[4], const T* __restrict__ At, const T* __restrict__ Bs,
                                           int i, int j0) {
#pragma unroll
    for (int k = 0; k < SB; ++k) {
        const T a = At[k * SC_ASTRIDE + i];
        T b[4];
        vload4(Bs + k * SB + j0, b);
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q] = Sem<T>::relax(c[q], a, b[q]);
    }
}

// Closure of the block held in registers across the CTA (Algorithm 16 on a
// 32 x 32 block): at step k every thread needs P[i][k] and P[k][j0..j0+3].
// The owners publish row k+1 and column k+1 into double-buffered shared rows
// right after step k, so each step needs one CTA barrier.  Row and column k
// do not change during step k (P[k][k] is 0, or INF on padding).
template <typename T>
__device__ __forceinline__ void sc_closure(T (&c)[4], T* rowbuf, T* colbuf, int i, int j0) {
    if (i == 0) vstore4(rowbuf + j0, c[0], c[1], c[2], c[3]);
    if (j0 == 0) colbuf[i] = c[0];
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < SB; ++k) {
        const int buf = k & 1;
        const T a = colbuf[buf * SB + i];
        T b[4];
        vload4(rowbuf + buf * SB + j0, b);
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q] = Sem<T>::relax(c[q], a, b[q]);
        if (k + 1 < SB) {
            const int k1 = k + 1;
            if (i == k1) vstore4(rowbuf + (buf ^ 1) * SB + j0, c[0], c[1], c[2], c[3]);
            if ((k1 >> 2) == (j0 >> 2)) {
                const int q = k1 & 3;
                colbuf[(buf ^ 1) * SB + i] = q == 0 ? c[0] : q == 1 ? c[1] : q == 2 ? c[2] : c[3];
            }
        }
        __syncthreads();
    }
}

template <typename T>
__device__ __forceinline__ void sc_store4(T* __restrict__ D, long long ld, int n, int row, int col, bool vec,
                                          const T (&c)[4]) {
    gstore4(D, ld, n, row, col, vec, c[0], c[1], c[2], c[3]);
}

// The operands of one block product, fetched into registers ahead of use.
template <typename T>
struct ScFetch {
    T a[4], b[4], c[4];
};

template <typename T>
__device__ __forceinline__ void sc_fetch(ScFetch<T>& f, const T* __restrict__ D, long long ld, int n, bool vec,
                                         int arow, int acol, int brow, int bcol, int crow, int ccol) {
    sc_load4(D, ld, n, arow, acol, vec, f.a);
    sc_load4(D, ld, n, brow, bcol, vec, f.b);
    sc_load4(D, ld, n, crow, ccol, vec, f.c);
}

// Put fetched operands into shared memory: A transposed, B row-major.
template <typename T>
__device__ __forceinline__ void sc_stage(const ScFetch<T>& f, T* At, T* Bs, int i, int j0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) At[(j0 + q) * SC_ASTRIDE + i] = f.a[q];
    vstore4(Bs + i * SB + j0, f.b[0], f.b[1], f.b[2], f.b[3]);
}

// 16 bytes global -> shared through L2 only (cp.async.cg), of which the
// first `bytes` are read and the rest zero-filled.
__device__ __forceinline__ void sc_cp16(uint32_t dst, const void* src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// This thread's share of one block copy: the 16-byte chunk at row t / 8,
// columns 4 (t % 8) .. + 3, of the SB x SB block whose corner is (row0, col0).
template <typename T>
__device__ __forceinline__ void sc_issue_chunk(uint32_t dst, const T* __restrict__ D, long long ld, int n,
                                               int row, int col) {
    int bytes = 0;
    const T* src = D;
    if (row < n && col < n) {
        bytes = (n - col >= 4 ? 4 : n - col) * (int)sizeof(T);
        src = D + (long long)row * ld + col;
    }
    sc_cp16(dst, src, bytes);
}

// After this thread's copy of its chunk has landed: entries outside the
// matrix become INF, inputs above INF are clamped.
template <typename T>
__device__ __forceinline__ void sc_fix_chunk(T* p, int n, int row, int col) {
    T v[4];
    vload4(p, v);
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = (row < n && col + q < n) ? Sem<T>::clamp(v[q]) : Sem<T>::inf();
    vstore4(p, v[0], v[1], v[2], v[3]);
}

// Work items of one phase, spread over the cluster's CTAs.
//   phase 2 of round r: q in [0, 2(nbs-1)): row blocks (r, J != r), then
//     column blocks (I != r, r).  Row block: A = P (transposed), B = the
//     block itself.  Column block: A = the block itself (transposed), B = P.
//   phase 3 of round r: q in [0, (nbs-1)^2): block (I, J), I, J != r, row-major
//     over the others.  A = D[I, r] (transposed), B = D[r, J].
struct ScBlock {
    int ci, cj;  // the output block
    int ai, aj;  // A operand block (used transposed)
    int bi, bj;  // B operand block
};

__device__ __forceinline__ ScBlock sc_p2_block(int q, int r, int nbs) {
    ScBlock b;
    if (q < nbs - 1) {
        const int J = q + (q >= r ? 1 : 0);
        b.ci = r; b.cj = J; b.ai = r; b.aj = r; b.bi = r; b.bj = J;
    } else {
        const int qq = q - (nbs - 1);
        const int I = qq + (qq >= r ? 1 : 0);
        b.ci = I; b.cj = r; b.ai = I; b.aj = r; b.bi = r; b.bj = r;
    }
    return b;
}

__device__ __forceinline__ ScBlock sc_p3_block(int q, int r, int nbs) {
    const int m = nbs - 1;
    const int ti = q / m, tj = q - ti * m;
    ScBlock b;
    b.ci = ti + (ti >= r ? 1 : 0);
    b.cj = tj + (tj >= r ? 1 : 0);
    b.ai = b.ci; b.aj = r; b.bi = r; b.bj = b.cj;
    return b;
}

// The t-th phase-3 block (in run order) of CTA `rank` of `ncta` in round r,
// as an index into sc_p3_block's row-major enumeration, or -1 when the CTA
// has no more.  With lookahead (`look`), CTA 0 takes only the block that
// becomes (r+1, r+1), which it then closes with all its threads; the other
// CTAs share the rest round-robin.  Without, all CTAs share all blocks.
// Every block goes to exactly one CTA.
__host__ __device__ inline int sc_p3_elem(int t, int r, int nbs, int rank, int ncta, bool look) {
    const int m = nbs - 1;
    const int total = m * m;
    if (!look) {
        const int e = rank + t * ncta;
        return e < total ? e : -1;
    }
    const int diag = r * m + r;  // (r+1, r+1) is (r, r) among the others
    if (rank == 0 && t == 0) return diag;
    const int o = ncta > 1 ? ncta - 1 : 1;  // CTAs sharing the rest
    int e;
    if (ncta > 1) {
        if (rank == 0) return -1;
        e = (rank - 1) + t * o;
    } else {
        e = t - 1;
    }
    if (e >= total - 1) return -1;
    return e >= diag ? e + 1 : e;
}

__device__ __forceinline__ ScBlock sc_none() {
    ScBlock b;
    b.ci = -1; b.cj = b.ai = b.aj = b.bi = b.bj = 0;
    return b;
}

__device__ __forceinline__ void sc_group_bar(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(SC_GT) : "memory");
}

// v (rows i0..i0+3, columns j0..j0+3 of the block) = min(v, A (x) B), A
// transposed in At (row stride SC_ATS), B row-major.
template <typename T>
__device__ __forceinline__ void sc_product16(T (&v)[4][4], const T* __restrict__ At, const T* __restrict__ Bs,
                                             int i0, int j0) {
#pragma unroll 8
    for (int k = 0; k < SB; ++k) {
        T a[4], b[4];
        vload4(At + k * SC_ATS + i0, a);
        vload4(Bs + k * SB + j0, b);
#pragma unroll
        for (int ri = 0; ri < 4; ++ri)
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) v[ri][ci] = Sem<T>::relax(v[ri][ci], a[ri], b[ci]);
    }
}

// Closure of the block held by one group (4 x 4 per thread), as sc_closure
// with the group's barrier: row k+1 and column k+1 are published right after
// step k into double-buffered shared rows.
template <typename T>
__device__ __forceinline__ void sc_closure16(T (&v)[4][4], T* rowbuf, T* colbuf, int i0, int j0, int bar) {
    if (i0 == 0) vstore4(rowbuf + j0, v[0][0], v[0][1], v[0][2], v[0][3]);
    if (j0 == 0) vstore4(colbuf + i0, v[0][0], v[1][0], v[2][0], v[3][0]);
    sc_group_bar(bar);
#pragma unroll 2
    for (int kc = 0; kc < SB / 4; ++kc) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int k = kc * 4 + kk;
            const int buf = kk & 1;  // == k & 1
            T a[4], b[4];
            vload4(colbuf + buf * SB + i0, a);
            vload4(rowbuf + buf * SB + j0, b);
#pragma unroll
            for (int ri = 0; ri < 4; ++ri)
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) v[ri][ci] = Sem<T>::relax(v[ri][ci], a[ri], b[ci]);
            if (k + 1 < SB) {
                const int rr = (kk + 1) & 3;            // register row / column of k + 1
                const int grp = kk < 3 ? kc : kc + 1;   // its 4-wide group
                if ((i0 >> 2) == grp)
                    vstore4(rowbuf + (buf ^ 1) * SB + j0, v[rr][0], v[rr][1], v[rr][2], v[rr][3]);
                if ((j0 >> 2) == grp)
                    vstore4(colbuf + (buf ^ 1) * SB + i0, v[0][rr], v[1][rr], v[2][rr], v[3][rr]);
            }
            sc_group_bar(bar);
        }
    }
}

// One group's share of a phase (aligned D): get(u) gives the group's u-th
// block (ci < 0: no more).  Each thread copies, and once they have landed
// fixes up, rows rc + 8m (m = 0..3), columns j0..j0+3 of A, B and C; it
// transposes its A chunks.  With close_first, the first block's result is
// closed (phase 1 of the next round) before it is stored.
template <typename T, typename Get>
__device__ __forceinline__ void sc_run_group(T* __restrict__ D, long long ld, int n, T* gmem, Get get,
                                             bool close_first, bool raw, T* rowbuf, T* colbuf, int tg, int bar) {
    const int rc = tg >> 3, j0 = (tg & 7) * 4;  // copy chunk row (of each 8) and column
    const int i0 = rc * 4;                      // output rows i0..i0+3
    T* const at0 = gmem;
    T* const at1 = gmem + SB * SC_ATS;
    T* stage0 = gmem + 2 * SB * SC_ATS;
    auto issue = [&](const ScBlock& b, int st) {
        T* base = stage0 + st * SC_GSTAGE_ELEMS;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int row = rc + 8 * m;
            sc_issue_chunk(smem_u32(base + row * SC_ARS + j0), D, ld, n, b.ai * SB + row, b.aj * SB + j0);
            sc_issue_chunk(smem_u32(base + SB * SC_ARS + row * SB + j0), D, ld, n, b.bi * SB + row, b.bj * SB + j0);
            sc_issue_chunk(smem_u32(base + SB * SC_ARS + SB * SB + row * SB + j0), D, ld, n, b.ci * SB + row,
                           b.cj * SB + j0);
        }
    };
    for (int q = 0; q < SC_GSTAGES - 1; ++q) {
        const ScBlock b = get(q);
        if (b.ci >= 0) issue(b, q);
        cp_async_commit();  // one group per slot, empty or not
    }
    for (int u = 0;; ++u) {
        const ScBlock b = get(u);
        if (b.ci < 0) break;
        T* As = stage0 + (u % SC_GSTAGES) * SC_GSTAGE_ELEMS;
        T* Bs = As + SB * SC_ARS;
        T* Cs = Bs + SB * SB;
        T* At = (u & 1) ? at1 : at0;
        cp_async_wait<SC_GSTAGES - 2>();  // this thread's chunks of block u have landed
        // Clamp inputs above INF while some block may still hold them (the
        // first round reads every block once and stores it clamped); set
        // entries outside the matrix to INF in the ragged last blocks.
        const bool fa = raw || (b.ai + 1) * SB > n || (b.aj + 1) * SB > n;
        const bool fb = raw || (b.bi + 1) * SB > n || (b.bj + 1) * SB > n;
        const bool fc = raw || (b.ci + 1) * SB > n || (b.cj + 1) * SB > n;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int row = rc + 8 * m;
            if (fa) sc_fix_chunk(As + row * SC_ARS + j0, n, b.ai * SB + row, b.aj * SB + j0);
            T x[4];
            vload4(As + row * SC_ARS + j0, x);
#pragma unroll
            for (int q = 0; q < 4; ++q) At[(j0 + q) * SC_ATS + row] = x[q];
            if (fb) sc_fix_chunk(Bs + row * SB + j0, n, b.bi * SB + row, b.bj * SB + j0);
            if (fc) sc_fix_chunk(Cs + row * SB + j0, n, b.ci * SB + row, b.cj * SB + j0);
        }
        // block u is complete in shared memory; block u - 1's stage and
        // transposed A are free
        sc_group_bar(bar);
        T v[4][4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) vload4(Cs + (i0 + ri) * SB + j0, v[ri]);
        const ScBlock bn = get(u + SC_GSTAGES - 1);
        if (bn.ci >= 0) issue(bn, (u + SC_GSTAGES - 1) % SC_GSTAGES);
        cp_async_commit();
        sc_product16(v, At, Bs, i0, j0);
        if (close_first && u == 0) sc_closure16(v, rowbuf, colbuf, i0, j0, bar);
#pragma unroll
        for (int ri = 0; ri < 4; ++ri)
            gstore4(D, ld, n, b.ci * SB + i0 + ri, b.cj * SB + j0, true, v[ri][0], v[ri][1], v[ri][2], v[ri][3]);
    }
    cp_async_wait<0>();
}

template <typename T>
__global__ void __launch_bounds__(SC_THREADS, 1)
fw_cluster_small(T* __restrict__ D, long long ld, int n, int vec) {
    __shared__ __align__(16) T At[SB * SC_ASTRIDE];
    __shared__ __align__(16) T Bs[SB * SB];
    __shared__ __align__(16) T rowbuf[2 * SB];
    __shared__ __align__(16) T colbuf[2 * SB];
    const int t = threadIdx.x;
    const int i = t >> 3, j0 = (t & 7) * 4;
    const int rank = (int)cluster_ctarank();
    const int ncta = (int)cluster_nctarank();
    const int nbs = (n + SB - 1) / SB;
    const bool vv = vec != 0;

    // Phase 1 of round 0.
    if (rank == 0) {
        T c[4];
        sc_load4(D, ld, n, i, j0, vv, c);
        sc_closure(c, rowbuf, colbuf, i, j0);
        sc_store4(D, ld, n, i, j0, vv, c);
    }
    cluster_barrier();

    if (vv) {
        extern __shared__ __align__(16) unsigned char sc_ring_raw[];
        const int g = t / SC_GT, tg = t % SC_GT;
        T* gmem = reinterpret_cast<T*>(sc_ring_raw) + (size_t)g * SC_GROUP_ELEMS;
        const int bar = 1 + g;  // named barrier of this group (0 is __syncthreads)
        // This CTA's blocks of the current phase, decoded once per phase, one
        // thread each (the decoding divides); -1 ends the list.  Group g
        // takes entries g, g + SC_GROUPS, ...
        __shared__ int list[SC_THREADS];
        for (int r = 0; r < nbs; ++r) {
            // phase 2, round r
            {
                const int q = rank + t * ncta;
                list[t] = q < 2 * (nbs - 1) ? q : -1;
            }
            __syncthreads();
            sc_run_group(D, ld, n, gmem,
                         [&](int u) {
                             const int e = g + u * SC_GROUPS;
                             return e < SC_THREADS && list[e] >= 0 ? sc_p2_block(list[e], r, nbs) : sc_none();
                         },
                         false, r == 0, rowbuf, colbuf, tg, bar);
            __syncthreads();
            cluster_barrier();
            if (nbs == 1) break;
            // phase 3, round r (+ phase 1 of round r + 1 on CTA 0)
            const bool look = r + 1 < nbs;
            const int m = nbs - 1;
            if (look && rank == 0 && ncta > 1) {
                // CTA 0: block (r+1, r+1) on all threads, then its closure
                const ScBlock bk = sc_p3_block(r * m + r, r, nbs);
                ScFetch<T> f;
                sc_fetch(f, D, ld, n, vv, bk.ai * SB + i, bk.aj * SB + j0, bk.bi * SB + i, bk.bj * SB + j0,
                         bk.ci * SB + i, bk.cj * SB + j0);
                sc_stage(f, At, Bs, i, j0);
                T c[4] = {f.c[0], f.c[1], f.c[2], f.c[3]};
                __syncthreads();
                sc_product(c, At, Bs, i, j0);
                sc_closure(c, rowbuf, colbuf, i, j0);
                sc_store4(D, ld, n, bk.ci * SB + i, bk.cj * SB + j0, vv, c);
                __syncthreads();
                cluster_barrier();
                continue;
            }
            list[t] = sc_p3_elem(t, r, nbs, rank, ncta, look);
            __syncthreads();
            sc_run_group(D, ld, n, gmem,
                         [&](int u) {
                             const int e = g + u * SC_GROUPS;
                             if (e >= SC_THREADS || list[e] < 0) return sc_none();
                             const int x = list[e];
                             const int ti = x / m;  // m <= 15
                             const int tj = x - ti * m;
                             ScBlock bk;
                             bk.ci = ti + (ti >= r ? 1 : 0);
                             bk.cj = tj + (tj >= r ? 1 : 0);
                             bk.ai = bk.ci; bk.aj = r; bk.bi = r; bk.bj = bk.cj;
                             return bk;
                         },
                         look && rank == 0 && g == 0, r == 0, rowbuf, colbuf, tg, bar);  // (one CTA)
            __syncthreads();
            cluster_barrier();
        }
        return;
    }

    // Unaligned matrices: operands through registers, one block ahead.
    for (int r = 0; r < nbs; ++r) {
        // ------------------------------------------------ phase 2, round r
        for (int q = rank; q < 2 * (nbs - 1); q += ncta) {
            const ScBlock bk = sc_p2_block(q, r, nbs);
            ScFetch<T> f;
            sc_fetch(f, D, ld, n, vv, bk.ai * SB + i, bk.aj * SB + j0, bk.bi * SB + i, bk.bj * SB + j0,
                     bk.ci * SB + i, bk.cj * SB + j0);
            __syncthreads();  // the previous block's shared operands have been read
            sc_stage(f, At, Bs, i, j0);
            __syncthreads();
            T c[4] = {f.c[0], f.c[1], f.c[2], f.c[3]};
            sc_product(c, At, Bs, i, j0);
            sc_store4(D, ld, n, bk.ci * SB + i, bk.cj * SB + j0, vv, c);
        }
        cluster_barrier();
        if (nbs == 1) break;
        // ------------------------------------------------ phase 3, round r
        // (+ phase 1 of round r + 1 on CTA 0)
        const bool look = r + 1 < nbs;
        ScFetch<T> nx;
        int qn = sc_p3_elem(0, r, nbs, rank, ncta, look);
        if (qn >= 0) {
            const ScBlock bk = sc_p3_block(qn, r, nbs);
            sc_fetch(nx, D, ld, n, vv, bk.ai * SB + i, bk.aj * SB + j0, bk.bi * SB + i, bk.bj * SB + j0,
                     bk.ci * SB + i, bk.cj * SB + j0);
        }
        for (int tt = 0; qn >= 0; ++tt) {
            const int q = qn;
            const ScBlock bk = sc_p3_block(q, r, nbs);
            __syncthreads();
            sc_stage(nx, At, Bs, i, j0);
            T c[4] = {nx.c[0], nx.c[1], nx.c[2], nx.c[3]};
            __syncthreads();
            // fetch the next block while this one computes
            qn = sc_p3_elem(tt + 1, r, nbs, rank, ncta, look);
            if (qn >= 0) {
                const ScBlock bn = sc_p3_block(qn, r, nbs);
                sc_fetch(nx, D, ld, n, vv, bn.ai * SB + i, bn.aj * SB + j0, bn.bi * SB + i, bn.bj * SB + j0,
                         bn.ci * SB + i, bn.cj * SB + j0);
            }
            sc_product(c, At, Bs, i, j0);
            if (look && rank == 0 && tt == 0) {
                // block (r+1, r+1) is final for round r: close it (phase 1 of r+1)
                sc_closure(c, rowbuf, colbuf, i, j0);
            }
            sc_store4(D, ld, n, bk.ci * SB + i, bk.cj * SB + j0, vv, c);
        }
        cluster_barrier();
    }
}

}  // namespace apsp
