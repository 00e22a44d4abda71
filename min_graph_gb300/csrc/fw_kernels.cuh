// Blocked Floyd-Warshall kernels for sm_103a.
//
// Method: Katz & Kider's blocked Floyd-Warshall as described on the thesis
// page (1library.co excerpt, section 4.6, Algorithms 16-18).  The n x n
// matrix is cut into TB x TB tiles and processed in rounds.  Round r has the
// primary tile K = [r*TB, (r+1)*TB) and three phases:
//   phase 1: Floyd-Warshall closure of D[K,K] (one CTA).
//   phase 2: row panel D[K,J] <- min(D[K,J], P (x) D[K,J]) and column panel
//            D[I,K] <- min(D[I,K], D[I,K] (x) P), where P = closed D[K,K] and
//            (x) is the min-plus product.
//   phase 3: every other tile D[I,J] <- min(D[I,J], D[I,K] (x) D[K,J]).
// The page's tile is 16 x 16 and its phase 2 runs the k-loop in place.  Here
// the tile is 128 x 128, and phase 2 is written as a min-plus product with
// the already-closed primary tile.  That gives the same distances: the page's
// in-place loop over k in K computes exactly this product.
//
// Phases 2 and 3 share one register-blocked tile product (mm_slab): 256
// threads, each holding an 8 x 8 block of the 128 x 128 output in registers.
// The A operand is read from shared memory k-major (As[k][i]) and the B
// operand row-major (Bs[k][j]), each 4 consecutive entries at a time.  The
// inner step is the fused integer add-min (__viaddmin_s32), or fminf of an
// IEEE sum for fp32.
//
// Phase 3 reads both panels from a compact workspace copy that phase 2
// writes (row panel as is, column panel transposed), so its k-slabs are
// plain contiguous rows that cp.async streams into shared memory.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace apsp {

constexpr int TB = 128;            // round block = CTA tile edge
constexpr int P1_THREADS = 512;    // phase 1: 128 rows x 4 quarters
constexpr int MM_THREADS = 256;    // phases 2 and 3
constexpr int KS = 32;             // phase 3 k-slab depth
constexpr int P3_STAGES = 3;       // phase 3 shared-memory ring
constexpr int P1_QPAD = 36;        // phase 1 row buffer quarter stride (bank spread)

template <typename T> struct Sem;

template <> struct Sem<int32_t> {
    static constexpr int32_t kInf = 0x3FFFFFFF;
    __device__ static __forceinline__ int32_t inf() { return kInf; }
    __device__ static __forceinline__ int32_t clamp(int32_t x) { return min(x, kInf); }
    // min(a + b, acc); a, b <= INF so a + b <= 2*INF < 2^31.
    __device__ static __forceinline__ int32_t relax(int32_t acc, int32_t a, int32_t b) {
        return __viaddmin_s32(a, b, acc);
    }
};

template <> struct Sem<float> {
    __device__ static __forceinline__ float inf() { return __int_as_float(0x7f800000); }
    __device__ static __forceinline__ float clamp(float x) { return x; }
    __device__ static __forceinline__ float relax(float acc, float a, float b) {
        return fminf(acc, __fadd_rn(a, b));
    }
};

// 16-byte vector of four T, through a generic pointer (global or shared).
template <typename T> struct V4;
template <> struct V4<int32_t> { using t = int4; };
template <> struct V4<float> { using t = float4; };

template <typename T>
__device__ __forceinline__ void vload4(const T* p, T* o) {
    const typename V4<T>::t v = *reinterpret_cast<const typename V4<T>::t*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}

template <typename T>
__device__ __forceinline__ void vstore4(T* p, T a, T b, T c, T d) {
    typename V4<T>::t v;
    v.x = a; v.y = b; v.z = c; v.w = d;
    *reinterpret_cast<typename V4<T>::t*>(p) = v;
}

// Four consecutive entries D[row][col..col+3], INF outside the n x n matrix,
// clamped to INF.  vec: base 16-byte aligned and ld % 4 == 0 (col % 4 == 0
// always holds here).
template <typename T>
__device__ __forceinline__ void gload4(const T* __restrict__ D, long long ld, int n, int row,
                                       int col, bool vec, T* o) {
    if (row < n && vec && col + 4 <= n) {
        const typename V4<T>::t v =
            *reinterpret_cast<const typename V4<T>::t*>(D + (long long)row * ld + col);
        o[0] = Sem<T>::clamp(v.x); o[1] = Sem<T>::clamp(v.y);
        o[2] = Sem<T>::clamp(v.z); o[3] = Sem<T>::clamp(v.w);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = (row < n && col + q < n) ? Sem<T>::clamp(D[(long long)row * ld + col + q])
                                            : Sem<T>::inf();
    }
}

// Store four consecutive entries, skipping anything outside the n x n matrix.
template <typename T>
__device__ __forceinline__ void gstore4(T* __restrict__ D, long long ld, int n, int row, int col,
                                        bool vec, T a, T b, T c, T d) {
    if (row >= n) return;
    if (vec && col + 4 <= n) {
        vstore4(D + (long long)row * ld + col, a, b, c, d);
    } else {
        T* p = D + (long long)row * ld + col;
        if (col + 0 < n) p[0] = a;
        if (col + 1 < n) p[1] = b;
        if (col + 2 < n) p[2] = c;
        if (col + 3 < n) p[3] = d;
    }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Thread layout of the 128 x 128 tile product: 8 warps as 4 (rows) x 2
// (cols), each warp 32 x 64; inside a warp 4 x 8 lanes, each lane owning
// rows {rA0..rA0+3, rA1..rA1+3} and cols {cB0..cB0+3, cB1..cB1+3}.  For a
// fixed k the lanes of a warp read 4 distinct 16-byte A chunks and 8 distinct
// B chunks, all within one shared-memory row: one wavefront each, no bank
// conflicts.
struct MMLayout {
    int rA0, rA1, cB0, cB1;
    __device__ __forceinline__ explicit MMLayout(int tid) {
        const int w = tid >> 5, lane = tid & 31;
        const int wr = w >> 1, wc = w & 1;
        const int tr = lane >> 3, tc = lane & 7;
        rA0 = wr * 32 + tr * 4;
        rA1 = rA0 + 16;
        cB0 = wc * 64 + tc * 4;
        cB1 = cB0 + 32;
    }
    __device__ __forceinline__ int row(int ri) const { return ri < 4 ? rA0 + ri : rA1 + (ri - 4); }
    __device__ __forceinline__ int col(int ci) const { return ci < 4 ? cB0 + ci : cB1 + (ci - 4); }
};

// acc[i][j] = min(acc[i][j], min_k As[k][i] + Bs[k][j]) over k in [0, KLEN).
// Fragments for step k+1 are loaded while step k computes (two register
// sets), which hides shared-memory latency without letting the compiler
// hoist loads further ahead than the register budget allows.
template <typename T, int KLEN, int UNROLL>
__device__ __forceinline__ void mm_slab(T (&acc)[8][8], const T* __restrict__ As,
                                        const T* __restrict__ Bs, const MMLayout& L) {
    static_assert(UNROLL % 2 == 0 && KLEN % UNROLL == 0, "even unroll");
    T a[2][8], b[2][8];
    vload4(As + L.rA0, a[0]);
    vload4(As + L.rA1, a[0] + 4);
    vload4(Bs + L.cB0, b[0]);
    vload4(Bs + L.cB1, b[0] + 4);
#pragma unroll UNROLL
    for (int k = 0; k < KLEN; ++k) {
        const int cur = k & 1, nxt = cur ^ 1;
        if (k + 1 < KLEN) {
            vload4(As + (k + 1) * TB + L.rA0, a[nxt]);
            vload4(As + (k + 1) * TB + L.rA1, a[nxt] + 4);
            vload4(Bs + (k + 1) * TB + L.cB0, b[nxt]);
            vload4(Bs + (k + 1) * TB + L.cB1, b[nxt] + 4);
        }
#pragma unroll
        for (int ri = 0; ri < 8; ++ri)
#pragma unroll
            for (int ci = 0; ci < 8; ++ci)
                acc[ri][ci] = Sem<T>::relax(acc[ri][ci], a[cur][ri], b[cur][ci]);
    }
}

// ----------------------------------------------------------------- phase 1
//
// Closure of the primary tile P = D[K,K] (Algorithm 16 of the thesis page:
// standard Floyd-Warshall on the primary block, in shared memory, one
// block).  Thread t owns row i = t/4 and the 32 columns of quarter q = t%4 in
// registers.  At step k every thread needs P[i][k] and row k.  Their owners
// publish them into a double-buffered shared row/column buffer after step
// k-1, so each step needs one barrier.  Row k and column k do not change
// during step k because P[k][k] >= 0.  The closed tile goes back to D and
// into the workspace as prim (row-major) and primT (transposed), which
// phase 2 reads.
template <typename T>
__global__ void __launch_bounds__(P1_THREADS, 1)
fw_phase1_diag(T* __restrict__ D, long long ld, int n, int r, T* __restrict__ prim,
               T* __restrict__ primT, int vec) {
    __shared__ __align__(16) T rowbuf[2][4 * P1_QPAD];
    __shared__ __align__(16) T colbuf[2][TB];
    const int t = threadIdx.x, i = t >> 2, q = t & 3;
    const int k0 = r * TB;
    T v[32];
#pragma unroll
    for (int m = 0; m < 8; ++m) gload4(D, ld, n, k0 + i, k0 + q * 32 + 4 * m, vec != 0, v + 4 * m);

    if (i == 0) {
#pragma unroll
        for (int c = 0; c < 32; ++c) rowbuf[0][q * P1_QPAD + c] = v[c];
    }
    if (q == 0) colbuf[0][i] = v[0];
    __syncthreads();

    for (int kc = 0; kc < 4; ++kc) {
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
            const int k = kc * 32 + kk;
            const int buf = kk & 1;  // == k & 1
            const T a = colbuf[buf][i];
            T b[32];
#pragma unroll
            for (int m = 0; m < 8; ++m) vload4(&rowbuf[buf][q * P1_QPAD + 4 * m], b + 4 * m);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = Sem<T>::relax(v[c], a, b[c]);
            if (k + 1 < TB) {
                if (i == k + 1) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) rowbuf[buf ^ 1][q * P1_QPAD + c] = v[c];
                }
                if (kk < 31) {
                    if (q == kc) colbuf[buf ^ 1][i] = v[(kk + 1) & 31];
                } else {
                    if (q == kc + 1) colbuf[buf ^ 1][i] = v[0];
                }
                __syncthreads();
            }
        }
    }

#pragma unroll
    for (int m = 0; m < 8; ++m)
        gstore4(D, ld, n, k0 + i, k0 + q * 32 + 4 * m, vec != 0, v[4 * m], v[4 * m + 1],
                v[4 * m + 2], v[4 * m + 3]);
#pragma unroll
    for (int m = 0; m < 8; ++m)
        vstore4(prim + i * TB + q * 32 + 4 * m, v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
#pragma unroll
    for (int c = 0; c < 32; ++c) primT[(q * 32 + c) * TB + i] = v[c];
}

// ----------------------------------------------------------------- phase 2
//
// Row and column panels of the primary tile (Algorithm 17 of the thesis
// page, grid (nb-1, 2): y = 0 row panel, y = 1 column panel; blockIdx.x
// skips the primary tile the way the page's skipPrimaryBlock map does).
//   row panel tile (K,J):    new = min(old, P (x) old)  -> As = P^T, Bs = old
//   column panel tile (I,K): new = min(old, old (x) P)  -> As = old^T, Bs = P
// The result goes to D and to the workspace panel that phase 3 reads: rowp
// (TB x npad) as is, colpT (TB x npad) transposed.
template <typename T>
__global__ void __launch_bounds__(MM_THREADS, 1)
fw_phase2_panels(T* __restrict__ D, long long ld, int n, int r, T* __restrict__ rowp,
                 T* __restrict__ colpT, const T* __restrict__ prim, const T* __restrict__ primT,
                 int npad, int vec) {
    extern __shared__ __align__(128) unsigned char p2_smem[];
    T* As = reinterpret_cast<T*>(p2_smem);
    T* Bs = As + TB * TB;
    const int tid = threadIdx.x;
    const int bx = blockIdx.x;
    const int other = bx + (bx >= r ? 1 : 0);
    const int k0 = r * TB, t0 = other * TB;
    const bool is_row = (blockIdx.y == 0);
    const MMLayout L(tid);
    T acc[8][8];

    if (is_row) {
        for (int c = tid; c < TB * TB / 4; c += MM_THREADS) {
            const int kk = c >> 5, qq = (c & 31) * 4;
            T x[4];
            vload4(primT + kk * TB + qq, x);
            vstore4(As + kk * TB + qq, x[0], x[1], x[2], x[3]);
            gload4(D, ld, n, k0 + kk, t0 + qq, vec != 0, x);
            vstore4(Bs + kk * TB + qq, x[0], x[1], x[2], x[3]);
        }
        __syncthreads();
#pragma unroll
        for (int ri = 0; ri < 8; ++ri)
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = Bs[L.row(ri) * TB + L.col(ci)];
    } else {
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            gload4(D, ld, n, t0 + L.row(ri), k0 + L.cB0, vec != 0, &acc[ri][0]);
            gload4(D, ld, n, t0 + L.row(ri), k0 + L.cB1, vec != 0, &acc[ri][4]);
        }
        // transpose through registers: As[k][i] = old[i][k]
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
            const int k = L.col(ci);
            vstore4(As + k * TB + L.rA0, acc[0][ci], acc[1][ci], acc[2][ci], acc[3][ci]);
            vstore4(As + k * TB + L.rA1, acc[4][ci], acc[5][ci], acc[6][ci], acc[7][ci]);
        }
        for (int c = tid; c < TB * TB / 4; c += MM_THREADS) {
            const int kk = c >> 5, qq = (c & 31) * 4;
            T x[4];
            vload4(prim + kk * TB + qq, x);
            vstore4(Bs + kk * TB + qq, x[0], x[1], x[2], x[3]);
        }
        __syncthreads();
    }

    mm_slab<T, TB, 4>(acc, As, Bs, L);

    if (is_row) {
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            const int i = L.row(ri);
            gstore4(D, ld, n, k0 + i, t0 + L.cB0, vec != 0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            gstore4(D, ld, n, k0 + i, t0 + L.cB1, vec != 0, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
            vstore4(rowp + (long long)i * npad + t0 + L.cB0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            vstore4(rowp + (long long)i * npad + t0 + L.cB1, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
        }
    } else {
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            const int i = L.row(ri);
            gstore4(D, ld, n, t0 + i, k0 + L.cB0, vec != 0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            gstore4(D, ld, n, t0 + i, k0 + L.cB1, vec != 0, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
        }
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
            const int k = L.col(ci);
            vstore4(colpT + (long long)k * npad + t0 + L.rA0, acc[0][ci], acc[1][ci], acc[2][ci], acc[3][ci]);
            vstore4(colpT + (long long)k * npad + t0 + L.rA1, acc[4][ci], acc[5][ci], acc[6][ci], acc[7][ci]);
        }
    }
}

// ----------------------------------------------------------------- phase 3
//
// Every tile (I,J) with I != K and J != K (Algorithm 18 of the thesis page,
// grid (nb-1)^2 with the primary row and column skipped):
//   D[I,J] <- min(D[I,J], D[I,K] (x) D[K,J]).
// The panels are read-only in this phase, so k can go in any order.  The
// panels come from the workspace (colpT gives As[k][i], rowp gives Bs[k][j])
// in KS-deep slabs through a P3_STAGES-deep cp.async ring.  The C tile goes
// straight from global memory into the accumulators, and its load overlaps
// the first slabs' copies.
template <typename T>
__global__ void __launch_bounds__(MM_THREADS, 2)
fw_phase3_minplus(T* __restrict__ D, long long ld, int n, int r, int nbm1,
                  const T* __restrict__ rowp, const T* __restrict__ colpT, int npad, int vec) {
    extern __shared__ __align__(128) unsigned char p3_smem[];
    T* sm = reinterpret_cast<T*>(p3_smem);
    const int tid = threadIdx.x;
    const int ti = blockIdx.x / nbm1, tj = blockIdx.x - ti * nbm1;
    const int I = ti + (ti >= r ? 1 : 0), J = tj + (tj >= r ? 1 : 0);
    const int row0 = I * TB, col0 = J * TB;
    const MMLayout L(tid);
    constexpr int NSLAB = TB / KS;
    constexpr int SLAB = KS * TB;  // elements per operand slab

    // Each thread copies the 16-byte chunks c = tid + m * MM_THREADS of a
    // slab: row kk = c / 32, column 4 * (c % 32).  Offsets stay 32-bit.
    const unsigned sm_base = static_cast<unsigned>(__cvta_generic_to_shared(sm));
    const unsigned my_sm = ((tid >> 5) * TB + (tid & 31) * 4) * 4;
    const unsigned my_g = (tid >> 5) * npad + (tid & 31) * 4;
    const unsigned row_step_g = (MM_THREADS / 32) * npad;
    auto issue = [&](int s, int st) {
        const unsigned sa = sm_base + st * 2 * SLAB * 4 + my_sm;
        const unsigned g = (unsigned)(s * KS) * npad + my_g;
        const T* ga = colpT + row0 + g;
        const T* gb = rowp + col0 + g;
#pragma unroll
        for (int m = 0; m < SLAB / 4 / MM_THREADS; ++m) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa + m * (MM_THREADS / 32) * TB * 4),
                         "l"(ga + m * row_step_g) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa + SLAB * 4 + m * (MM_THREADS / 32) * TB * 4),
                         "l"(gb + m * row_step_g) : "memory");
        }
        cp_async_commit();
    };

    issue(0, 0);
    if (NSLAB > 1) issue(1, 1);

    T acc[8][8];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        gload4(D, ld, n, row0 + L.row(ri), col0 + L.cB0, vec != 0, &acc[ri][0]);
        gload4(D, ld, n, row0 + L.row(ri), col0 + L.cB1, vec != 0, &acc[ri][4]);
    }

#pragma unroll 1
    for (int s = 0; s < NSLAB; ++s) {
        if (s + 1 < NSLAB) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        if (s + 2 < NSLAB) issue(s + 2, (s + 2) % P3_STAGES);
        const T* As = sm + (s % P3_STAGES) * 2 * SLAB;
        mm_slab<T, KS, 2>(acc, As, As + SLAB, L);
    }

#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        const int i = row0 + L.row(ri);
        gstore4(D, ld, n, i, col0 + L.cB0, vec != 0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
        gstore4(D, ld, n, i, col0 + L.cB1, vec != 0, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
    }
}

constexpr size_t kPhase2Smem = 2ull * TB * TB * 4;
constexpr size_t kPhase3Smem = (size_t)P3_STAGES * 2 * KS * TB * 4;

}  // namespace apsp
