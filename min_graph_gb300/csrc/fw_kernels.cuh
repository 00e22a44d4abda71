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
// Phases 2 and 3 share one register-blocked tile product (mm_core.cuh): 256
// threads, each holding an 8 x 8 block of the 128 x 128 output in registers.
// The A operand is read from shared memory k-major (As[k][i]) and the B
// operand row-major (Bs[k][j]), 4 consecutive entries at a time.  The inner
// step is the fused integer add-min (__viaddmin_s32) for int32, and an IEEE
// add followed by a minimum for fp32.  Measured on sm_103a, the fused
// add-min keeps the ALU pipe fully busy at 64 relaxations per clock per SM.
// The two-k alternatives in mm_core.cuh (integer adds + three-input minimum,
// packed adds) run slower there, limited by issue and dispatch rather than
// by the ALU pipe.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "mm_core.cuh"
#include "tma.cuh"

namespace apsp {

constexpr int P1_THREADS = 512;    // phase 1: 128 rows x 4 quarters
constexpr int MM_THREADS = 256;    // tile-product threads (8 warps)
constexpr int KS = 32;             // k-slab depth in phase 3
constexpr int P3_STAGES = 3;       // cp.async ring depth (fallback phase 3)

template <typename T> struct Sem;

template <> struct Sem<int32_t> {
    static constexpr int32_t kInf = 0x3FFFFFFF;
    __device__ static __forceinline__ int32_t inf() { return kInf; }
    __device__ static __forceinline__ int32_t clamp(int32_t x) { return min(x, kInf); }
    // min(acc, a + b), one relaxation (fused integer add-min).
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

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Tile-product core used by phases 2 and 3 for each element type.
template <typename T> struct Core { static constexpr int value = kCoreFused; };

// ----------------------------------------------------------------- phase 1
//
// Closure of the primary tile P = D[K,K] (Algorithm 16 of the thesis page:
// standard Floyd-Warshall on the primary block, in shared memory, one
// block).  512 threads.  Each holds a 4 x 8 block of P in registers: rows
// i0..i0+3 (i0 = 4 * (t / 16)) and columns j0..j0+7 (j0 = 8 * (t % 16)).
// At step k a thread needs P[i][k] for its 4 rows (one 16-byte shared load)
// and P[k][j] for its 8 columns (two), which is 32 relaxations per 3 loads.
// The owners publish row k+1 and column k+1 into a double-buffered shared
// row/column buffer right after step k, so each step needs one barrier.  Row
// k and column k do not change during step k because P[k][k] >= 0.  The closed
// tile goes back to D and into the workspace as prim (row-major) and primT
// (transposed), which phase 2 reads.
template <typename T>
__global__ void __launch_bounds__(P1_THREADS, 1)
fw_phase1_diag(T* __restrict__ D, long long ld, int n, int r, T* __restrict__ prim,
               T* __restrict__ primT, int vec) {
    __shared__ __align__(16) T rowbuf[2][TB];
    __shared__ __align__(16) T colbuf[2][TB];
    const int t = threadIdx.x;
    const int g = t >> 4;           // row group: rows 4g .. 4g+3
    const int h = t & 15;           // column group: cols 8h .. 8h+7
    const int i0 = 4 * g, j0 = 8 * h;
    const int k0 = r * TB;
    T v[4][8];
#pragma unroll
    for (int ri = 0; ri < 4; ++ri) {
        gload4(D, ld, n, k0 + i0 + ri, k0 + j0, vec != 0, &v[ri][0]);
        gload4(D, ld, n, k0 + i0 + ri, k0 + j0 + 4, vec != 0, &v[ri][4]);
    }
    // publish row 0 and column 0
    if (g == 0) {
        vstore4(&rowbuf[0][j0], v[0][0], v[0][1], v[0][2], v[0][3]);
        vstore4(&rowbuf[0][j0 + 4], v[0][4], v[0][5], v[0][6], v[0][7]);
    }
    if (h == 0) vstore4(&colbuf[0][i0], v[0][0], v[1][0], v[2][0], v[3][0]);
    __syncthreads();

#pragma unroll 2  // 7% fewer cycles per k-step than rolled (measured)
    for (int kc = 0; kc < TB / 8; ++kc) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int k = kc * 8 + kk;
            const int buf = kk & 1;  // == k & 1
            T a[4], b[8];
            vload4(&colbuf[buf][i0], a);
            vload4(&rowbuf[buf][j0], b);
            vload4(&rowbuf[buf][j0 + 4], b + 4);
#pragma unroll
            for (int ri = 0; ri < 4; ++ri)
#pragma unroll
                for (int ci = 0; ci < 8; ++ci) v[ri][ci] = Sem<T>::relax(v[ri][ci], a[ri], b[ci]);
            if (k + 1 < TB) {
                // row k+1 lives in row group (k+1)/4 at register row (k+1)%4
                const int rr = (kk + 1) & 3;  // == (k+1) % 4, a compile-time value
                if (g == (k + 1) >> 2) {
                    vstore4(&rowbuf[buf ^ 1][j0], v[rr][0], v[rr][1], v[rr][2], v[rr][3]);
                    vstore4(&rowbuf[buf ^ 1][j0 + 4], v[rr][4], v[rr][5], v[rr][6], v[rr][7]);
                }
                // column k+1 lives in column group (k+1)/8 at register column (k+1)%8
                if (kk < 7) {
                    if (h == kc) vstore4(&colbuf[buf ^ 1][i0], v[0][kk + 1], v[1][kk + 1], v[2][kk + 1], v[3][kk + 1]);
                } else {
                    if (h == kc + 1) vstore4(&colbuf[buf ^ 1][i0], v[0][0], v[1][0], v[2][0], v[3][0]);
                }
                __syncthreads();
            }
        }
    }

#pragma unroll
    for (int ri = 0; ri < 4; ++ri) {
        const int i = i0 + ri;
        gstore4(D, ld, n, k0 + i, k0 + j0, vec != 0, v[ri][0], v[ri][1], v[ri][2], v[ri][3]);
        gstore4(D, ld, n, k0 + i, k0 + j0 + 4, vec != 0, v[ri][4], v[ri][5], v[ri][6], v[ri][7]);
        vstore4(prim + i * TB + j0, v[ri][0], v[ri][1], v[ri][2], v[ri][3]);
        vstore4(prim + i * TB + j0 + 4, v[ri][4], v[ri][5], v[ri][6], v[ri][7]);
    }
#pragma unroll
    for (int ci = 0; ci < 8; ++ci) vstore4(primT + (j0 + ci) * TB + i0, v[0][ci], v[1][ci], v[2][ci], v[3][ci]);
}

// ----------------------------------------------------------------- phase 2
//
// Row and column panels of the primary tile (Algorithm 17 of the thesis
// page, grid (nb-1, 2): y = 0 row panel, y = 1 column panel; blockIdx.x
// skips the primary tile the way the page's skipPrimaryBlock map does).
//   row panel tile (K,J):    new = min(old, P (x) old)  -> As = P^T, Bs = old
//   column panel tile (I,K): new = min(old, old (x) P)  -> As = old^T, Bs = P
// The accumulators start from the old tile (read from D).  As holds all 128
// k in shared memory.  The B operand streams in two 64-row halves, which
// keeps the CTA at 96 KiB of shared memory, so two CTAs share an SM and one
// CTA's loads overlap the other's compute.  The result goes to D and to the
// workspace panel that phase 3 reads: rowp (TB x npad) as is, colpT
// (TB x npad) transposed.
constexpr int P2_KH = TB / 2;  // k rows per B half

template <typename T>
__global__ void __launch_bounds__(MM_THREADS, (std::is_same<T, int32_t>::value ? 2 : 1))
fw_phase2_panels(T* __restrict__ D, long long ld, int n, int r, T* __restrict__ rowp,
                 T* __restrict__ colpT, const T* __restrict__ prim, const T* __restrict__ primT,
                 int npad, int vec) {
    extern __shared__ __align__(128) unsigned char p2_smem[];
    T* As = reinterpret_cast<T*>(p2_smem);  // [TB][TB]
    T* Bs = As + TB * TB;                    // [P2_KH][TB]
    const int tid = threadIdx.x;
    const int bx = blockIdx.x;
    const int other = bx + (bx >= r ? 1 : 0);
    const int k0 = r * TB, t0 = other * TB;
    const bool is_row = (blockIdx.y == 0);
    const MMLayout L(tid);
    // Full, aligned tiles stage their straight copies with cp.async; ragged
    // or unaligned tiles take element-wise loads.
    const bool fast = vec != 0 && k0 + TB <= n && t0 + TB <= n;
    const int orow0 = is_row ? k0 : t0, ocol0 = is_row ? t0 : k0;  // this CTA's tile in D

    T acc[8][8];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        gload4(D, ld, n, orow0 + L.row(ri), ocol0 + L.cB0, vec != 0, &acc[ri][0]);
        gload4(D, ld, n, orow0 + L.row(ri), ocol0 + L.cB1, vec != 0, &acc[ri][4]);
    }
    if (is_row) {
        for (int c = tid; c < TB * TB / 4; c += MM_THREADS)
            cp_async16(smem_u32(As + c * 4), primT + c * 4);
    } else {
        // transpose the old tile through registers: As[k][i] = old[i][k]
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
            const int k = L.col(ci);
            vstore4(As + k * TB + L.rA0, acc[0][ci], acc[1][ci], acc[2][ci], acc[3][ci]);
            vstore4(As + k * TB + L.rA1, acc[4][ci], acc[5][ci], acc[6][ci], acc[7][ci]);
        }
    }

#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        const int kb = hh * P2_KH;
        if (hh > 0) __syncthreads();  // everyone is done with the previous half
        if (is_row) {
            if (fast) {
                for (int c = tid; c < P2_KH * TB / 4; c += MM_THREADS) {
                    const int kk = c >> 5, qq = (c & 31) * 4;
                    cp_async16(smem_u32(Bs + kk * TB + qq), D + (long long)(k0 + kb + kk) * ld + t0 + qq);
                }
            } else {
                for (int c = tid; c < P2_KH * TB / 4; c += MM_THREADS) {
                    const int kk = c >> 5, qq = (c & 31) * 4;
                    T x[4];
                    gload4(D, ld, n, k0 + kb + kk, t0 + qq, vec != 0, x);
                    vstore4(Bs + kk * TB + qq, x[0], x[1], x[2], x[3]);
                }
            }
        } else {
            for (int c = tid; c < P2_KH * TB / 4; c += MM_THREADS)
                cp_async16(smem_u32(Bs + c * 4), prim + kb * TB + c * 4);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        if constexpr (std::is_same<T, int32_t>::value) {
            if (is_row && fast) {  // entries above INF read as INF
                for (int c = tid; c < P2_KH * TB / 4; c += MM_THREADS) {
                    T x[4];
                    vload4(Bs + c * 4, x);
                    vstore4(Bs + c * 4, Sem<T>::clamp(x[0]), Sem<T>::clamp(x[1]), Sem<T>::clamp(x[2]),
                            Sem<T>::clamp(x[3]));
                }
                __syncthreads();
            }
        }
        mm_core_fused<T, P2_KH, 8, 1>(acc, As + kb * TB, Bs, L);  // phase 2 runs the rolled core
    }

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

// Tile (I, J) of the t-th phase-3 work item in round r: row-major over the
// (nb-1) x (nb-1) grid of non-primary tiles, skipping row and column r.
__device__ __forceinline__ void phase3_tile(int t, int nbm1, int r, int& I, int& J) {
    const int ti = t / nbm1, tj = t - ti * nbm1;
    I = ti + (ti >= r ? 1 : 0);
    J = tj + (tj >= r ? 1 : 0);
}

// ------------------------------------------------- phase 3, cp.async version
//
// Every tile (I,J) with I != K and J != K (Algorithm 18 of the thesis page,
// grid (nb-1)^2 with the primary row and column skipped):
//   D[I,J] <- min(D[I,J], D[I,K] (x) D[K,J]).
// One CTA per tile.  The panels come from the workspace (colpT gives
// As[k][i], rowp gives Bs[k][j]) in KS-deep slabs through a cp.async ring.
// This version serves matrices whose base or leading dimension rules out
// TMA (not 16-byte aligned); fw_phase3_persistent serves the rest.
template <typename T>
__global__ void __launch_bounds__(MM_THREADS, 1)
fw_phase3_minplus(T* __restrict__ D, long long ld, int n, int r, int nbm1,
                  const T* __restrict__ rowp, const T* __restrict__ colpT, int npad, int vec) {
    extern __shared__ __align__(128) unsigned char p3_smem[];
    T* sm = reinterpret_cast<T*>(p3_smem);
    const int tid = threadIdx.x;
    int I, J;
    phase3_tile(blockIdx.x, nbm1, r, I, J);
    const int row0 = I * TB, col0 = J * TB;
    const MMLayout L(tid);
    constexpr int NSLAB = TB / KS;
    constexpr int SLAB = KS * TB;  // elements per operand slab

    // Each thread copies the 16-byte chunks c = tid + m * MM_THREADS of a
    // slab: row kk = c / 32, column 4 * (c % 32).
    const uint32_t sm_base = smem_u32(sm);
    const uint32_t my_sm = ((tid >> 5) * TB + (tid & 31) * 4) * 4;
    const unsigned my_g = (tid >> 5) * npad + (tid & 31) * 4;
    const unsigned row_step_g = (MM_THREADS / 32) * npad;
    auto issue = [&](int s, int st) {
        const uint32_t sa = sm_base + st * 2 * SLAB * 4 + my_sm;
        const unsigned g = (unsigned)(s * KS) * npad + my_g;
        const T* ga = colpT + row0 + g;
        const T* gb = rowp + col0 + g;
#pragma unroll
        for (int m = 0; m < SLAB / 4 / MM_THREADS; ++m) {
            cp_async16(sa + m * (MM_THREADS / 32) * TB * 4, ga + m * row_step_g);
            cp_async16(sa + SLAB * 4 + m * (MM_THREADS / 32) * TB * 4, gb + m * row_step_g);
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
        mm_core<T, Core<T>::value, KS>(acc, As, As + SLAB, L);
    }

#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        const int i = row0 + L.row(ri);
        gstore4(D, ld, n, i, col0 + L.cB0, vec != 0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
        gstore4(D, ld, n, i, col0 + L.cB1, vec != 0, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
    }
}

// --------------------------------------------- phase 3, persistent TMA version
//
// Same update as fw_phase3_minplus, restructured for sm_103a: one CTA per SM
// walks a static round-robin list of tiles.  A producer warp (one elected
// thread) streams, by TMA, each tile's C block (128 x 128 of D) into a
// shared buffer and its panel k-slabs (A from colpT, B from rowp) into a
// P3P_STAGES-deep ring.  The loads run ahead across tile boundaries, so the
// next tile's data arrive while the current one computes.  Eight consumer
// warps own the 128 x 128 accumulator block in registers.  They read C once
// from shared memory, run the paired-k product over the ring, and store the
// result straight from registers.  Full/empty mbarriers order the two sides,
// and every wait is bounded (tma.cuh).
constexpr uint32_t P3P_SLAB_BYTES = KS * TB * 4;             // 16 KiB per operand slab
constexpr uint32_t P3P_STAGE_BYTES = 2 * P3P_SLAB_BYTES;     // A + B
constexpr uint32_t P3P_C_BYTES = TB * TB * 4;                // 64 KiB
// Shared memory of the persistent phase 3 with a ring of `stages` slabs.
constexpr size_t phase3p_smem(int stages) {
    return 1024 + P3P_C_BYTES + (size_t)stages * P3P_STAGE_BYTES + 256;
}

// NC = accumulator columns per consumer thread: 8 (256 consumers, 2 warps per
// SM sub-partition) or 4 (512 consumers, 4 warps per sub-partition, which
// hides barrier waits and epilogues better).
template <int NC>
constexpr int p3p_threads() { return TileMap<NC>::kThreads + 32; }

template <typename T, int NC, int P3P_STAGES>
__global__ void __launch_bounds__(p3p_threads<NC>(), 1)
fw_phase3_persistent(T* __restrict__ D, long long ld, int n, int r, int nbm1, int ntiles,
                     const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b, int* __restrict__ err,
                     unsigned long long timeout_ns, int inject) {
    constexpr int CONSUMERS = TileMap<NC>::kThreads;
    constexpr int CWARPS = CONSUMERS / 32;
    extern __shared__ unsigned char p3p_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(p3p_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    T* cbuf = reinterpret_cast<T*>(base);
    unsigned char* ring = base + P3P_C_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + P3P_STAGES * P3P_STAGE_BYTES);
    const uint32_t bar_full = smem_u32(bars);                   // [P3P_STAGES]
    const uint32_t bar_empty = bar_full + 8 * P3P_STAGES;       // [P3P_STAGES]
    const uint32_t bar_cfull = bar_empty + 8 * P3P_STAGES;
    const uint32_t bar_cempty = bar_cfull + 8;
    const int tid = threadIdx.x;
    constexpr int NSLAB = TB / KS;

    if (tid == 0) {
        for (int s = 0; s < P3P_STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, CWARPS);
        }
        mbar_init(bar_cfull, 1);
        mbar_init(bar_cempty, CWARPS);
        mbar_init_fence();
    }
    __syncthreads();

    if (tid >= CONSUMERS) {
        // ------------------------------------------------------ producer
        if (tid != CONSUMERS) return;
        tma_prefetch_desc(&tm_c);
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        const uint32_t cdst = smem_u32(cbuf);
        const uint32_t rdst = smem_u32(ring);
        uint32_t g = 0;   // slabs issued so far
        int it = 0;       // tiles whose C load was issued
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            int I, J;
            phase3_tile(t, nbm1, r, I, J);
            if (it > 0 && !mbar_wait_bounded(bar_cempty, (it - 1) & 1, err, timeout_ns)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(bar_cfull, P3P_C_BYTES);
            tma_load_2d(cdst, &tm_c, J * TB, I * TB, bar_cfull);
            ++it;
            for (int s = 0; s < NSLAB; ++s) {
                const uint32_t st = g % P3P_STAGES, use = g / P3P_STAGES;
                if (use > 0 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1, err, timeout_ns)) {
                    ok = false;
                    break;
                }
                if (inject && g == 0 && blockIdx.x == 0) {
                    // Test hook: this slab is never issued, so the consumers'
                    // bounded wait on it must run out (APSP_ETIMEOUT).
                    ++g;
                    continue;
                }
                const uint32_t dst = rdst + st * P3P_STAGE_BYTES;
                mbar_arrive_expect_tx(bar_full + 8 * st, P3P_STAGE_BYTES);
                tma_load_2d(dst, &tm_a, I * TB, s * KS, bar_full + 8 * st);
                tma_load_2d(dst + P3P_SLAB_BYTES, &tm_b, J * TB, s * KS, bar_full + 8 * st);
                ++g;
            }
        }
        if (!ok) {
            // Drain: wait (bounded) for every copy still in flight before the
            // CTA may exit, so no TMA write lands in freed shared memory.
            for (uint32_t q = (g > P3P_STAGES ? g - P3P_STAGES : 0); q < g; ++q)
                mbar_wait_bounded(bar_full + 8 * (q % P3P_STAGES), (q / P3P_STAGES) & 1, err,
                                  timeout_ns, false);
            if (it > 0) mbar_wait_bounded(bar_cfull, (it - 1) & 1, err, timeout_ns, false);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const TileMap<NC> L(tid);
    const int lane = tid & 31;
    uint32_t g = 0;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        int I, J;
        phase3_tile(t, nbm1, r, I, J);
        T acc[8][NC];
        if (!mbar_wait_bounded(bar_cfull, it & 1, err, timeout_ns)) return;
        load_tile(acc, cbuf, L);
#pragma unroll
        for (int ri = 0; ri < 8; ++ri)
#pragma unroll
            for (int ci = 0; ci < NC; ++ci) acc[ri][ci] = Sem<T>::clamp(acc[ri][ci]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cempty);
        for (int s = 0; s < NSLAB; ++s, ++g) {
            const uint32_t st = g % P3P_STAGES, use = g / P3P_STAGES;
            if (!mbar_wait_bounded(bar_full + 8 * st, use & 1, err, timeout_ns)) return;
            const T* As = reinterpret_cast<const T*>(ring + st * P3P_STAGE_BYTES);
            mm_core_fused<T, KS, NC>(acc, As, As + KS * TB, L);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        }
        const int row0 = I * TB, col0 = J * TB;
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            const int i = row0 + L.row(ri);
            gstore4(D, ld, n, i, col0 + L.cB0, true, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            if constexpr (NC == 8)
                gstore4(D, ld, n, i, col0 + L.cB1, true, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
        }
    }
}

constexpr size_t kPhase2Smem = (size_t)(TB + P2_KH) * TB * 4;
constexpr size_t kPhase3Smem = (size_t)P3_STAGES * 2 * KS * TB * 4;

}  // namespace apsp
