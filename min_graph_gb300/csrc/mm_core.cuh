// Register-blocked min-plus tile product cores for sm_103a.
//
// A 256-thread CTA computes acc[i][j] = min(acc[i][j], min_k A[i][k] +
// B[k][j]) for a 128 x 128 block held in registers (8 x 8 per thread, see
// MMLayout), reading the operands from shared memory.  This is the O(n^3)
// step of blocked Floyd-Warshall: phase 3 of the thesis page (1library.co
// excerpt, section 4.6, Algorithm 18) and, with the closed primary tile as
// one operand, phase 2 (Algorithm 17).
//
// Cores differ only in how one relaxation step is issued:
//   kCoreFused  one k at a time; int32 uses the fused add-min (__viaddmin_s32),
//               fp32 uses fminf of an IEEE sum.
//   kCoreMin3   two k at a time: two adds, then one three-input minimum.
//   kCorePacked two k at a time, with the operands k-pair interleaved in
//               shared memory (A2[k/2][i][2], B2[k/2][j][2]): one packed add
//               forms both sums, then one three-input minimum.  The
//               round-fused schedule's fp32 phase 3 runs this core.
//               fp32: add.rn.f32x2.  int32: one 64-bit add of the two 32-bit
//               halves.  Each sum is at most 2*INF < 2^32, so no carry crosses
//               from the low half into the high half.
// For int32, the three-input minimum is taken over the IEEE-754 bit patterns
// (min.f32).  Every operand is a non-negative int32 <= INF = 0x3FFFFFFF, and
// for non-negative floats the IEEE order is the integer order of the bit
// patterns.  A sum is at most 2*INF, so it only reaches the +inf/NaN
// patterns when it exceeds INF, and min.f32 drops a NaN input in favour of
// the others.  The accumulator is never NaN (<= INF), and min returns one
// input's bits unchanged (no flush to zero).  So the result is exactly the
// integer minimum, for every input in the library's contract.
//
// Every core double-buffers its operand fragments in two named register sets
// (load step s+1 while computing step s), so no register copies are needed.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

namespace apsp {

constexpr int TB = 128;  // tile edge

constexpr int kCoreFused = 0;
constexpr int kCoreMin3 = 1;
constexpr int kCorePacked = 2;
// Mixed int32 cores: the first R of the 8 accumulator rows take the fused
// add-min (ALU pipe only); the other rows take two adds + a three-input
// minimum, which moves the adds to the FMA pipe.  kCoreMixAdd + R lets the
// compiler place the adds.  kCoreMixMad + R writes each add as a multiply-add
// by an opaque 1, which runs on the FMA pipe.
constexpr int kCoreMixAdd = 16;
constexpr int kCoreMixMad = 32;

// Thread layouts of the 128 x 128 tile product.  Each thread owns 8 rows
// {rA0..rA0+3, rA1..rA1+3} (rA1 = rA0 + 16) and NC columns:
//   NC = 8: 256 threads, 8 warps as 4 (rows) x 2 (cols) of 32 x 64; columns
//           {cB0..cB0+3, cB1..cB1+3} with cB1 = cB0 + 32.
//   NC = 4: 512 threads, 16 warps as 4 x 4 of 32 x 32; columns cB0..cB0+3.
// Inside a warp the lanes are 4 (rows) x 8 (cols).  In the k-major layout,
// for a fixed k the lanes of a warp read 4 distinct 16-byte A chunks and 8
// distinct B chunks, all within one shared-memory row: one wavefront each.
template <int NC>
struct TileMap {
    static_assert(NC == 8 || NC == 4, "8 or 4 columns per thread");
    static constexpr int kThreads = NC == 8 ? 256 : 512;
    int rA0, rA1, cB0, cB1;
    __device__ __forceinline__ explicit TileMap(int tid) {
        const int w = tid >> 5, lane = tid & 31;
        const int tr = lane >> 3, tc = lane & 7;
        const int wr = NC == 8 ? (w >> 1) : (w >> 2);
        const int wc = NC == 8 ? (w & 1) : (w & 3);
        rA0 = wr * 32 + tr * 4;
        rA1 = rA0 + 16;
        cB0 = wc * (8 * NC) + tc * 4;
        cB1 = cB0 + 32;
    }
    __device__ __forceinline__ int row(int ri) const { return ri < 4 ? rA0 + ri : rA1 + (ri - 4); }
    __device__ __forceinline__ int col(int ci) const { return ci < 4 ? cB0 + ci : cB1 + (ci - 4); }
};
using MMLayout = TileMap<8>;

// ------------------------------------------------------------ elementwise ops

__device__ __forceinline__ float min3_f32(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <typename T> struct CoreOps;

template <> struct CoreOps<int32_t> {
    __device__ static __forceinline__ int32_t from_bits(int x) { return x; }
    __device__ static __forceinline__ int32_t relax1(int32_t acc, int32_t a, int32_t b) {
        return __viaddmin_s32(a, b, acc);
    }
    __device__ static __forceinline__ int32_t relax2(int32_t acc, int32_t a0, int32_t b0, int32_t a1,
                                                     int32_t b1) {
        return __float_as_int(min3_f32(__int_as_float(acc), __int_as_float(a0 + b0),
                                       __int_as_float(a1 + b1)));
    }
    // {a0, a1} + {b0, b1} as one 64-bit add (no carry between halves).
    __device__ static __forceinline__ int32_t relax2p(int32_t acc, unsigned long long pa,
                                                      unsigned long long pb) {
        const unsigned long long s = pa + pb;
        return __float_as_int(min3_f32(__int_as_float(acc), __uint_as_float((unsigned)s),
                                       __uint_as_float((unsigned)(s >> 32))));
    }
};

template <> struct CoreOps<float> {
    __device__ static __forceinline__ float from_bits(int x) { return __int_as_float(x); }
    __device__ static __forceinline__ float relax1(float acc, float a, float b) {
        return fminf(acc, __fadd_rn(a, b));
    }
    __device__ static __forceinline__ float relax2(float acc, float a0, float b0, float a1, float b1) {
        return min3_f32(acc, __fadd_rn(a0, b0), __fadd_rn(a1, b1));
    }
    // {a0, a1} + {b0, b1} as one paired IEEE add (round to nearest).
    __device__ static __forceinline__ float relax2p(float acc, unsigned long long pa,
                                                    unsigned long long pb) {
        unsigned long long s;
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(pa), "l"(pb));
        return min3_f32(acc, __uint_as_float((unsigned)s), __uint_as_float((unsigned)(s >> 32)));
    }
};

// a + b as a multiply-add by `one` (== 1 at run time, unknown to the
// compiler), so the sum is formed on the FMA pipe.
__device__ __forceinline__ int32_t add_on_fma(int32_t a, int32_t b, int32_t one) {
    int32_t d;
    asm("mad.lo.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(one), "r"(b));
    return d;
}

// ------------------------------------------------------------ fragment loads

// Four consecutive T from shared memory (16-byte aligned).
template <typename T>
__device__ __forceinline__ void lds4(const T* p, T* o) {
    const int4 v = *reinterpret_cast<const int4*>(p);
    o[0] = CoreOps<T>::from_bits(v.x);
    o[1] = CoreOps<T>::from_bits(v.y);
    o[2] = CoreOps<T>::from_bits(v.z);
    o[3] = CoreOps<T>::from_bits(v.w);
}

// Two consecutive 64-bit k-pairs from shared memory (16-byte aligned).
__device__ __forceinline__ void lds2x64(const void* p, unsigned long long* o) {
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
    o[0] = v.x;
    o[1] = v.y;
}

// k-major layout: A at As[k * TB + i], B at Bs[k * TB + j].
template <typename T, int NC>
__device__ __forceinline__ void frag_k(const T* __restrict__ As, const T* __restrict__ Bs, int k,
                                       const TileMap<NC>& L, T* a, T* b) {
    lds4(As + k * TB + L.rA0, a);
    lds4(As + k * TB + L.rA1, a + 4);
    lds4(Bs + k * TB + L.cB0, b);
    if constexpr (NC == 8) lds4(Bs + k * TB + L.cB1, b + 4);
}

// k-pair interleaved layout: A at A2[(kp * TB + i) * 2 + (k & 1)], same for B.
template <typename T>
__device__ __forceinline__ void frag_kp(const T* __restrict__ A2, const T* __restrict__ B2, int kp,
                                        const MMLayout& L, unsigned long long* pa,
                                        unsigned long long* pb) {
    const T* a = A2 + (kp * TB) * 2;
    const T* b = B2 + (kp * TB) * 2;
    lds2x64(a + 2 * L.rA0, pa);
    lds2x64(a + 2 * L.rA0 + 4, pa + 2);
    lds2x64(a + 2 * L.rA1, pa + 4);
    lds2x64(a + 2 * L.rA1 + 4, pa + 6);
    lds2x64(b + 2 * L.cB0, pb);
    lds2x64(b + 2 * L.cB0 + 4, pb + 2);
    lds2x64(b + 2 * L.cB1, pb + 4);
    lds2x64(b + 2 * L.cB1 + 4, pb + 6);
}

// ------------------------------------------------------------ cores

template <typename T, int NC>
__device__ __forceinline__ void step1(T (&acc)[8][NC], const T* a, const T* b) {
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) acc[ri][ci] = CoreOps<T>::relax1(acc[ri][ci], a[ri], b[ci]);
}

template <typename T>
__device__ __forceinline__ void step2(T (&acc)[8][8], const T* a0, const T* b0, const T* a1,
                                      const T* b1) {
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci)
            acc[ri][ci] = CoreOps<T>::relax2(acc[ri][ci], a0[ri], b0[ci], a1[ri], b1[ci]);
}

template <typename T>
__device__ __forceinline__ void step2p(T (&acc)[8][8], const unsigned long long* pa,
                                       const unsigned long long* pb) {
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = CoreOps<T>::relax2p(acc[ri][ci], pa[ri], pb[ci]);
}

template <int R, bool MAD>
__device__ __forceinline__ void step_mix(int32_t (&acc)[8][8], const int32_t* a0, const int32_t* b0,
                                         const int32_t* a1, const int32_t* b1, int32_t one) {
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
            if (ri < R) {
                acc[ri][ci] = __viaddmin_s32(a1[ri], b1[ci], __viaddmin_s32(a0[ri], b0[ci], acc[ri][ci]));
            } else {
                const int32_t s0 = MAD ? add_on_fma(a0[ri], b0[ci], one) : a0[ri] + b0[ci];
                const int32_t s1 = MAD ? add_on_fma(a1[ri], b1[ci], one) : a1[ri] + b1[ci];
                acc[ri][ci] = __float_as_int(
                    min3_f32(__int_as_float(acc[ri][ci]), __int_as_float(s0), __int_as_float(s1)));
            }
        }
}

// acc = min(acc, A (x) B) over k in [0, KLEN).  As/Bs: k-major for the fused,
// min3 and mixed cores, k-pair interleaved for the packed core.  `one` must
// be 1 (used by the kCoreMixMad cores only).
// Unroll of the k-pair loop, measured on GB300: int32 (one fused add-min per
// relaxation) runs 6% faster on ba16384 unrolled 8 times than not at all
// (full unrolling gains 0.3% more there, but loses 1.5% on er8192); fp32 (add,
// then min) runs 7% slower at any unroll.
template <typename T>
constexpr int kCoreUnroll = std::is_same<T, int32_t>::value ? 8 : 1;

template <typename T, int KLEN, int NC, int UNROLL = kCoreUnroll<T>>
__device__ __forceinline__ void mm_core_fused(T (&acc)[8][NC], const T* __restrict__ As,
                                              const T* __restrict__ Bs, const TileMap<NC>& L) {
    static_assert(KLEN % 2 == 0, "even k-length");
    T xa[8], xb[NC], ya[8], yb[NC];
    frag_k(As, Bs, 0, L, xa, xb);
#pragma unroll UNROLL
    for (int k = 0; k < KLEN; k += 2) {
        frag_k(As, Bs, k + 1, L, ya, yb);
        step1(acc, xa, xb);
        if (k + 2 < KLEN) frag_k(As, Bs, k + 2, L, xa, xb);
        step1(acc, ya, yb);
    }
}

// The packed core on k-pair interleaved operands: acc = min(acc, A (x) B)
// over k in [0, KLEN), two k-steps per packed add.  Unrolling its k-pair
// loop twice made the round-fused fp32 solve of n = 32768 4.5% faster than
// not unrolling (four times: the same; eight: 1% slower than two).
template <typename T, int KLEN, int UNROLL = 1>
__device__ __forceinline__ void mm_core_packed(T (&acc)[8][8], const T* __restrict__ As,
                                               const T* __restrict__ Bs, const MMLayout& L) {
    static_assert(KLEN % 4 == 0, "k-length a multiple of 4");
    unsigned long long xa[8], xb[8], ya[8], yb[8];
    frag_kp(As, Bs, 0, L, xa, xb);
#pragma unroll UNROLL
    for (int kp = 0; kp < KLEN / 2; kp += 2) {
        frag_kp(As, Bs, kp + 1, L, ya, yb);
        step2p<T>(acc, xa, xb);
        if (kp + 2 < KLEN / 2) frag_kp(As, Bs, kp + 2, L, xa, xb);
        step2p<T>(acc, ya, yb);
    }
}

template <typename T, int CORE, int KLEN>
__device__ __forceinline__ void mm_core(T (&acc)[8][8], const T* __restrict__ As,
                                        const T* __restrict__ Bs, const MMLayout& L, int one = 1) {
    if constexpr (CORE >= kCoreMixAdd) {
        static_assert(sizeof(T) == 4 && KLEN % 4 == 0, "mixed cores are int32, k-length % 4 == 0");
        constexpr int R = CORE & 15;
        constexpr bool MAD = CORE >= kCoreMixMad;
        T xa0[8], xb0[8], xa1[8], xb1[8], ya0[8], yb0[8], ya1[8], yb1[8];
        frag_k(As, Bs, 0, L, xa0, xb0);
        frag_k(As, Bs, 1, L, xa1, xb1);
#pragma unroll 1
        for (int k = 0; k < KLEN; k += 4) {
            frag_k(As, Bs, k + 2, L, ya0, yb0);
            frag_k(As, Bs, k + 3, L, ya1, yb1);
            step_mix<R, MAD>(acc, xa0, xb0, xa1, xb1, one);
            if (k + 4 < KLEN) {
                frag_k(As, Bs, k + 4, L, xa0, xb0);
                frag_k(As, Bs, k + 5, L, xa1, xb1);
            }
            step_mix<R, MAD>(acc, ya0, yb0, ya1, yb1, one);
        }
    } else if constexpr (CORE == kCoreFused) {
        mm_core_fused<T, KLEN, 8>(acc, As, Bs, L);
    } else if constexpr (CORE == kCoreMin3) {
        static_assert(KLEN % 4 == 0, "k-length a multiple of 4");
        T xa0[8], xb0[8], xa1[8], xb1[8], ya0[8], yb0[8], ya1[8], yb1[8];
        frag_k(As, Bs, 0, L, xa0, xb0);
        frag_k(As, Bs, 1, L, xa1, xb1);
#pragma unroll 1
        for (int k = 0; k < KLEN; k += 4) {
            frag_k(As, Bs, k + 2, L, ya0, yb0);
            frag_k(As, Bs, k + 3, L, ya1, yb1);
            step2(acc, xa0, xb0, xa1, xb1);
            if (k + 4 < KLEN) {
                frag_k(As, Bs, k + 4, L, xa0, xb0);
                frag_k(As, Bs, k + 5, L, xa1, xb1);
            }
            step2(acc, ya0, yb0, ya1, yb1);
        }
    } else {
        mm_core_packed<T, KLEN, 1>(acc, As, Bs, L);
    }
}

// acc = the NC columns of this thread's 8 rows of a 128 x 128 row-major
// tile in shared memory.
template <typename T, int NC>
__device__ __forceinline__ void load_tile(T (&acc)[8][NC], const T* __restrict__ tile,
                                          const TileMap<NC>& L) {
#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        lds4(tile + L.row(ri) * TB + L.cB0, &acc[ri][0]);
        if constexpr (NC == 8) lds4(tile + L.row(ri) * TB + L.cB1, &acc[ri][4]);
    }
}

}  // namespace apsp
