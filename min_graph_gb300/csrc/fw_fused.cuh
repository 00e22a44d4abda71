// Round-fused persistent blocked Floyd-Warshall (lookahead), sm_103a.
//
// The three phases of the thesis page (1library.co excerpt, section 4.6,
// Algorithms 16-18) keep their arithmetic; what changes is the scheduling.
// Launch r runs, on one CTA per SM, the phase-3 tiles of round r together
// with phase 1 and phase 2 of round r+1:
//
//   first               phase 3 (round r): the tiles in row r+1 and column
//                       r+1 ("critical"; the diagonal (r+1, r+1) first)
//   then one item       phase 1 (round r+1): close tile (r+1, r+1)
//   then x tiles        phase 3 (round r): ordinary tiles
//   then 2(nb-1) tiles  phase 2 (round r+1): row panel (r+1, J), column
//                       panel (I, r+1)
//   the rest            phase 3 (round r): ordinary tiles
// When a launch holds few tiles (fused_split), every phase-3 and phase-2
// tile is split along k into `split` consecutive items of one or two
// k-slabs; the parts merge into D by min-reduction, and the part that
// completes a tile counts it done (a critical tile: its round flag; a
// phase-2 tile: a finisher item, queued on the same CTA, that writes the
// tile's panel copy for the next launch).
//
// CTAs take items in this order from a global counter.  Each item depends
// only on items before it: phase 1 of r+1 on the critical tile (r+1, r+1),
// and a phase-2 item on phase 1 of r+1 and on its own critical tile.  So
// whichever CTAs are running always make progress, and no deadlock is
// possible.  Waits on those dependencies are bounded spins on round-stamped
// flags in global memory.  Launch r+1 may start on the SMs that launch r
// frees (programmatic dependent launch) but touches no global memory before
// launch r has completed.  Phase 1 and phase 2 of round r+1 thus run inside
// round r's phase-3 work, instead of as two latency-bound launches between
// rounds.  The row/column panel buffers alternate between rounds, so phase 2
// of r+1 never overwrites what phase 3 of r is reading.  A prologue launch
// (r = -1) runs phase 1 and phase 2 of round 0; the last launch runs phase 3
// only.
//
// Each CTA is one producer warpgroup (one thread takes items, waits for
// their inputs, and issues TMA loads and reductions) and eight consumer
// warps (the arithmetic, on the tile-product core of mm_core.cuh).
//   phase-3 tile:  A slabs <- column panel; B slabs <- row panel.  The
//                  accumulators start at INF, the consumers stage the result
//                  in the C buffer, and the producer merges it into D with a
//                  TMA min-reduction in L2 (D is never loaded into the SM).
//                  int32 runs the fused add-min on k-major panels; fp32 runs
//                  the packed core on k-pair interleaved panels (kPanelPack
//                  in fw_launch.h), one packed add and one three-input
//                  minimum per two relaxations.
//   row panel:     C <- D tile (also the B operand, read in shared memory);
//                  A slabs <- transposed closed primary tile
//   column panel:  C <- D tile; the consumers write its transpose into the
//                  ring as the A operand; B slabs <- closed primary tile
//                  (a phase-2 tile in one piece stores D and its panel copy
//                  with plain stores; a part stages and merges like phase 3)
//   phase 1:       C <- D tile; closed in registers with a published row and
//                  column per step (as fw_phase1_diag)
// A TMA load of a tile that crosses the edge of the matrix reads zeros
// outside it.  Phase-1 and phase-2 items overwrite those positions with INF
// before using them; phase 3 never stores them.
#pragma once

#include "fw_kernels.cuh"
#include "fw_launch.h"

namespace apsp {

constexpr int FZ_STAGES = 4;
constexpr int FZ_CONSUMERS = 256;
// One producer warpgroup, of which one thread works.  Nine warps would put
// three on one SM sub-partition and cap every thread at 168 registers; with
// twelve, the producer warpgroup hands registers to the consumers
// (setmaxnreg) and the consumers' tile product compiles without spills.
// Measured: ba16384 240.05 -> 237.58 ms, er8192 30.54 -> 30.10 ms.
constexpr int FZ_THREADS = FZ_CONSUMERS + 128;
constexpr int FZ_REG_LAUNCH = 168;    // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int FZ_REG_CONSUMER = 208;  // per consumer thread after the hand-over
constexpr int FZ_REG_PRODUCER = 88;   // per producer-warpgroup thread (less spills its item logic)
static_assert(FZ_CONSUMERS * FZ_REG_CONSUMER + 128 * FZ_REG_PRODUCER <= FZ_THREADS * FZ_REG_LAUNCH,
              "the register hand-over must fit in what the block is launched with");
constexpr uint32_t FZ_SLAB = KS * TB * 4;       // 16 KiB
constexpr uint32_t FZ_STAGE = 2 * FZ_SLAB;      // A half + B half
constexpr uint32_t FZ_C = TB * TB * 4;          // 64 KiB
constexpr uint32_t FZ_MISC = 4096;              // barriers, item slots, phase-1 buffers
constexpr size_t kFusedSmem = 1024 + FZ_C + (size_t)FZ_STAGES * FZ_STAGE + FZ_MISC;
constexpr int FZ_NAMED_BAR = 1;                 // consumer-only named barrier id

// Phase-3 epilogue by TMA reduction: D <- min(D, tile) is a signed 32-bit
// minimum in L2, through an INT32-typed tensor map of D (the bulk tensor
// reduction has no fp32 minimum).  For fp32 the integer order of the bit
// patterns is the order of the values, because within the library's
// contract every entry is +0, a positive float or +inf (a -0.0 input is the
// smallest pattern and acts as zero).

enum : int { kItemP3 = 0, kItemP1 = 1, kItemP2Row = 2, kItemP2Col = 3, kItemFin = 4 };
enum : int { kCritNone = 0, kCritDiag = 1, kCritRow = 2, kCritCol = 3 };

struct FusedItem {
    int kind, I, J, crit;
    int s0, s1;  // a phase-3 item's k-slabs: [s0, s1) of the tile's TB / KS
};

// A phase-3 tile may be split into `split` items along k (fused_split in
// fw_launch.h), so that a launch with few tiles still fills the GPU and a
// critical tile finishes sooner.  The parts of a tile merge into D by the
// same min-reduction, and min is associative, so the result does not depend
// on the split.

// Number of items of launch r (r = -1: prologue).  Phase-2 tiles split
// like phase-3 tiles; the finisher items that rewrite a split phase-2
// tile's panel copy are handed out on top of these.
__host__ __device__ inline long long fused_items(int r, int nb, int split) {
    const long long p2 = 2LL * (nb - 1) * split;
    if (r < 0) return 1 + p2;
    const long long p3 = (long long)(nb - 1) * (nb - 1) * split;
    if (r + 1 >= nb) return p3;
    return p3 + 1 + p2;
}

// Ordinary phase-3 tiles taken before phase 2 of round r+1: enough work for
// the other CTAs while one CTA runs phase 1 of r+1.
__host__ __device__ inline int fused_head(int nb, int grid) {
    const long long reg = (long long)(nb - 2) * (nb - 2);
    const long long want = 3LL * grid;
    return (int)(reg < want ? reg : want);
}

__device__ __forceinline__ FusedItem fused_item(int l, int r, int nb, int x, int split) {
    FusedItem it;
    it.crit = kCritNone;
    it.s0 = 0;
    it.s1 = TB / KS;
    const int rn = r + 1;
    const int per = (TB / KS) / split;  // slabs per part
    if (r < 0) {  // prologue: phase 1 and phase 2 of round 0
        if (l == 0) { it.kind = kItemP1; it.I = it.J = 0; return it; }
        const int q = (l - 1) / split;
        it.s0 = ((l - 1) % split) * per;
        it.s1 = it.s0 + per;
        if (q < nb - 1) { it.kind = kItemP2Row; it.I = 0; it.J = q + 1; }
        else { it.kind = kItemP2Col; it.I = q - (nb - 1) + 1; it.J = 0; }
        return it;
    }
    it.kind = kItemP3;
    if (rn >= nb) {  // last round: phase 3 only
        phase3_tile(l / split, nb - 1, r, it.I, it.J);
        it.s0 = (l % split) * per;
        it.s1 = it.s0 + per;
        return it;
    }
    const int c1 = 2 * nb - 3;
    if (l < c1 * split) {  // the parts of one critical tile are consecutive
        const int t = l / split;
        it.s0 = (l % split) * per;
        it.s1 = it.s0 + per;
        if (t == 0) { it.I = it.J = rn; it.crit = kCritDiag; }
        else if (t < nb - 1) { const int q = t - 1; it.I = rn; it.J = q + (q >= r ? 2 : 0); it.crit = kCritRow; }
        else { const int q = t - (nb - 1); it.I = q + (q >= r ? 2 : 0); it.J = rn; it.crit = kCritCol; }
        return it;
    }
    l -= c1 * split;
    if (l == 0) { it.kind = kItemP1; it.I = it.J = rn; return it; }
    l -= 1;
    const int np2 = 2 * (nb - 1) * split;
    const int xi = x * split;
    int q;
    if (l < xi) {
        q = l;
    } else if (l < xi + np2) {  // the parts of one phase-2 tile are consecutive
        const int p = (l - xi) / split;
        it.s0 = ((l - xi) % split) * per;
        it.s1 = it.s0 + per;
        if (p < nb - 1) { it.kind = kItemP2Row; it.I = rn; it.J = p + (p >= rn ? 1 : 0); }
        else { const int pp = p - (nb - 1); it.kind = kItemP2Col; it.I = pp + (pp >= rn ? 1 : 0); it.J = rn; }
        return it;
    } else {
        q = l - np2;
    }
    const int nb2 = nb > 2 ? nb - 2 : 1;  // ordinary tiles exist only when nb > 2
    const int t = q / split;
    it.s0 = (q % split) * per;
    it.s1 = it.s0 + per;
    const int ti = t / nb2, tj = t - ti * nb2;
    it.I = ti + (ti >= r ? 2 : 0);
    it.J = tj + (tj >= r ? 2 : 0);
    return it;
}

__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync %0, %1;" ::"n"(FZ_NAMED_BAR), "n"(FZ_CONSUMERS) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *flag == value (bounded).  Afterwards the data published with
// the flag is visible to this thread and to its later TMA (async proxy) reads.
__device__ __forceinline__ bool flag_wait(const int* flag, int value, int* err,
                                          unsigned long long timeout_ns) {
    if (ld_acquire(flag) != value) {
        const unsigned long long t0 = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            __nanosleep(64);
            if (ld_acquire(flag) == value) break;
            if ((it & 31u) == 0u) {
                if (*reinterpret_cast<volatile int*>(err) != 0) return false;
                if (global_timer_ns() - t0 > timeout_ns) {
                    atomicOr(err, kDeviceErrTimeout);
                    return false;
                }
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// All consumer threads have issued their global stores for this item:
// publish them (GPU scope, and to the async proxy) and set *flag = value.
__device__ __forceinline__ void flag_signal(int* flag, int value) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    consumer_barrier();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicExch(flag, value);
    }
}

// Set the positions of this thread's 8 x 8 block that fall outside the n x n
// matrix to INF (tile at D[row0.., col0..]).
template <typename T>
__device__ __forceinline__ void mask_outside(T (&acc)[8][8], const MMLayout& L, int row0, int col0,
                                             int n) {
    if (row0 + TB <= n && col0 + TB <= n) return;
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci)
            if (row0 + L.row(ri) >= n || col0 + L.col(ci) >= n) acc[ri][ci] = Sem<T>::inf();
}

// The workspace copy of this thread's 8 x 8 block of row-panel tile (rn, J)
// (tile row i is panel row k = i), in the layout kPanelPack<T> names.
template <typename T>
__device__ __forceinline__ void store_row_panel(T* rp, const T (&acc)[8][8], const MMLayout& L, int col0,
                                                int npad) {
    if constexpr (kPanelPack<T> == 1) {
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            const int i = L.row(ri);
            vstore4(rp + (long long)i * npad + col0 + L.cB0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            vstore4(rp + (long long)i * npad + col0 + L.cB1, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
        }
    } else {
        // rows i and i + 1 (i even) form one k-pair row of the panel
#pragma unroll
        for (int ri = 0; ri < 8; ri += 2) {
            T* p = rp + (long long)(L.row(ri) >> 1) * (2 * npad) + 2 * col0;
            vstore4(p + 2 * L.cB0, acc[ri][0], acc[ri + 1][0], acc[ri][1], acc[ri + 1][1]);
            vstore4(p + 2 * L.cB0 + 4, acc[ri][2], acc[ri + 1][2], acc[ri][3], acc[ri + 1][3]);
            vstore4(p + 2 * L.cB1, acc[ri][4], acc[ri + 1][4], acc[ri][5], acc[ri + 1][5]);
            vstore4(p + 2 * L.cB1 + 4, acc[ri][6], acc[ri + 1][6], acc[ri][7], acc[ri + 1][7]);
        }
    }
}

// The workspace copy, transposed, of this thread's block of column-panel
// tile (I, rn) (tile column k is panel row k), in the layout kPanelPack<T>
// names.
template <typename T>
__device__ __forceinline__ void store_col_panel(T* cp, const T (&acc)[8][8], const MMLayout& L, int row0,
                                                int npad) {
    if constexpr (kPanelPack<T> == 1) {
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) {
            const int k = L.col(ci);
            vstore4(cp + (long long)k * npad + row0 + L.rA0, acc[0][ci], acc[1][ci], acc[2][ci], acc[3][ci]);
            vstore4(cp + (long long)k * npad + row0 + L.rA1, acc[4][ci], acc[5][ci], acc[6][ci], acc[7][ci]);
        }
    } else {
        // columns k and k + 1 (k even) form one k-pair row of the panel
#pragma unroll
        for (int ci = 0; ci < 8; ci += 2) {
            T* p = cp + (long long)(L.col(ci) >> 1) * (2 * npad) + 2 * row0;
            vstore4(p + 2 * L.rA0, acc[0][ci], acc[0][ci + 1], acc[1][ci], acc[1][ci + 1]);
            vstore4(p + 2 * L.rA0 + 4, acc[2][ci], acc[2][ci + 1], acc[3][ci], acc[3][ci + 1]);
            vstore4(p + 2 * L.rA1, acc[4][ci], acc[4][ci + 1], acc[5][ci], acc[5][ci + 1]);
            vstore4(p + 2 * L.rA1 + 4, acc[6][ci], acc[6][ci + 1], acc[7][ci], acc[7][ci + 1]);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(FZ_THREADS, 1)
fw_round_fused(T* __restrict__ D, long long ld, int n, int r, int nb, int npad, int nitems, int split,
               const __grid_constant__ FusedMaps maps, const FusedPtrs ptrs,
               unsigned long long timeout_ns, int inject) {
    extern __shared__ unsigned char fz_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(fz_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    T* cbuf = reinterpret_cast<T*>(base);
    unsigned char* ring = base + FZ_C;
    unsigned char* misc = ring + FZ_STAGES * FZ_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    volatile int* slots = reinterpret_cast<volatile int*>(misc + 128);
    T* p1row = reinterpret_cast<T*>(misc + 1024);  // [2][TB]
    T* p1col = p1row + 2 * TB;                      // [2][TB]
    const uint32_t bar_full = smem_u32(bars);
    const uint32_t bar_empty = bar_full + 8 * FZ_STAGES;
    const uint32_t bar_cfull = bar_empty + 8 * FZ_STAGES;
    const uint32_t bar_cempty = bar_cfull + 8;
    const uint32_t bar_staged = bar_cempty + 8;  // merge epilogue: tile staged in the C buffer
    const uint32_t bar_sfree = bar_staged + 8;   // merge epilogue: staged tile read by the reduction
    const int tid = threadIdx.x;
    const int rn = r + 1;
    const int x = fused_head(nb, gridDim.x);
    const int per = (TB / KS) / split;  // k-slabs per phase-3 item
    int* err = ptrs.err;

    if (tid == 0) {
        for (int s = 0; s < FZ_STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, FZ_CONSUMERS / 32);
        }
        mbar_init(bar_cfull, 1);
        mbar_init(bar_cempty, FZ_CONSUMERS / 32);
        mbar_init(bar_staged, FZ_CONSUMERS / 32);
        mbar_init(bar_sfree, 1);
        mbar_init_fence();
    }
    __syncthreads();
    // A launch may start while the previous one drains (programmatic
    // dependent launch): nothing in global memory is touched before the
    // previous launch has completed and its writes are visible.  Without a
    // programmatic predecessor this returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (tid >= FZ_CONSUMERS) {
        // ================================================== producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(FZ_REG_PRODUCER));
        if (tid != FZ_CONSUMERS) return;
        const uint32_t cdst = smem_u32(cbuf);
        const uint32_t rdst = smem_u32(ring);
        const int pb = r & 1, nbuf = rn & 1;  // panel buffers read / written
        uint32_t g = 0;
        int it = 0;
        bool ok = true;
        // Merge epilogue: the phase-3 item whose tile the consumers stage in
        // the C buffer, still to be merged into D, and the merges issued.
        bool pend = false;
        FusedItem pw;
        pw.kind = kItemP3;
        pw.I = pw.J = 0;
        pw.crit = kCritNone;
        uint32_t merges = 0;
        // Split phase-2 tiles whose parts have all merged, waiting for their
        // finisher item: code J for row tile (rn, J), nb + I for column tile
        // (I, rn).  One merge per loop turn, so two entries suffice.
        int fin[2] = {-1, -1};
        int nfin = 0;
        // Merge the pending tile: D <- min(D, staged tile) by a TMA reduction
        // in L2.  A critical tile's flag is set once the reduction's writes
        // are complete; otherwise it is enough that the buffer has been read.
        auto merge_pending = [&]() -> bool {
            if (!pend) return true;
            pend = false;
            if (!mbar_wait_bounded(bar_staged, merges & 1, err, timeout_ns)) return false;
            tma_reduce_min_2d(&maps.cmin, pw.J * TB, pw.I * TB, cdst);
            bulk_commit();
            if (pw.kind != kItemP3) {
                // A phase-2 part: once the tile's last part has merged, queue
                // the finisher that rewrites the tile's panel copy.
                bulk_wait_all();
                const int c = pw.kind == kItemP2Row ? 1 + pw.J : 1 + nb + pw.I;
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                if (atomicAdd(ptrs.parts + c, 1) == split - 1) {
                    atomicExch(ptrs.parts + c, 0);
                    fin[nfin++] = pw.kind == kItemP2Row ? pw.J : nb + pw.I;
                }
            } else if (pw.crit != kCritNone) {
                // The tile is complete once all its parts have merged: the
                // last part to finish sets the round flag and clears the
                // count for the next launch.
                bulk_wait_all();
                const int c = pw.crit == kCritDiag ? 0 : pw.crit == kCritRow ? 1 + pw.J : 1 + nb + pw.I;
                int* f = pw.crit == kCritDiag ? ptrs.flag_diag
                         : pw.crit == kCritRow ? ptrs.flag_row + pw.J
                                               : ptrs.flag_col + pw.I;
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                if (atomicAdd(ptrs.parts + c, 1) == split - 1) {
                    atomicExch(ptrs.parts + c, 0);
                    __threadfence();
                    atomicExch(f, rn);
                }
            } else {
                bulk_wait_read_all();
            }
            mbar_arrive(bar_sfree);
            ++merges;
            return true;
        };
        for (;;) {
            FusedItem w;
            w.kind = kItemP3;
            w.I = w.J = 0;
            w.crit = kCritNone;
            w.s0 = 0;
            w.s1 = TB / KS;
            int l = -1;  // the item's index (-2 - code for a finisher)
            bool stop = false;
            if (nfin == 0) {
                l = atomicAdd(ptrs.counters + rn, 1);
                stop = l >= nitems;
                if (!stop) w = fused_item(l, r, nb, x, split);
                // this CTA takes no further items: the next launch may start
                // on the SMs that drain
                else asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            } else {
                w.kind = kItemFin;
            }
            // Items merged through the C buffer: phase-3 tiles, and phase-2
            // parts when tiles are split.
            const bool merged = !stop && (w.kind == kItemP3 ||
                                          (split > 1 && (w.kind == kItemP2Row || w.kind == kItemP2Col)));
            // Everything but a phase-3 item needs the C buffer, and may wait
            // for the pending tile's flag: merge it first.  So does the end.
            if (w.kind != kItemP3 || stop) ok = merge_pending();
            if (ok && stop && nfin > 0) continue;  // that merge completed a phase-2 tile: finish it first
            if (w.kind == kItemFin) {
                const int code = fin[0];
                fin[0] = fin[1];
                --nfin;
                l = -2 - code;
                w.I = code < nb ? rn : code - nb;
                w.J = code < nb ? code : rn;
            } else if (ok && !stop) {
                if (w.kind == kItemP1 && r >= 0)
                    ok = flag_wait(ptrs.flag_diag, rn, err, timeout_ns);
                else if (w.kind == kItemP2Row)
                    ok = flag_wait(ptrs.flag_p1, rn, err, timeout_ns) &&
                         (r < 0 || w.J == r || flag_wait(ptrs.flag_row + w.J, rn, err, timeout_ns));
                else if (w.kind == kItemP2Col)
                    ok = flag_wait(ptrs.flag_p1, rn, err, timeout_ns) &&
                         (r < 0 || w.I == r || flag_wait(ptrs.flag_col + w.I, rn, err, timeout_ns));
            }
            if (it > 0 && !mbar_wait_bounded(bar_cempty, (it - 1) & 1, err, timeout_ns)) ok = false;
            if (stop || !ok) {
                slots[2 * (it & 1)] = -1;
                mbar_arrive(bar_cfull);  // no bytes expected: releases the consumers
                break;
            }
            // the consumers get the item decoded: kind, critical class and
            // slab range in one word, the tile in the other
            slots[2 * (it & 1)] = w.kind | (w.crit << 4) | (w.s0 << 8) | (w.s1 << 16);
            slots[2 * (it & 1) + 1] = (w.I << 16) | w.J;
            if (w.kind == kItemP3) {
                mbar_arrive(bar_cfull);  // no C tile: the consumers start from INF
            } else {
                // phase 1, phase 2 (or its part) and finishers start from the
                // D tile; a finisher's tile is complete (its parts' merges
                // were waited for before they were counted)
                if (w.kind == kItemFin) asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(bar_cfull, FZ_C);
                tma_load_2d(cdst, &maps.c, w.J * TB, w.I * TB, bar_cfull);
            }
            ++it;
            if (w.kind == kItemP1 || w.kind == kItemFin) continue;  // no slabs
            for (int s = w.s0; s < w.s1; ++s) {
                const uint32_t st = g % FZ_STAGES, use = g / FZ_STAGES;
                if (use > 0 && !mbar_wait_bounded(bar_empty + 8 * st, (use - 1) & 1, err, timeout_ns)) {
                    ok = false;
                    break;
                }
                if (inject && l == 0 && s == w.s0) {
                    // Test hook: the first slab of item 0 (a phase-3 tile in
                    // every launch r >= 0) is never issued, so the consumers'
                    // bounded wait on it must run out (APSP_ETIMEOUT).
                    ++g;
                    continue;
                }
                const uint32_t dst = rdst + st * FZ_STAGE;
                if (w.kind == kItemP3) {
                    constexpr int PK = kPanelPack<T>;  // panels k-pair interleaved when 2
                    mbar_arrive_expect_tx(bar_full + 8 * st, FZ_STAGE);
                    tma_load_2d(dst, &maps.colpT[pb], w.I * TB * PK, s * (KS / PK), bar_full + 8 * st);
                    tma_load_2d(dst + FZ_SLAB, &maps.rowp[pb], w.J * TB * PK, s * (KS / PK), bar_full + 8 * st);
                } else if (w.kind == kItemP2Row) {
                    mbar_arrive_expect_tx(bar_full + 8 * st, FZ_SLAB);
                    tma_load_2d(dst, &maps.primT, 0, s * KS, bar_full + 8 * st);
                } else {
                    mbar_arrive_expect_tx(bar_full + 8 * st, FZ_SLAB);
                    tma_load_2d(dst + FZ_SLAB, &maps.prim, 0, s * KS, bar_full + 8 * st);
                }
                ++g;
            }
            if (!ok) break;
            if (merged) {
                // this item's slabs are issued: merge the previous tile (its
                // consumers are finishing it now)
                ok = merge_pending();
                pw = w;
                pend = true;
                if (!ok) break;
            }
        }
        (void)nbuf;
        if (!ok) {
            // Drain every copy still in flight before the CTA may exit.
            for (uint32_t q = (g > FZ_STAGES ? g - FZ_STAGES : 0); q < g; ++q)
                mbar_wait_bounded(bar_full + 8 * (q % FZ_STAGES), (q / FZ_STAGES) & 1, err, timeout_ns,
                                  false);
            if (it > 0) mbar_wait_bounded(bar_cfull, (it - 1) & 1, err, timeout_ns, false);
        }
        bulk_wait_all();  // no reduction may still read shared memory or write D
        return;
    }

    // ====================================================== consumers
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(FZ_REG_CONSUMER));
    const MMLayout L(tid);
    const int lane = tid & 31;
    const int pb = r & 1, nbuf = rn & 1;
    uint32_t g = 0;
    uint32_t staged = 0;  // merge epilogue: tiles staged so far
    for (int it = 0;; ++it) {
        if (!mbar_wait_bounded(bar_cfull, it & 1, err, timeout_ns)) return;
        const int p0 = slots[2 * (it & 1)];
        if (p0 == -1) return;
        const int p1 = slots[2 * (it & 1) + 1];
        FusedItem w;
        w.kind = p0 & 15;
        w.crit = (p0 >> 4) & 15;
        w.s0 = (p0 >> 8) & 255;
        w.s1 = (p0 >> 16) & 255;
        w.I = (int)((unsigned)p1 >> 16);
        w.J = p1 & 0xFFFF;
        const int row0 = w.I * TB, col0 = w.J * TB;

        if (w.kind == kItemP3) {
            // ------------------------------------------------ phase 3 (round r)
            // The accumulators start at INF instead of the D tile; the tile
            // is staged in the C buffer and the producer's TMA reduction
            // takes D <- min(D, tile) in L2.  min(D, INF, products) equals
            // min(clamp(D), products), so this also clamps inputs above INF.
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cempty);  // the slot has been read
            T acc[8][8];
#pragma unroll
            for (int ri = 0; ri < 8; ++ri)
#pragma unroll
                for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = Sem<T>::inf();
            for (int q = 0; q < per; ++q, ++g) {  // the item's k-slabs, in ring order
                const uint32_t st = g % FZ_STAGES, use = g / FZ_STAGES;
                if (!mbar_wait_bounded(bar_full + 8 * st, use & 1, err, timeout_ns)) return;
                const T* As = reinterpret_cast<const T*>(ring + st * FZ_STAGE);
                if constexpr (kPanelPack<T> == 2)
                    mm_core_packed<T, KS, 2>(acc, As, As + KS * TB, L);  // k-pair interleaved slabs
                else
                    mm_core_fused<T, KS, 8>(acc, As, As + KS * TB, L);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            }
            // the previous staged tile must have been read by its reduction
            if (staged > 0 && !mbar_wait_bounded(bar_sfree, (staged - 1) & 1, err, timeout_ns)) return;
#pragma unroll
            for (int ri = 0; ri < 8; ++ri) {
                vstore4(cbuf + L.row(ri) * TB + L.cB0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
                vstore4(cbuf + L.row(ri) * TB + L.cB1, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
            }
            // the reduction reads the buffer through the async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_staged);
            ++staged;
            continue;
        }

        if (w.kind == kItemP1) {
            // ------------------------------------------------ phase 1 (round rn)
            // 16 x 16 thread grid, 8 x 8 per thread: rows 8 gq.., cols 8 hq..
            const int gq = tid >> 4, hq = tid & 15;
            const int i0 = 8 * gq, j0 = 8 * hq;
            T v[8][8];
#pragma unroll
            for (int ri = 0; ri < 8; ++ri) {
                lds4(cbuf + (i0 + ri) * TB + j0, &v[ri][0]);
                lds4(cbuf + (i0 + ri) * TB + j0 + 4, &v[ri][4]);
#pragma unroll
                for (int ci = 0; ci < 8; ++ci) {
                    v[ri][ci] = Sem<T>::clamp(v[ri][ci]);
                    if (row0 + i0 + ri >= n || col0 + j0 + ci >= n) v[ri][ci] = Sem<T>::inf();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cempty);
            if (gq == 0) {
                vstore4(p1row + j0, v[0][0], v[0][1], v[0][2], v[0][3]);
                vstore4(p1row + j0 + 4, v[0][4], v[0][5], v[0][6], v[0][7]);
            }
            if (hq == 0) {
                vstore4(p1col + i0, v[0][0], v[1][0], v[2][0], v[3][0]);
                vstore4(p1col + i0 + 4, v[4][0], v[5][0], v[6][0], v[7][0]);
            }
            consumer_barrier();
#pragma unroll 2  // 7% fewer cycles per k-step than rolled (measured)
            for (int kc = 0; kc < TB / 8; ++kc) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int k = kc * 8 + kk;
                    const int buf = kk & 1;
                    T a[8], b[8];
                    lds4(p1col + buf * TB + i0, a);
                    lds4(p1col + buf * TB + i0 + 4, a + 4);
                    lds4(p1row + buf * TB + j0, b);
                    lds4(p1row + buf * TB + j0 + 4, b + 4);
#pragma unroll
                    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
                        for (int ci = 0; ci < 8; ++ci) v[ri][ci] = Sem<T>::relax(v[ri][ci], a[ri], b[ci]);
                    if (k + 1 < TB) {
                        const int rr = (kk + 1) & 7;  // compile-time register row/column of k+1
                        const int grp = kk < 7 ? kc : kc + 1;
                        if (gq == grp) {
                            vstore4(p1row + (buf ^ 1) * TB + j0, v[rr][0], v[rr][1], v[rr][2], v[rr][3]);
                            vstore4(p1row + (buf ^ 1) * TB + j0 + 4, v[rr][4], v[rr][5], v[rr][6], v[rr][7]);
                        }
                        if (hq == grp) {
                            vstore4(p1col + (buf ^ 1) * TB + i0, v[0][rr], v[1][rr], v[2][rr], v[3][rr]);
                            vstore4(p1col + (buf ^ 1) * TB + i0 + 4, v[4][rr], v[5][rr], v[6][rr], v[7][rr]);
                        }
                        consumer_barrier();
                    }
                }
            }
            T* prim = static_cast<T*>(ptrs.prim);
            T* primT = static_cast<T*>(ptrs.primT);
#pragma unroll
            for (int ri = 0; ri < 8; ++ri) {
                const int i = i0 + ri;
                gstore4(D, ld, n, row0 + i, col0 + j0, true, v[ri][0], v[ri][1], v[ri][2], v[ri][3]);
                gstore4(D, ld, n, row0 + i, col0 + j0 + 4, true, v[ri][4], v[ri][5], v[ri][6], v[ri][7]);
                vstore4(prim + i * TB + j0, v[ri][0], v[ri][1], v[ri][2], v[ri][3]);
                vstore4(prim + i * TB + j0 + 4, v[ri][4], v[ri][5], v[ri][6], v[ri][7]);
            }
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) {
                vstore4(primT + (j0 + ci) * TB + i0, v[0][ci], v[1][ci], v[2][ci], v[3][ci]);
                vstore4(primT + (j0 + ci) * TB + i0 + 4, v[4][ci], v[5][ci], v[6][ci], v[7][ci]);
            }
            flag_signal(ptrs.flag_p1, rn);
            continue;
        }

        T acc[8][8];
        load_tile(acc, cbuf, L);

        if (w.kind == kItemFin) {
            // ------------- finisher: panel copy of a split phase-2 tile
            // All parts have merged into D, so the tile loaded is final (and
            // at most INF).  Write the copy that the next launch's phase 3
            // reads: the row panel as is, the column panel transposed.
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cempty);
            mask_outside(acc, L, row0, col0, n);
            if (w.I == rn)
                store_row_panel(static_cast<T*>(nbuf ? ptrs.rowp[1] : ptrs.rowp[0]), acc, L, col0, npad);
            else
                store_col_panel(static_cast<T*>(nbuf ? ptrs.colpT[1] : ptrs.colpT[0]), acc, L, row0, npad);
            continue;
        }

        if (r <= 0) {  // from launch 1 on, every tile read was stored (clamped) by an earlier round
#pragma unroll
            for (int ri = 0; ri < 8; ++ri)
#pragma unroll
                for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = Sem<T>::clamp(acc[ri][ci]);
        }

        if (w.kind == kItemP2Row) {
            // -------------------------------- phase 2, row panel tile (rn, J)
            // B is the tile itself: put the clamped, edge-masked values back in
            // the shared buffer, then run the product over A slabs (P^T).
            mask_outside(acc, L, row0, col0, n);
            consumer_barrier();  // every warp has read the raw tile
#pragma unroll
            for (int ri = 0; ri < 8; ++ri) {
                vstore4(cbuf + L.row(ri) * TB + L.cB0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
                vstore4(cbuf + L.row(ri) * TB + L.cB1, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
            }
            // the buffer is refilled by TMA later: order these writes first
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            consumer_barrier();
            for (int s = w.s0; s < w.s1; ++s, ++g) {
                const uint32_t st = g % FZ_STAGES, use = g / FZ_STAGES;
                if (!mbar_wait_bounded(bar_full + 8 * st, use & 1, err, timeout_ns)) return;
                const T* As = reinterpret_cast<const T*>(ring + st * FZ_STAGE);
                mm_core_fused<T, KS, 8, 1>(acc, As, cbuf + s * KS * TB, L);  // phase 2: not unrolled
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cempty);
            if (split > 1) {
                consumer_barrier();  // every warp is done with the tile as B
            } else {
#pragma unroll
                for (int ri = 0; ri < 8; ++ri) {
                    const int i = L.row(ri);
                    gstore4(D, ld, n, row0 + i, col0 + L.cB0, true, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
                    gstore4(D, ld, n, row0 + i, col0 + L.cB1, true, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
                }
                store_row_panel(static_cast<T*>(nbuf ? ptrs.rowp[1] : ptrs.rowp[0]), acc, L, col0, npad);
                continue;
            }
        } else {
            // ----------------------------- phase 2, column panel tile (I, rn)
            // A is the tile's transpose: the consumers write it (the columns
            // of this item's k-slabs) into the A halves of the ring stages
            // this item uses, then run the product over B slabs (P).
            mask_outside(acc, L, row0, col0, n);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cempty);
            consumer_barrier();  // every warp is done with the stages' previous use
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) {
                const int k = L.col(ci);
                const int sk = k / KS;
                if (sk >= w.s0 && sk < w.s1) {
                    T* Ast = reinterpret_cast<T*>(ring + ((g + sk - w.s0) % FZ_STAGES) * FZ_STAGE) + (k % KS) * TB;
                    vstore4(Ast + L.rA0, acc[0][ci], acc[1][ci], acc[2][ci], acc[3][ci]);
                    vstore4(Ast + L.rA1, acc[4][ci], acc[5][ci], acc[6][ci], acc[7][ci]);
                }
            }
            // these stages are refilled by TMA later: order these writes first
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            consumer_barrier();
            for (int s = w.s0; s < w.s1; ++s, ++g) {
                const uint32_t st = g % FZ_STAGES, use = g / FZ_STAGES;
                if (!mbar_wait_bounded(bar_full + 8 * st, use & 1, err, timeout_ns)) return;
                const T* As = reinterpret_cast<const T*>(ring + st * FZ_STAGE);
                mm_core_fused<T, KS, 8, 1>(acc, As, As + KS * TB, L);  // phase 2: not unrolled
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            }
            if (split == 1) {
#pragma unroll
                for (int ri = 0; ri < 8; ++ri) {
                    const int i = L.row(ri);
                    gstore4(D, ld, n, row0 + i, col0 + L.cB0, true, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
                    gstore4(D, ld, n, row0 + i, col0 + L.cB1, true, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
                }
                store_col_panel(static_cast<T*>(nbuf ? ptrs.colpT[1] : ptrs.colpT[0]), acc, L, row0, npad);
                continue;
            }
        }
        // A part of a split phase-2 tile: stage it for the producer's merge
        // into D (the panel copy is the finisher's job, once every part has
        // merged).  Its accumulators started from the tile itself.
        if (staged > 0 && !mbar_wait_bounded(bar_sfree, (staged - 1) & 1, err, timeout_ns)) return;
#pragma unroll
        for (int ri = 0; ri < 8; ++ri) {
            vstore4(cbuf + L.row(ri) * TB + L.cB0, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
            vstore4(cbuf + L.row(ri) * TB + L.cB1, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_staged);
        ++staged;
    }
}

}  // namespace apsp
