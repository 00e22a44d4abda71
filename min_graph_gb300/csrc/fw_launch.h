// Internal launch interface between the C-ABI round driver (apsp_api.cu)
// and the per-type kernel translation units (fw_i32.cu, fw_f32.cu).
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

namespace apsp {

// Everything one round's launches need.  Pointers are device pointers.
struct RoundArgs {
    void* d;        // n x n matrix, leading dimension ld
    long long ld;
    int n;
    int nb;         // number of tiles per axis, ceil(n / TB)
    int vec;        // 1: d is 16-byte aligned and ld % 4 == 0
    void* rowp;     // workspace: row panel, TB x npad
    void* colpT;    // workspace: column panel transposed, TB x npad
    void* prim;     // workspace: closed primary tile, TB x TB
    void* primT;    // workspace: its transpose
    int npad;       // nb * TB
    int tma;        // 1: the persistent TMA phase 3 may run (tensor maps valid)
    int sms;        // SM count of the device (persistent grid size)
    int* err;       // device error word (bounded-wait timeouts)
    unsigned long long timeout_ns;  // bound on every device-side wait
    int inject;     // test hook: persistent phase 3 skips one slab (forces a timeout)
    int p3_cols;    // persistent phase 3 accumulator columns per thread: 8 or 4
    int p3_stages;  // persistent phase 3 slab ring depth: 4 or 5 (8 columns only)
    CUtensorMap tm_c;   // D, n x n, box TB x TB
    CUtensorMap tm_a;   // colpT, TB x npad, box KS x TB
    CUtensorMap tm_b;   // rowp,  TB x npad, box KS x TB
};

// Tensor maps and buffers of the round-fused schedule (fw_fused.cuh).
struct FusedMaps {
    CUtensorMap c;          // D: n x n, box TB x TB
    CUtensorMap cmin;       // the same view of D typed INT32: the phase-3 min-reduction's element type
    CUtensorMap rowp[2];    // row panel buffers (alternate rounds): TB x npad, box KS x TB
    CUtensorMap colpT[2];   // transposed column panel buffers
    CUtensorMap prim;       // closed primary tile TB x TB, box KS x TB
    CUtensorMap primT;      // its transpose
};

struct FusedPtrs {
    void* rowp[2];
    void* colpT[2];
    void* prim;
    void* primT;
    int* flag_diag;   // [1]   round-stamped completion flags
    int* flag_p1;     // [1]
    int* flag_row;    // [nb]
    int* flag_col;    // [nb]
    int* counters;    // [nb + 1]: item counter of launch r at index r + 1
    int* parts;       // [2 nb + 1]: parts of each critical tile merged so far in this launch
    int* err;
};

struct FusedArgs {
    void* d;
    long long ld;
    int n, nb, npad, sms;
    unsigned long long timeout_ns;
    int inject;     // test hook: withhold one k-slab in this launch (forces a timeout)
    int split;      // items per phase-3 tile along k: 1, 2 or 4
    int overlap;    // 1: launches r >= 0 may start while launch r - 1 drains (programmatic dependent launch)
    FusedMaps maps;
    FusedPtrs ptrs;
};

// Items per phase-3 tile along k in the round-fused schedule (1, 2 or 4; it
// divides the tile's four k-slabs).  A launch with fewer than four tiles per
// SM splits its tiles by 4, so that it fills the GPU and each round's
// critical tiles (on the path through phase 1 and phase 2) finish sooner.
inline int fused_split(int nb, int sms) { return (long long)nb * nb < 4LL * sms ? 4 : 1; }

// Panel layout of the round-fused schedule, per element type.  1: k-major
// (panel row k holds D[k][j], or D[i][k] for the transposed column panel).
// 2: k-pair interleaved, element (k, x) at row k / 2, column 2x + k % 2 of a
// panel twice as wide and half as high, so that phase 3 reads both k-steps
// of a pair in one 64-bit operand.  fp32 uses 2 (a packed add.rn.f32x2 and
// a three-input minimum per two relaxations); int32 uses 1 (its fused
// add-min takes one k-step at a time).
template <typename T>
constexpr int kPanelPack = std::is_same<T, float>::value ? 2 : 1;

// Opt the kernels into their shared-memory sizes on the current device.
template <typename T> cudaError_t kernels_init();
template <typename T> cudaError_t launch_phase1(const RoundArgs& a, int r, cudaStream_t s);
template <typename T> cudaError_t launch_phase2(const RoundArgs& a, int r, cudaStream_t s);
template <typename T> cudaError_t launch_phase3(const RoundArgs& a, int r, cudaStream_t s);

// Launch r of the round-fused schedule (r = -1: prologue).  Returns
// cudaSuccess without launching when the launch has no work items.
template <typename T> cudaError_t launch_fused(const FusedArgs& a, int r, cudaStream_t s);

// Small matrices (n <= kSmallMaxN) run in one launch of a thread-block
// cluster (fw_cluster.cuh).  small_cluster_size<T>() is the cluster size the
// current device can place (16, else 8), or 0 if neither.
constexpr int kSmallMaxN = 512;
template <typename T> int small_cluster_size();
template <typename T> cudaError_t launch_small(T* d, long long ld, int n, int vec, int cluster, cudaStream_t s);

// Bytes of workspace the round driver needs for n vertices: the device
// error word, the panels and primary tiles of the three-kernel schedule,
// then the second panel buffers, flags and counters of the fused schedule.
size_t workspace_bytes(int n);

// k-slab depth of the persistent phase 3 (the panel tensor maps' box height).
int phase3_slab_rows();

}  // namespace apsp
