// Internal launch interface between the C-ABI round driver (apsp_api.cu)
// and the per-type kernel translation units (fw_i32.cu, fw_f32.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

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
};

// Opt the kernels into their shared-memory sizes on the current device.
template <typename T> cudaError_t kernels_init();
template <typename T> cudaError_t launch_phase1(const RoundArgs& a, int r, cudaStream_t s);
template <typename T> cudaError_t launch_phase2(const RoundArgs& a, int r, cudaStream_t s);
template <typename T> cudaError_t launch_phase3(const RoundArgs& a, int r, cudaStream_t s);

// Bytes of workspace the round driver needs for n vertices.
size_t workspace_bytes(int n);

}  // namespace apsp
