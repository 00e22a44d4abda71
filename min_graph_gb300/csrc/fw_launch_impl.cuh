// Launch wrappers for one element type; included once per type by
// fw_i32.cu and fw_f32.cu so that the two instantiations compile in parallel.
#pragma once

#include "fw_cluster.cuh"
#include "fw_fused.cuh"
#include "fw_kernels.cuh"
#include "fw_launch.h"

namespace apsp {

static_assert(kSmallMaxN == SC_MAX_N, "small-matrix limit out of date");

template <typename T>
cudaError_t small_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int cluster, cudaStream_t s) {
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)cluster);
    cfg->blockDim = dim3(SC_THREADS);
    cfg->dynamicSmemBytes = sc_smem_bytes<T>();
    cfg->stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    return cudaSuccess;
}

template <typename T>
int small_cluster_size_impl() {
    // 16 CTAs is beyond the portable cluster size: opt in, then ask the
    // device whether it can place one such cluster at all.
    if (cudaFuncSetAttribute(fw_cluster_small<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sc_smem_bytes<T>()) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cudaFuncSetAttribute(fw_cluster_small<T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
        cudaGetLastError();
    const int sizes[2] = {16, 8};
    for (int c : sizes) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[1];
        small_config<T>(&cfg, attr, c, nullptr);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fw_cluster_small<T>, &cfg) == cudaSuccess && clusters > 0)
            return c;
        cudaGetLastError();
    }
    return 0;
}

template <typename T>
cudaError_t launch_small_impl(T* d, long long ld, int n, int vec, int cluster, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    small_config<T>(&cfg, attr, cluster, s);
    return cudaLaunchKernelEx(&cfg, fw_cluster_small<T>, d, ld, n, vec);
}

template <typename T>
cudaError_t kernels_init_impl() {
    // Load phase 1 now too (it needs no attribute): under lazy module loading
    // a kernel is loaded at its first use, and that load may allocate.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fw_phase1_diag<T>);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fw_phase2_panels<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPhase2Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fw_phase3_minplus<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPhase3Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fw_phase3_persistent<T, 8, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)phase3p_smem(4));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fw_phase3_persistent<T, 8, 5>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)phase3p_smem(5));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fw_phase3_persistent<T, 4, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)phase3p_smem(4));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fw_round_fused<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kFusedSmem);
}

template <typename T>
cudaError_t launch_fused_impl(const FusedArgs& a, int r, cudaStream_t s) {
    const long long items = fused_items(r, a.nb, a.split);
    if (items <= 0) return cudaSuccess;
    const int grid = (int)(items < a.sms ? items : a.sms);
    // Launches after the prologue follow another launch of this kernel on the
    // stream: let them start (barrier setup) while that one drains.  The
    // kernel waits for its predecessor's completion before it reads memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(FZ_THREADS);
    cfg.dynamicSmemBytes = kFusedSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (r >= 0 && a.overlap) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fw_round_fused<T>, static_cast<T*>(a.d), a.ld, a.n, r, a.nb, a.npad,
                              (int)items, a.split, a.maps, a.ptrs, a.timeout_ns, a.inject);
}

template <typename T>
cudaError_t launch_phase1_impl(const RoundArgs& a, int r, cudaStream_t s) {
    fw_phase1_diag<T><<<1, P1_THREADS, 0, s>>>(static_cast<T*>(a.d), a.ld, a.n, r,
                                               static_cast<T*>(a.prim), static_cast<T*>(a.primT),
                                               a.vec);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_phase2_impl(const RoundArgs& a, int r, cudaStream_t s) {
    if (a.nb < 2) return cudaSuccess;
    fw_phase2_panels<T><<<dim3(a.nb - 1, 2), MM_THREADS, kPhase2Smem, s>>>(
        static_cast<T*>(a.d), a.ld, a.n, r, static_cast<T*>(a.rowp), static_cast<T*>(a.colpT),
        static_cast<const T*>(a.prim), static_cast<const T*>(a.primT), a.npad, a.vec);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_phase3_impl(const RoundArgs& a, int r, cudaStream_t s) {
    if (a.nb < 2) return cudaSuccess;
    const unsigned tiles = (unsigned)(a.nb - 1) * (unsigned)(a.nb - 1);
    if (a.tma) {
        const unsigned grid = tiles < (unsigned)a.sms ? tiles : (unsigned)a.sms;
        if (a.p3_cols == 4)
            fw_phase3_persistent<T, 4, 4><<<grid, p3p_threads<4>(), phase3p_smem(4), s>>>(
                static_cast<T*>(a.d), a.ld, a.n, r, a.nb - 1, (int)tiles, a.tm_c, a.tm_a, a.tm_b,
                a.err, a.timeout_ns, a.inject);
        else if (a.p3_stages == 5)
            fw_phase3_persistent<T, 8, 5><<<grid, p3p_threads<8>(), phase3p_smem(5), s>>>(
                static_cast<T*>(a.d), a.ld, a.n, r, a.nb - 1, (int)tiles, a.tm_c, a.tm_a, a.tm_b,
                a.err, a.timeout_ns, a.inject);
        else
            fw_phase3_persistent<T, 8, 4><<<grid, p3p_threads<8>(), phase3p_smem(4), s>>>(
                static_cast<T*>(a.d), a.ld, a.n, r, a.nb - 1, (int)tiles, a.tm_c, a.tm_a, a.tm_b,
                a.err, a.timeout_ns, a.inject);
        return cudaGetLastError();
    }
    fw_phase3_minplus<T><<<tiles, MM_THREADS, kPhase3Smem, s>>>(
        static_cast<T*>(a.d), a.ld, a.n, r, a.nb - 1, static_cast<const T*>(a.rowp),
        static_cast<const T*>(a.colpT), a.npad, a.vec);
    return cudaGetLastError();
}

}  // namespace apsp

#define APSP_INSTANTIATE_LAUNCHERS(T)                                                            \
    namespace apsp {                                                                             \
    template <> cudaError_t kernels_init<T>() { return kernels_init_impl<T>(); }                \
    template <> cudaError_t launch_phase1<T>(const RoundArgs& a, int r, cudaStream_t s) {        \
        return launch_phase1_impl<T>(a, r, s);                                                   \
    }                                                                                            \
    template <> cudaError_t launch_phase2<T>(const RoundArgs& a, int r, cudaStream_t s) {        \
        return launch_phase2_impl<T>(a, r, s);                                                   \
    }                                                                                            \
    template <> cudaError_t launch_phase3<T>(const RoundArgs& a, int r, cudaStream_t s) {        \
        return launch_phase3_impl<T>(a, r, s);                                                   \
    }                                                                                            \
    template <> cudaError_t launch_fused<T>(const FusedArgs& a, int r, cudaStream_t s) {         \
        return launch_fused_impl<T>(a, r, s);                                                    \
    }                                                                                            \
    template <> int small_cluster_size<T>() { return small_cluster_size_impl<T>(); }            \
    template <> cudaError_t launch_small<T>(T* d, long long ld, int n, int vec, int cluster,     \
                                            cudaStream_t s) {                                    \
        return launch_small_impl<T>(d, ld, n, vec, cluster, s);                                  \
    }                                                                                            \
    }
