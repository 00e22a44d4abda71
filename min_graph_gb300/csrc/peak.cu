// Relaxation-step throughput microbenchmark (see include/apsp_peak.h).
//
// Each thread keeps an 8 x 8 block of independent accumulators, like the
// phase-3 tile product.  An empty asm statement marks the operands as changed
// on every iteration, so the compiler can neither hoist nor fold the
// repeated min operations.  It emits no instruction.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/apsp_peak.h"

namespace {

__device__ __forceinline__ void touch(int32_t& x) { asm volatile("" : "+r"(x)); }
__device__ __forceinline__ void touch(float& x) { asm volatile("" : "+f"(x)); }

template <int V>
struct Op;

template <>
struct Op<0> {  // fused add-min
    using T = int32_t;
    static constexpr int kPerStep = 1;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return __viaddmin_s32(a[ri], b[ci], acc);
    }
};
template <>
struct Op<1> {  // add, then min
    using T = int32_t;
    static constexpr int kPerStep = 1;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return min(acc, a[ri] + b[ci]);
    }
};
template <>
struct Op<2> {  // two relaxations per three-input min
    using T = int32_t;
    static constexpr int kPerStep = 2;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return __vimin3_s32(acc, a[ri] + b[ci], a[8 + ri] + b[8 + ci]);
    }
};
template <>
struct Op<3> {  // fp32 add, then min
    using T = float;
    static constexpr int kPerStep = 1;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return fminf(acc, __fadd_rn(a[ri], b[ci]));
    }
};
template <>
struct Op<4> {  // fp32, two relaxations per step
    using T = float;
    static constexpr int kPerStep = 2;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return fminf(acc, fminf(__fadd_rn(a[ri], b[ci]), __fadd_rn(a[8 + ri], b[8 + ci])));
    }
};

template <int V>
__global__ void peak_kernel(const typename Op<V>::T* __restrict__ in, typename Op<V>::T* __restrict__ out,
                            long long* __restrict__ cycles, int iters) {
    using T = typename Op<V>::T;
    T a[16], b[16], acc[8][8];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        a[q] = in[(threadIdx.x + q) & 255];
        b[q] = in[(threadIdx.x + 7 * q + 3) & 255];
    }
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = in[(ri * 8 + ci + threadIdx.x) & 255];
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int q = 0; q < 16; ++q) { touch(a[q]); touch(b[q]); }
#pragma unroll
        for (int ri = 0; ri < 8; ++ri)
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = Op<V>::step(acc[ri][ci], a, b, ri, ci);
    }
    __syncthreads();
    const long long t1 = clock64();
    T r = acc[0][0];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) r = (ri + ci) ? (r < acc[ri][ci] ? r : acc[ri][ci]) : r;
    out[blockIdx.x * blockDim.x + threadIdx.x] = r;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int V>
int run(int blocks, int threads, int iters, double* rpc, double* ms_out, long long* total_out) {
    using T = typename Op<V>::T;
    T* in = nullptr;
    T* out = nullptr;
    long long* cyc = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // The clock-based rate assumes every block is resident at once.
    int per_sm = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, peak_kernel<V>, threads, 0);
    if (e == cudaSuccess && (long long)per_sm * sms < blocks) return -2;
    if (e == cudaSuccess) e = cudaMalloc(&in, 256 * sizeof(T));
    if (e == cudaSuccess) e = cudaMalloc(&out, (size_t)blocks * threads * sizeof(T));
    if (e == cudaSuccess) e = cudaMalloc(&cyc, (size_t)blocks * sizeof(long long));
    if (e == cudaSuccess) e = cudaMemset(in, 0, 256 * sizeof(T));
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) {
        peak_kernel<V><<<blocks, threads>>>(in, out, cyc, 1);  // warm-up
        cudaEventRecord(e0);
        peak_kernel<V><<<blocks, threads>>>(in, out, cyc, iters);
        cudaEventRecord(e1);
        e = cudaEventSynchronize(e1);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        long long* hc = new long long[blocks];
        e = cudaMemcpy(hc, cyc, (size_t)blocks * sizeof(long long), cudaMemcpyDeviceToHost);
        long long maxc = 1;
        for (int i = 0; i < blocks; ++i) maxc = hc[i] > maxc ? hc[i] : maxc;
        delete[] hc;
        const long long total = (long long)blocks * threads * (long long)iters * 64 * Op<V>::kPerStep;
        if (rpc) *rpc = (double)total / ((double)maxc * (double)(sms > 0 ? sms : 1));
        if (ms_out) *ms_out = ms;
        if (total_out) *total_out = total;
    }
    if (e != cudaSuccess) rc = (int)e;
    cudaFree(in);
    cudaFree(out);
    cudaFree(cyc);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return rc;
}

}  // namespace

extern "C" int apsp_peak_variants(void) { return 5; }

extern "C" int apsp_peak_addmin(int variant, int blocks, int threads, int iters, double* rpc,
                                double* ms, long long* total) {
    if (blocks <= 0 || threads <= 0 || threads > 1024 || iters <= 0) return -1;
    switch (variant) {
        case 0: return run<0>(blocks, threads, iters, rpc, ms, total);
        case 1: return run<1>(blocks, threads, iters, rpc, ms, total);
        case 2: return run<2>(blocks, threads, iters, rpc, ms, total);
        case 3: return run<3>(blocks, threads, iters, rpc, ms, total);
        case 4: return run<4>(blocks, threads, iters, rpc, ms, total);
        default: return -1;
    }
}
