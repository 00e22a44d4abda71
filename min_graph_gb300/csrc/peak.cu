// Relaxation-step throughput microbenchmark (see include/apsp_peak.h).
//
// Each thread keeps an 8 x 8 block of independent accumulators, like the
// phase-3 tile product.  An empty asm statement marks the operands as changed
// on every iteration, so the compiler can neither hoist nor fold the
// repeated min operations.  It emits no instruction.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/apsp_peak.h"
#include "mm_core.cuh"

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

// Variants 5-7 take an opaque 1 (`one`, marked changed each iteration like
// the operands) so that a * one + b stays a multiply-add.
template <>
struct Op<5> {  // int32 adds as multiply-add, three-input integer min
    using T = int32_t;
    static constexpr int kPerStep = 2;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        return __vimin3_s32(acc, a[ri] * a[15] + b[ci], a[8 + ri] * a[15] + b[8 + ci]);
    }
};
template <>
struct Op<6> {  // int32 adds, fp32 three-input min over the non-negative bit patterns
    using T = int32_t;
    static constexpr int kPerStep = 2;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        const float m = fminf(__int_as_float(acc), fminf(__int_as_float(a[ri] + b[ci]),
                                                         __int_as_float(a[8 + ri] + b[8 + ci])));
        return __float_as_int(m);
    }
};
template <>
struct Op<7> {  // int32 adds as multiply-add, fp32 three-input min over bit patterns
    using T = int32_t;
    static constexpr int kPerStep = 2;
    __device__ static __forceinline__ T step(T acc, const T* a, const T* b, int ri, int ci) {
        const float m = fminf(__int_as_float(acc),
                              fminf(__int_as_float(a[ri] * a[15] + b[ci]),
                                    __int_as_float(a[8 + ri] * a[15] + b[8 + ci])));
        return __float_as_int(m);
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
    if (V >= 5) a[15] = (T)1;  // the opaque multiplier (in[] is all zeros)
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

// Shared-memory-fed probe: the real phase-3 inner loop (mm_core) run over a
// resident 32-deep slab of operands, `iters` times.  Operands come from
// shared memory exactly as in the kernels, so nothing can be hoisted out of
// the loop.  Variant ids >= 8 select (type, core):
//   8 int32 fused, 9 int32 min3, 10 int32 packed,
//   11 fp32 fused, 12 fp32 min3, 13 fp32 packed.
template <typename T, int CORE, int MINB>
__global__ void __launch_bounds__(256, MINB)
core_kernel(const T* __restrict__ in, T* __restrict__ out, long long* __restrict__ cycles, int iters,
            int one) {
    constexpr int KLEN = 32;
    extern __shared__ __align__(16) unsigned char core_smem[];
    T* As = reinterpret_cast<T*>(core_smem);
    T* Bs = As + KLEN * apsp::TB;
    for (int q = threadIdx.x; q < 2 * KLEN * apsp::TB; q += blockDim.x) As[q] = in[q & 255];
    __syncthreads();
    const apsp::MMLayout L(threadIdx.x);
    T acc[8][8];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) acc[ri][ci] = in[(ri * 8 + ci + threadIdx.x) & 255];
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) apsp::mm_core<T, CORE, KLEN>(acc, As, Bs, L, one);
    __syncthreads();
    const long long t1 = clock64();
    T r = acc[0][0];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri)
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) r = r < acc[ri][ci] ? r : acc[ri][ci];
    out[blockIdx.x * blockDim.x + threadIdx.x] = r;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <typename T, int CORE, int MINB = 1>
int run_core(int blocks, int iters, double* rpc, double* ms_out, long long* total_out) {
    const int threads = 256;
    const size_t smem = 2 * 32 * apsp::TB * sizeof(T);
    T* in = nullptr;
    T* out = nullptr;
    long long* cyc = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(core_kernel<T, CORE, MINB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, core_kernel<T, CORE, MINB>, threads, smem);
    if (e == cudaSuccess && (long long)per_sm * sms < blocks) return -2;
    if (e == cudaSuccess) e = cudaMalloc(&in, 256 * sizeof(T));
    if (e == cudaSuccess) e = cudaMalloc(&out, (size_t)blocks * threads * sizeof(T));
    if (e == cudaSuccess) e = cudaMalloc(&cyc, (size_t)blocks * sizeof(long long));
    if (e == cudaSuccess) e = cudaMemset(in, 0, 256 * sizeof(T));
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) {
        core_kernel<T, CORE, MINB><<<blocks, threads, smem>>>(in, out, cyc, 1, 1);
        cudaEventRecord(e0);
        core_kernel<T, CORE, MINB><<<blocks, threads, smem>>>(in, out, cyc, iters, 1);
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
        const long long total = (long long)blocks * threads * (long long)iters * 64 * 32;
        if (rpc) *rpc = (double)total / ((double)maxc * (double)(sms > 0 ? sms : 1));
        if (ms_out) *ms_out = ms;
        if (total_out) *total_out = total;
    }
    cudaFree(in);
    cudaFree(out);
    cudaFree(cyc);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return e == cudaSuccess ? 0 : (int)e;
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

// L2 read probe: grid-stride 16-byte loads over a buffer small enough to
// stay in L2, `passes` times; the XOR of what was read is stored once per
// thread so the loads cannot be dropped.
__global__ void l2_read_kernel(const int4* __restrict__ buf, long long n16, int passes, int* __restrict__ sink) {
    int acc = 0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (int p = 0; p < passes; ++p) {
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
            const int4 v = __ldcg(buf + i);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    }
    sink[(long long)blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

extern "C" int apsp_peak_l2_read(long long bytes, int blocks, int threads, int passes, double* gbs, double* ms) {
    if (bytes < 16 || bytes > (256ll << 20) || blocks <= 0 || threads <= 0 || threads > 1024 || passes <= 0)
        return -1;
    const long long n16 = bytes / 16;
    int4* buf = nullptr;
    int* sink = nullptr;
    cudaError_t e = cudaMalloc(&buf, n16 * 16);
    if (e == cudaSuccess) e = cudaMalloc(&sink, (size_t)blocks * threads * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(buf, 1, n16 * 16);
    cudaEvent_t a = nullptr, b = nullptr;
    if (e == cudaSuccess) e = cudaEventCreate(&a);
    if (e == cudaSuccess) e = cudaEventCreate(&b);
    float t = 0.f;
    if (e == cudaSuccess) {
        l2_read_kernel<<<blocks, threads>>>(buf, n16, 1, sink);  // warm: brings the buffer into L2
        cudaEventRecord(a);
        l2_read_kernel<<<blocks, threads>>>(buf, n16, passes, sink);
        cudaEventRecord(b);
        e = cudaEventSynchronize(b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, a, b);
    }
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
    cudaFree(buf);
    cudaFree(sink);
    if (e != cudaSuccess) return (int)e;
    if (ms) *ms = t;
    if (gbs) *gbs = (double)n16 * 16 * passes / (t * 1e-3) / 1e9;
    return 0;
}

extern "C" int apsp_peak_variants(void) { return 21; }

extern "C" int apsp_peak_addmin(int variant, int blocks, int threads, int iters, double* rpc,
                                double* ms, long long* total) {
    if (blocks <= 0 || threads <= 0 || threads > 1024 || iters <= 0) return -1;
    switch (variant) {
        case 8: return run_core<int32_t, apsp::kCoreFused>(blocks, iters, rpc, ms, total);
        case 9: return run_core<int32_t, apsp::kCoreMin3>(blocks, iters, rpc, ms, total);
        case 10: return run_core<int32_t, apsp::kCorePacked>(blocks, iters, rpc, ms, total);
        case 11: return run_core<float, apsp::kCoreFused>(blocks, iters, rpc, ms, total);
        case 12: return run_core<float, apsp::kCoreMin3>(blocks, iters, rpc, ms, total);
        case 13: return run_core<float, apsp::kCorePacked>(blocks, iters, rpc, ms, total);
        case 14: return run_core<int32_t, apsp::kCoreFused, 2>(blocks, iters, rpc, ms, total);
        case 15: return run_core<float, apsp::kCorePacked, 2>(blocks, iters, rpc, ms, total);
        case 16: return run_core<int32_t, apsp::kCoreMixAdd + 2>(blocks, iters, rpc, ms, total);
        case 17: return run_core<int32_t, apsp::kCoreMixAdd + 3>(blocks, iters, rpc, ms, total);
        case 18: return run_core<int32_t, apsp::kCoreMixMad + 2>(blocks, iters, rpc, ms, total);
        case 19: return run_core<int32_t, apsp::kCoreMixMad + 3>(blocks, iters, rpc, ms, total);
        case 20: return run_core<int32_t, apsp::kCoreMixMad + 4>(blocks, iters, rpc, ms, total);
        case 0: return run<0>(blocks, threads, iters, rpc, ms, total);
        case 1: return run<1>(blocks, threads, iters, rpc, ms, total);
        case 2: return run<2>(blocks, threads, iters, rpc, ms, total);
        case 3: return run<3>(blocks, threads, iters, rpc, ms, total);
        case 4: return run<4>(blocks, threads, iters, rpc, ms, total);
        case 5: return run<5>(blocks, threads, iters, rpc, ms, total);
        case 6: return run<6>(blocks, threads, iters, rpc, ms, total);
        case 7: return run<7>(blocks, threads, iters, rpc, ms, total);
        default: return -1;
    }
}
