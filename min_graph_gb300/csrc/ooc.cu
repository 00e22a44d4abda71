// Out-of-core blocked Floyd-Warshall (host-resident matrix), sm_103a.
//
// The thesis page (1library.co excerpt, section 4.7) names a modification
// for graphs of any size, but its text is not on the page; this is our own
// reading of it.  It is blocked Floyd-Warshall one level up: super-blocks of
// K x K (K a multiple of the 128 tile) in host memory, one super-round per
// diagonal super-block R, and the same three phases:
//   1. close D[R,R] on the GPU with the in-core solver (apsp_solve);
//   2. row panel    D[R,J] <- min(D[R,J], P (x) D[R,J])   (P = closed D[R,R])
//      column panel D[I,R] <- min(D[I,R], D[I,R] (x) P)
//      A single product with the closed P gives the exact panel, as the
//      in-core phase 2 does.  The column panel is kept transposed, and in
//      that form its update is CT <- min(CT, P^T (x) CT);
//   3. every other super-block D[I,J] <- min(D[I,J], D[I,R] (x) D[R,J]),
//      streamed through the GPU.
// (x) is the min-plus product.  The panels stay on the device for the whole
// super-round: the row panel as K x npad, the column panel transposed, also
// K x npad.  Phase 3 streams the other blocks through a ring of 3 staging
// buffers on three streams (host->device copy, product, device->host copy)
// joined by events, so copies overlap the products when the host matrix is
// pinned.  Per super-round the matrix crosses the link twice, against K
// relaxations per element, so K of a few thousand keeps the link far from
// the bottleneck.
//
// Every device buffer is padded to multiples of 128 with INF.  INF along the
// k dimension never wins a minimum (INF + x >= INF >= any stored value), and
// padding rows and columns are never copied back.  Entries above INF read from
// the host are clamped to INF before any sum (int32: INF + INF < 2^31).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "../../include/apsp.h"
#include "../../include/apsp_ooc.h"
#include "fw_kernels.cuh"

namespace apsp {
void set_last_cuda_error(int e);  // defined with apsp_last_cuda_error()
}

namespace {

using apsp::KS;
using apsp::MM_THREADS;
using apsp::MMLayout;
using apsp::P3_STAGES;
using apsp::Sem;
using apsp::TB;

apsp_status_t ooc_fail(cudaError_t e) {
    apsp::set_last_cuda_error((int)e);
    return APSP_ECUDA;
}

// One 4-byte asynchronous copy global -> shared (cached in L1 and L2).
__device__ __forceinline__ void cp_async4(uint32_t smem, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem), "l"(gmem) : "memory");
}

// C (M x N, ldc) <- min(C, A (x) B) for A = AT^T (AT: K x M, lda) and B
// (K x N, ldb).  M and N are multiples of 128 and K of 32; every row starts
// 16-byte aligned.  One CTA per 128 x 128 C tile, k-slabs of 32 staged by
// cp.async through a 3-deep ring, the same register-blocked tile-product
// cores as the in-core phase 3.  int32 copies 16-byte row pieces into k-major
// slabs for the fused add-min.  fp32 runs the packed core, whose slabs hold
// k-pairs interleaved (element (k, i) at (k / 2 * 128 + i) * 2 + k % 2): each
// element is copied on its own (4 bytes), a warp's 32 copies reading 128
// consecutive bytes of one panel row.
template <typename T>
__global__ void __launch_bounds__(MM_THREADS, 1)
minplus_accum_kernel(T* __restrict__ C, long long ldc, int tiles_n, const T* __restrict__ AT, long long lda,
                     const T* __restrict__ B, long long ldb, int K) {
    extern __shared__ __align__(128) unsigned char mp_smem[];
    T* sm = reinterpret_cast<T*>(mp_smem);
    const int tid = threadIdx.x;
    const int row0 = (blockIdx.x / tiles_n) * TB, col0 = (blockIdx.x % tiles_n) * TB;
    const MMLayout L(tid);
    constexpr int SLAB = KS * TB;
    const int nslab = K / KS;
    const uint32_t sm_base = apsp::smem_u32(sm);
    const uint32_t my_sm = ((tid >> 5) * TB + (tid & 31) * 4) * 4;
    const int kk0 = tid >> 5, c4 = (tid & 31) * 4;
    constexpr bool kPacked = std::is_same<T, float>::value;
    static_assert(MM_THREADS == 2 * TB, "the packed copy gives each thread one k parity");
    auto issue = [&](int s, int st) {
        if constexpr (kPacked) {
            const int par = tid / TB, i = tid % TB;  // rows k = 2m + par of the slab, column i
            const uint32_t sa = sm_base + st * 2 * SLAB * 4 + (i * 2 + par) * 4;
#pragma unroll
            for (int m = 0; m < KS / 2; ++m) {
                const long long k = (long long)s * KS + 2 * m + par;
                cp_async4(sa + m * TB * 2 * 4, AT + k * lda + row0 + i);
                cp_async4(sa + SLAB * 4 + m * TB * 2 * 4, B + k * ldb + col0 + i);
            }
        } else {
            const uint32_t sa = sm_base + st * 2 * SLAB * 4 + my_sm;
#pragma unroll
            for (int m = 0; m < SLAB / 4 / MM_THREADS; ++m) {
                const long long k = (long long)s * KS + kk0 + m * (MM_THREADS / 32);
                apsp::cp_async16(sa + m * (MM_THREADS / 32) * TB * 4, AT + k * lda + row0 + c4);
                apsp::cp_async16(sa + SLAB * 4 + m * (MM_THREADS / 32) * TB * 4, B + k * ldb + col0 + c4);
            }
        }
        apsp::cp_async_commit();
    };
    issue(0, 0);
    if (nslab > 1) issue(1, 1);

    T acc[8][8];
#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        apsp::gload4(C, ldc, INT_MAX, row0 + L.row(ri), col0 + L.cB0, true, &acc[ri][0]);
        apsp::gload4(C, ldc, INT_MAX, row0 + L.row(ri), col0 + L.cB1, true, &acc[ri][4]);
    }
#pragma unroll 1
    for (int s = 0; s < nslab; ++s) {
        if (s + 1 < nslab)
            apsp::cp_async_wait<1>();
        else
            apsp::cp_async_wait<0>();
        __syncthreads();
        if (s + 2 < nslab) issue(s + 2, (s + 2) % P3_STAGES);
        const T* As = sm + (s % P3_STAGES) * 2 * SLAB;
        if constexpr (kPacked)
            apsp::mm_core_packed<T, KS, 2>(acc, As, As + SLAB, L);
        else
            apsp::mm_core<T, apsp::Core<T>::value, KS>(acc, As, As + SLAB, L);
    }
#pragma unroll
    for (int ri = 0; ri < 8; ++ri) {
        const int i = row0 + L.row(ri);
        apsp::gstore4(C, ldc, INT_MAX, i, col0 + L.cB0, true, acc[ri][0], acc[ri][1], acc[ri][2], acc[ri][3]);
        apsp::gstore4(C, ldc, INT_MAX, i, col0 + L.cB1, true, acc[ri][4], acc[ri][5], acc[ri][6], acc[ri][7]);
    }
}

// buf (rows_pad x cols_pad, ld): real entries clamped to INF, the rest INF.
template <typename T>
__global__ void clamp_pad_kernel(T* __restrict__ buf, long long ld, int rows, int cols, int rows_pad, int cols_pad) {
    const long long total = (long long)rows_pad * cols_pad;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(x / cols_pad), c = (int)(x % cols_pad);
        T* p = buf + (long long)r * ld + c;
        *p = (r < rows && c < cols) ? Sem<T>::clamp(*p) : Sem<T>::inf();
    }
}

// dst[c][r] = clamp(src[r][c]) over a rows_pad x cols_pad extent (INF
// outside rows x cols), through 32 x 32 shared-memory tiles.
template <typename T>
__global__ void transpose_kernel(T* __restrict__ dst, long long ldd, const T* __restrict__ src, long long lds,
                                 int rows, int cols, int rows_pad, int cols_pad) {
    __shared__ T tile[32][33];
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    for (int j = ty; j < 32; j += 8) {
        const int r = r0 + j, c = c0 + tx;
        tile[j][tx] = (r < rows && c < cols) ? Sem<T>::clamp(src[(long long)r * lds + c]) : Sem<T>::inf();
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int c = c0 + j, r = r0 + tx;  // dst row c, column r
        if (c < cols_pad && r < rows_pad) dst[(long long)c * ldd + r] = tile[tx][j];
    }
}

template <typename T>
apsp_status_t launch_minplus(T* C, long long ldc, int M, int N, const T* AT, long long lda, const T* B, long long ldb,
                             int K, cudaStream_t s) {
    const int tiles_n = N / TB;
    const int tiles = (M / TB) * tiles_n;
    const size_t smem = (size_t)P3_STAGES * 2 * KS * TB * sizeof(T);
    cudaError_t e = cudaFuncSetAttribute(minplus_accum_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return ooc_fail(e);
    minplus_accum_kernel<T><<<tiles, MM_THREADS, smem, s>>>(C, ldc, tiles_n, AT, lda, B, ldb, K);
    e = cudaGetLastError();
    return e == cudaSuccess ? APSP_OK : ooc_fail(e);
}

template <typename T>
apsp_status_t launch_clamp_pad(T* buf, long long ld, int rows, int cols, int rows_pad, int cols_pad, cudaStream_t s) {
    clamp_pad_kernel<T><<<1024, 256, 0, s>>>(buf, ld, rows, cols, rows_pad, cols_pad);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? APSP_OK : ooc_fail(e);
}

template <typename T>
apsp_status_t launch_transpose(T* dst, long long ldd, const T* src, long long lds, int rows, int cols, int rows_pad,
                               int cols_pad, cudaStream_t s) {
    dim3 grid((cols_pad + 31) / 32, (rows_pad + 31) / 32), block(32, 8);
    transpose_kernel<T><<<grid, block, 0, s>>>(dst, ldd, src, lds, rows, cols, rows_pad, cols_pad);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? APSP_OK : ooc_fail(e);
}

// A 2-D copy of rows x cols elements between host (pitch ldh) and device
// (pitch ldd).
template <typename T>
cudaError_t copy2d(T* dst, long long lddst, const T* src, long long ldsrc, int rows, int cols, cudaMemcpyKind kind,
                   cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, (size_t)lddst * sizeof(T), src, (size_t)ldsrc * sizeof(T), (size_t)cols * sizeof(T),
                             (size_t)rows, kind, s);
}

template <typename T>
apsp_status_t solve_in_core(T* d, int n, int ld, cudaStream_t s);

template <>
apsp_status_t solve_in_core<int32_t>(int32_t* d, int n, int ld, cudaStream_t s) {
    return apsp_solve_i32(d, n, ld, (apsp_stream_t)s);
}
template <>
apsp_status_t solve_in_core<float>(float* d, int n, int ld, cudaStream_t s) {
    return apsp_solve_f32(d, n, ld, (apsp_stream_t)s);
}

// Elements of device memory the solver needs for super-block K: P and P^T
// (K x K each), the two panels (K x npad each), 3 staging blocks (K x K).
size_t ooc_elems(int n, int K) {
    const size_t nR = (size_t)(n + K - 1) / K;
    const size_t npad = nR * K;
    return 5 * (size_t)K * K + 2 * (size_t)K * npad;
}

// The copy-in and copy-out streams of the block ring and their events.  On
// every exit, error paths included, the streams are drained first, so the
// device buffer is never freed under a copy still in flight.
struct Streams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t loaded[3] = {}, done[3] = {}, freed[3] = {};
    ~Streams() {
        if (in) cudaStreamSynchronize(in);
        if (out) cudaStreamSynchronize(out);
        for (int q = 0; q < 3; ++q) {
            if (loaded[q]) cudaEventDestroy(loaded[q]);
            if (done[q]) cudaEventDestroy(done[q]);
            if (freed[q]) cudaEventDestroy(freed[q]);
        }
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};

template <typename T>
apsp_status_t solve_ooc(T* H, int n, int ld, int K, T* base, cudaStream_t s) {
    const int nR = (n + K - 1) / K;
    const long long npad = (long long)nR * K;
    const long long KK = (long long)K * K;
    T* P = base;
    T* PT = P + KK;
    T* RP = PT + KK;
    T* CPT = RP + (long long)K * npad;
    T* stage[3] = {CPT + (long long)K * npad, CPT + (long long)K * npad + KK, CPT + (long long)K * npad + 2 * KK};

    Streams st;
    cudaError_t e = cudaStreamCreateWithFlags(&st.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st.out, cudaStreamNonBlocking);
    for (int q = 0; q < 3 && e == cudaSuccess; ++q) {
        e = cudaEventCreateWithFlags(&st.loaded[q], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.done[q], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.freed[q], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return ooc_fail(e);
    apsp_status_t rc;

    for (int R = 0; R < nR; ++R) {
        const int r0 = R * K, kr = std::min(K, n - r0);
        // 1. close the diagonal super-block in core
        e = copy2d(P, K, H + (long long)r0 * ld + r0, ld, kr, kr, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return ooc_fail(e);
        if ((rc = launch_clamp_pad(P, K, kr, kr, K, K, s)) != APSP_OK) return rc;
        if ((rc = solve_in_core(P, kr, K, s)) != APSP_OK) return rc;
        if ((rc = (apsp_status_t)apsp_stream_check((apsp_stream_t)s)) != APSP_OK) return rc;
        e = copy2d(H + (long long)r0 * ld + r0, ld, P, K, kr, kr, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return ooc_fail(e);
        if ((rc = launch_transpose(PT, K, P, K, K, K, K, K, s)) != APSP_OK) return rc;

        // 2a. row panel, one K-wide chunk at a time: stage <- D[R,J]; RP[:,J] <-
        //     min(stage, P (x) stage); D[R,J] <- RP[:,J]
        for (int J = 0; J < nR; ++J) {
            const int c0 = J * K, kc = std::min(K, n - c0);
            T* rpj = RP + c0;
            if (J == R) {
                e = cudaMemcpy2DAsync(rpj, npad * sizeof(T), P, K * sizeof(T), K * sizeof(T), K,
                                      cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) return ooc_fail(e);
                continue;
            }
            e = copy2d(stage[0], K, H + (long long)r0 * ld + c0, ld, kr, kc, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return ooc_fail(e);
            if ((rc = launch_clamp_pad(stage[0], K, kr, kc, K, K, s)) != APSP_OK) return rc;
            e = cudaMemcpy2DAsync(rpj, npad * sizeof(T), stage[0], K * sizeof(T), K * sizeof(T), K,
                                  cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return ooc_fail(e);
            if ((rc = launch_minplus(rpj, npad, K, K, PT, K, stage[0], K, K, s)) != APSP_OK) return rc;
            e = copy2d(H + (long long)r0 * ld + c0, ld, rpj, npad, kr, kc, cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) return ooc_fail(e);
        }
        // 2b. column panel, transposed: stage <- D[I,R]; CPT[:,I] <- min(stage^T,
        //     P^T (x) stage^T); D[I,R] <- CPT[:,I]^T
        for (int I = 0; I < nR; ++I) {
            const int i0 = I * K, ki = std::min(K, n - i0);
            T* cpti = CPT + i0;
            if (I == R) {
                e = cudaMemcpy2DAsync(cpti, npad * sizeof(T), PT, K * sizeof(T), K * sizeof(T), K,
                                      cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) return ooc_fail(e);
                continue;
            }
            e = copy2d(stage[0], K, H + (long long)i0 * ld + r0, ld, ki, kr, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return ooc_fail(e);
            if ((rc = launch_transpose(stage[1], K, stage[0], K, ki, kr, K, K, s)) != APSP_OK) return rc;
            e = cudaMemcpy2DAsync(cpti, npad * sizeof(T), stage[1], K * sizeof(T), K * sizeof(T), K,
                                  cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return ooc_fail(e);
            if ((rc = launch_minplus(cpti, npad, K, K, P, K, stage[1], K, K, s)) != APSP_OK) return rc;
            if ((rc = launch_transpose(stage[2], K, cpti, npad, K, K, K, K, s)) != APSP_OK) return rc;
            e = copy2d(H + (long long)i0 * ld + r0, ld, stage[2], K, ki, kr, cudaMemcpyDeviceToHost, s);
            if (e != cudaSuccess) return ooc_fail(e);
        }
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return ooc_fail(e);

        // 3. every other super-block through the 3-buffer ring
        for (int q = 0; q < 3; ++q) {
            e = cudaEventRecord(st.freed[q], st.out);
            if (e != cudaSuccess) return ooc_fail(e);
        }
        int b = 0;
        for (int I = 0; I < nR; ++I) {
            if (I == R) continue;
            const int i0 = I * K, ki = std::min(K, n - i0);
            for (int J = 0; J < nR; ++J, ++b) {
                if (J == R) {
                    --b;
                    continue;
                }
                const int c0 = J * K, kc = std::min(K, n - c0);
                const int q = b % 3;
                T* hblk = H + (long long)i0 * ld + c0;
                e = cudaStreamWaitEvent(st.in, st.freed[q], 0);
                if (e == cudaSuccess) e = copy2d(stage[q], K, hblk, ld, ki, kc, cudaMemcpyHostToDevice, st.in);
                if (e == cudaSuccess) e = cudaEventRecord(st.loaded[q], st.in);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(s, st.loaded[q], 0);
                if (e != cudaSuccess) return ooc_fail(e);
                if ((rc = launch_minplus(stage[q], K, K, K, CPT + i0, npad, RP + c0, npad, K, s)) != APSP_OK) return rc;
                e = cudaEventRecord(st.done[q], s);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(st.out, st.done[q], 0);
                if (e == cudaSuccess) e = copy2d(hblk, ld, stage[q], K, ki, kc, cudaMemcpyDeviceToHost, st.out);
                if (e == cudaSuccess) e = cudaEventRecord(st.freed[q], st.out);
                if (e != cudaSuccess) return ooc_fail(e);
            }
        }
        e = cudaStreamSynchronize(st.out);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return ooc_fail(e);
    }
    return APSP_OK;
}

template <typename T>
apsp_status_t solve_ooc_entry(T* host, int n, int ld, unsigned long long device_bytes, int block,
                              apsp_stream_t stream) {
    if (n < 0 || ld < n || (n > 0 && host == nullptr) || n > APSP_MAX_N) return APSP_EINVAL;
    if (block < 0 || block % TB != 0) return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    size_t budget = device_bytes;
    if (budget == 0) {
        size_t free_b = 0, total_b = 0;
        const cudaError_t e = cudaMemGetInfo(&free_b, &total_b);
        if (e != cudaSuccess) return ooc_fail(e);
        budget = free_b / 10 * 7;
    }
    const int npad128 = (n + TB - 1) / TB * TB;
    int K = block;
    if (K == 0) {  // the largest super-block (at most 16384) that fits the budget
        K = std::min(16384, npad128);
        while (K > TB && ooc_elems(n, K) * sizeof(T) > budget) K -= TB;
    }
    K = std::min(K, npad128);
    if (ooc_elems(n, K) * sizeof(T) > budget) return APSP_EINVAL;
    T* base = nullptr;
    cudaError_t e = cudaMalloc(&base, ooc_elems(n, K) * sizeof(T));
    if (e != cudaSuccess) {
        cudaGetLastError();
        apsp::set_last_cuda_error((int)e);
        return APSP_ENOMEM;
    }
    apsp_status_t rc = solve_ooc<T>(host, n, ld, K, base, s);
    cudaStreamSynchronize(s);
    cudaFree(base);
    return rc;
}

}  // namespace

extern "C" {

apsp_status_t apsp_solve_ooc_i32(int32_t* host, int n, int ld, unsigned long long device_bytes, int block,
                                 apsp_stream_t stream) {
    return solve_ooc_entry<int32_t>(host, n, ld, device_bytes, block, stream);
}

apsp_status_t apsp_solve_ooc_f32(float* host, int n, int ld, unsigned long long device_bytes, int block,
                                 apsp_stream_t stream) {
    return solve_ooc_entry<float>(host, n, ld, device_bytes, block, stream);
}

int apsp_ooc_block(int n, unsigned long long device_bytes, int elem_bytes) {
    if (n <= 0 || elem_bytes <= 0 || device_bytes == 0) return 0;
    const int npad128 = (n + TB - 1) / TB * TB;
    int K = std::min(16384, npad128);
    while (K > TB && ooc_elems(n, K) * (size_t)elem_bytes > device_bytes) K -= TB;
    return ooc_elems(n, K) * (size_t)elem_bytes <= device_bytes ? K : 0;
}

}  // extern "C"
