// C-ABI of libapsp: argument checks, the per-device workspace, the round
// driver and the precondition validator.
//
// Round driver (blocked Floyd-Warshall thesis page, 1library.co excerpt,
// section 4.6): the primary tile walks down the diagonal, one round per
// tile, and each round runs phase 1, phase 2 and phase 3 as separate kernels
// in stream order.  The matrix never leaves device memory (section 4.6.1:
// the whole graph lives in global memory).
#include <cuda.h>
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled (fetched through the runtime)
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "../../include/apsp.h"
#include "../../include/apsp_debug.h"
#include "fw_launch.h"

namespace {

constexpr int kTB = APSP_TILE;
constexpr size_t kErrBytes = 256;  // device error word at the start of the workspace
thread_local int g_last_cuda_error = 0;

apsp_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return APSP_ECUDA;
}

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    bool init_i32 = false, init_f32 = false;
    void* ws = nullptr;          // workspace: panels + primary tiles
    size_t ws_bytes = 0;
    void* stage = nullptr;       // staging matrix for the host-buffer entry points
    size_t stage_bytes = 0;
    void* stage2 = nullptr;      // second staging matrix (batched host solves)
    size_t stage2_bytes = 0;
    cudaStream_t copy = nullptr; // copy stream of the batched host solves
    cudaEvent_t bev[5] = {};     // their events: start, uploaded[2], solved[2]
    cudaEvent_t done = nullptr;  // end of the last solve that used ws
    int small_i32 = -1, small_f32 = -1;  // cluster size of the small-matrix path (-1: not asked yet, 0: none)
};

std::mutex g_mu;
std::vector<DeviceState> g_dev;
int g_inject = 0;  // test hook, consumed by the next persistent phase-3 launch
int g_fail_allocs = 0;  // test hook: the next this many workspace allocations fail
unsigned long long g_inject_timeout_ns = 0;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

// Phase timing (profiling hook).
struct Timing {
    bool enabled = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending[3];
    std::vector<cudaEvent_t> pool;
    double ms[3] = {0, 0, 0};
    long long launches[3] = {0, 0, 0};
};
Timing g_timing;

cudaEvent_t timing_event() {
    if (!g_timing.pool.empty()) {
        cudaEvent_t e = g_timing.pool.back();
        g_timing.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

apsp_status_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceState& st = g_dev[dev];
    if (!st.probed) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        st.supported = (major == 10 && minor == 3);
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        st.probed = true;
    }
    if (!st.supported) return APSP_EUNSUPPORTED;
    if (!st.done) {
        e = cudaEventCreateWithFlags(&st.done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *out = &st;
    return APSP_OK;
}

// Grow-only device buffer; waits for the last solve before freeing.  Sets
// *fresh when it allocated.
apsp_status_t ensure_buffer(DeviceState& st, void** buf, size_t* have, size_t need,
                            bool* fresh = nullptr) {
    if (fresh) *fresh = false;
    if (*have >= need) return APSP_OK;
    if (*buf) {
        cudaError_t e = cudaEventSynchronize(st.done);
        if (e != cudaSuccess) return cuda_fail(e);
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    cudaError_t e;
    if (g_fail_allocs > 0) {  // test hook: this allocation fails as if the device were full
        --g_fail_allocs;
        e = cudaErrorMemoryAllocation;
    } else {
        e = cudaMalloc(buf, need);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free allocation error
        *buf = nullptr;
        g_last_cuda_error = (int)e;
        return APSP_ENOMEM;
    }
    *have = need;
    if (fresh) *fresh = true;
    return APSP_OK;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// Row-major 2-D tensor map: `rows` x `cols` elements of 4 bytes, row pitch
// `pitch_bytes` (a multiple of 16), box `box_rows` x `box_cols`, no swizzle.
// Out-of-bounds parts of a box read as zero; the kernels never store them.
bool encode_2d(CUtensorMap* m, bool is_float, void* base, unsigned long long cols,
               unsigned long long rows, unsigned long long pitch_bytes, unsigned box_cols,
               unsigned box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, is_float ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base,
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// APSP_PHASE3=cpasync forces the one-CTA-per-tile cp.async phase 3 even when
// the persistent TMA kernel could run (for comparison and testing).
bool persistent_phase3_allowed() {
    const char* v = std::getenv("APSP_PHASE3");
    return !(v && std::strcmp(v, "cpasync") == 0);
}

// Items per phase-3 tile along k in the fused schedule: the size-based
// choice (fused_split), unless APSP_FUSED_SPLIT=1|2|4 forces one.
int fused_split_for(int nb, int sms) {
    const char* v = std::getenv("APSP_FUSED_SPLIT");
    if (v && (std::strcmp(v, "1") == 0 || std::strcmp(v, "2") == 0 || std::strcmp(v, "4") == 0))
        return v[0] - '0';
    return apsp::fused_split(nb, sms);
}

// APSP_FUSED_OVERLAP=0 launches each round only after the previous one has
// ended (no programmatic dependent launch), for comparison and testing.
bool fused_overlap_allowed() {
    const char* v = std::getenv("APSP_FUSED_OVERLAP");
    return !(v && std::strcmp(v, "0") == 0);
}

// APSP_P3_COLS=4|8 picks the persistent phase 3's accumulator columns per
// thread (512 or 256 consumer threads); the default is kDefaultP3Cols.
constexpr int kDefaultP3Cols = 8;
int phase3_cols() {
    const char* v = std::getenv("APSP_P3_COLS");
    if (v && std::strcmp(v, "4") == 0) return 4;
    if (v && std::strcmp(v, "8") == 0) return 8;
    return kDefaultP3Cols;
}

// APSP_P3_STAGES=4|5 picks the persistent phase 3's slab ring depth.
constexpr int kDefaultP3Stages = 4;
int phase3_stages() {
    const char* v = std::getenv("APSP_P3_STAGES");
    if (v && std::strcmp(v, "5") == 0) return 5;
    if (v && std::strcmp(v, "4") == 0) return 4;
    return kDefaultP3Stages;
}

// APSP_FUSED=0 selects the three-kernel schedule (phase 1, phase 2 and phase 3
// as separate launches per round) instead of the round-fused one.
bool fused_allowed() {
    const char* v = std::getenv("APSP_FUSED");
    return !(v && std::strcmp(v, "0") == 0);
}

// APSP_SMALL=0 sends small matrices through the round schedules too (for
// comparison and testing) instead of the one-cluster kernel.
bool small_allowed() {
    const char* v = std::getenv("APSP_SMALL");
    return !(v && std::strcmp(v, "0") == 0);
}

bool args_ok(const void* p, int n, int ld) {
    if (n < 0 || n > APSP_MAX_N || ld < n) return false;
    if (n > 0 && p == nullptr) return false;
    return true;
}

template <typename T>
cudaError_t init_kernels(DeviceState& st);
template <>
cudaError_t init_kernels<int32_t>(DeviceState& st) {
    if (st.init_i32) return cudaSuccess;
    cudaError_t e = apsp::kernels_init<int32_t>();
    st.init_i32 = (e == cudaSuccess);
    return e;
}
template <>
cudaError_t init_kernels<float>(DeviceState& st) {
    if (st.init_f32) return cudaSuccess;
    cudaError_t e = apsp::kernels_init<float>();
    st.init_f32 = (e == cudaSuccess);
    return e;
}

template <typename T>
cudaError_t launch_phase(int phase, const apsp::RoundArgs& a, int r, cudaStream_t s) {
    switch (phase) {
        case 0: return apsp::launch_phase1<T>(a, r, s);
        case 1: return apsp::launch_phase2<T>(a, r, s);
        default: return apsp::launch_phase3<T>(a, r, s);
    }
}

// Small matrices: the whole solve as one launch of a thread-block cluster
// (fw_cluster.cuh).  It needs no workspace.  Returns false (and enqueues
// nothing) when the path does not apply.
template <typename T>
bool solve_small(T* d, int n, int ld, cudaStream_t s, DeviceState& st, apsp_status_t* rc) {
    if (n > apsp::kSmallMaxN || !small_allowed()) return false;
    int& cluster = std::is_same<T, float>::value ? st.small_f32 : st.small_i32;
    if (cluster < 0) cluster = apsp::small_cluster_size<T>();
    if (cluster <= 0) return false;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) {
        *rc = cuda_fail(e);
        return true;
    }
    const bool timed = g_timing.enabled && cap == cudaStreamCaptureStatusNone;
    cudaEvent_t e0 = timed ? timing_event() : nullptr, e1 = timed ? timing_event() : nullptr;
    if (e0) cudaEventRecord(e0, s);
    const int vec = ((reinterpret_cast<uintptr_t>(d) & 15u) == 0 && (ld % 4) == 0) ? 1 : 0;
    e = apsp::launch_small<T>(d, ld, n, vec, cluster, s);
    if (e0 && e1) {
        cudaEventRecord(e1, s);
        g_timing.pending[2].emplace_back(e0, e1);
    }
    *rc = e == cudaSuccess ? APSP_OK : cuda_fail(e);
    return true;
}

// Enqueue a full solve.  Caller holds g_mu.
template <typename T>
apsp_status_t solve_locked(T* d, int n, int ld, cudaStream_t s, DeviceState& st) {
    cudaError_t e = init_kernels<T>(st);
    if (e != cudaSuccess) return cuda_fail(e);
    apsp_status_t small_rc = APSP_OK;
    if (solve_small<T>(d, n, ld, s, st, &small_rc)) return small_rc;
    const int nb = (n + kTB - 1) / kTB;
    const int npad = nb * kTB;
    bool fresh = false;
    apsp_status_t rc = ensure_buffer(st, &st.ws, &st.ws_bytes, apsp::workspace_bytes(n), &fresh);
    if (rc != APSP_OK) return rc;
    if (fresh) {
        e = cudaMemsetAsync(st.ws, 0, kErrBytes, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }

    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e);
    const bool capturing = (cap != cudaStreamCaptureStatusNone);
    if (!capturing) {
        e = cudaStreamWaitEvent(s, st.done, 0);
        if (e != cudaSuccess) return cuda_fail(e);
    }

    // Workspace layout: [error word, 256 B][rowp][colpT][prim][primT].
    char* w = static_cast<char*>(st.ws);
    apsp::RoundArgs a;
    a.d = d;
    a.ld = ld;
    a.n = n;
    a.nb = nb;
    a.vec = ((reinterpret_cast<uintptr_t>(d) & 15u) == 0 && (ld % 4) == 0) ? 1 : 0;
    a.npad = npad;
    a.err = reinterpret_cast<int*>(w);
    a.rowp = w + kErrBytes;
    a.colpT = w + kErrBytes + (size_t)kTB * npad * sizeof(T);
    a.prim = w + kErrBytes + 2 * (size_t)kTB * npad * sizeof(T);
    a.primT = w + kErrBytes + 2 * (size_t)kTB * npad * sizeof(T) + (size_t)kTB * kTB * sizeof(T);
    a.sms = st.sms;
    a.tma = 0;
    a.inject = 0;
    a.timeout_ns = kDefaultTimeoutNs;
    a.p3_cols = phase3_cols();
    a.p3_stages = phase3_stages();
    const bool is_float = std::is_same<T, float>::value;
    if (a.vec && nb > 1 && persistent_phase3_allowed()) {
        const int ks = apsp::phase3_slab_rows();
        a.tma = encode_2d(&a.tm_c, is_float, d, n, n, (unsigned long long)ld * sizeof(T), kTB, kTB) &&
                encode_2d(&a.tm_a, is_float, a.colpT, npad, kTB, (unsigned long long)npad * sizeof(T),
                          kTB, ks) &&
                encode_2d(&a.tm_b, is_float, a.rowp, npad, kTB, (unsigned long long)npad * sizeof(T),
                          kTB, ks);
    }

    const bool timed = g_timing.enabled && !capturing;
    auto timed_launch = [&](int slot, auto&& launch) -> cudaError_t {
        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (timed) {
            e0 = timing_event();
            e1 = timing_event();
            if (e0) cudaEventRecord(e0, s);
        }
        cudaError_t le = launch();
        if (timed && e0 && e1) {
            cudaEventRecord(e1, s);
            g_timing.pending[slot].emplace_back(e0, e1);
        }
        return le;
    };

    if (a.tma && fused_allowed()) {
        // Round-fused schedule: a prologue launch (phase 1 and 2 of round 0),
        // then one launch per round (phase 3 of r with phase 1 and 2 of r+1).
        apsp::FusedArgs f;
        f.d = d;
        f.ld = ld;
        f.n = n;
        f.nb = nb;
        f.npad = npad;
        f.sms = st.sms;
        f.timeout_ns = kDefaultTimeoutNs;
        f.inject = 0;
        char* x = w + kErrBytes + (2 * (size_t)kTB * npad + 2 * (size_t)kTB * kTB) * sizeof(T);
        f.ptrs.rowp[0] = a.rowp;
        f.ptrs.colpT[0] = a.colpT;
        f.ptrs.rowp[1] = x;
        f.ptrs.colpT[1] = x + (size_t)kTB * npad * sizeof(T);
        f.ptrs.prim = a.prim;
        f.ptrs.primT = a.primT;
        int* flags = reinterpret_cast<int*>(x + 2 * (size_t)kTB * npad * sizeof(T));
        f.ptrs.flag_diag = flags;
        f.ptrs.flag_p1 = flags + 1;
        f.ptrs.flag_row = flags + 2;
        f.ptrs.flag_col = flags + 2 + nb;
        f.ptrs.counters = flags + 2 + 2 * nb;
        f.ptrs.parts = flags + 3 + 3 * nb;
        f.split = fused_split_for(nb, st.sms);
        f.overlap = fused_overlap_allowed() ? 1 : 0;
        f.ptrs.err = a.err;
        const int ks = apsp::phase3_slab_rows();
        const unsigned long long pitch = (unsigned long long)npad * sizeof(T);
        bool ok = true;
        f.maps.c = a.tm_c;
        // Phase-3 tiles merge into D by a signed 32-bit min-reduction.  For
        // fp32 that is the order of the values too: within the contract
        // every entry is +0, positive or +inf (a -0.0 input acts as zero).
        if (is_float)
            ok = encode_2d(&f.maps.cmin, false, d, n, n, (unsigned long long)ld * sizeof(T), kTB, kTB);
        else
            f.maps.cmin = a.tm_c;
        // The panels in the layout apsp::kPanelPack<T> names: pk = 2 views a
        // TB x npad panel as TB / 2 rows of 2 npad, k-pair interleaved.
        const int pk = apsp::kPanelPack<T>;
        for (int b = 0; b < 2; ++b) {
            ok = ok && encode_2d(&f.maps.rowp[b], is_float, f.ptrs.rowp[b], (unsigned long long)npad * pk,
                                 kTB / pk, pitch * pk, kTB * pk, ks / pk);
            ok = ok && encode_2d(&f.maps.colpT[b], is_float, f.ptrs.colpT[b], (unsigned long long)npad * pk,
                                 kTB / pk, pitch * pk, kTB * pk, ks / pk);
        }
        ok = ok && encode_2d(&f.maps.prim, is_float, a.prim, kTB, kTB, kTB * sizeof(T), kTB, ks);
        ok = ok && encode_2d(&f.maps.primT, is_float, a.primT, kTB, kTB, kTB * sizeof(T), kTB, ks);
        if (ok) {
            // flags start at -1 (no round stamped yet), item counters and
            // critical-part counts at 0
            e = cudaMemsetAsync(flags, 0xFF, (size_t)(2 + 2 * nb) * sizeof(int), s);
            if (e == cudaSuccess)
                e = cudaMemsetAsync(f.ptrs.counters, 0, (size_t)(nb + 1 + 2 * nb + 1) * sizeof(int), s);
            if (e != cudaSuccess) return cuda_fail(e);
            for (int r = -1; r < nb; ++r) {
                const bool inject_here = (r == 0 && g_inject);
                if (inject_here) {
                    f.inject = 1;
                    f.timeout_ns = g_inject_timeout_ns;
                    g_inject = 0;
                }
                e = timed_launch(2, [&] { return apsp::launch_fused<T>(f, r, s); });
                if (inject_here) {
                    f.inject = 0;
                    f.timeout_ns = kDefaultTimeoutNs;
                }
                if (e != cudaSuccess) return cuda_fail(e);
            }
            if (!capturing) {
                e = cudaEventRecord(st.done, s);
                if (e != cudaSuccess) return cuda_fail(e);
            }
            return APSP_OK;
        }
    }

    for (int r = 0; r < nb; ++r) {
        for (int phase = 0; phase < 3; ++phase) {
            if (phase > 0 && nb < 2) break;
            e = timed_launch(phase, [&] {
                const bool inject_here = (phase == 2 && g_inject && a.tma);
                if (inject_here) {
                    a.inject = 1;
                    a.timeout_ns = g_inject_timeout_ns;
                    g_inject = 0;
                }
                cudaError_t le = launch_phase<T>(phase, a, r, s);
                if (inject_here) {
                    a.inject = 0;
                    a.timeout_ns = kDefaultTimeoutNs;
                }
                return le;
            });
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    if (!capturing) {
        e = cudaEventRecord(st.done, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return APSP_OK;
}

template <typename T>
apsp_status_t solve_device(T* d, int n, int ld, cudaStream_t s) {
    if (!args_ok(d, n, ld)) return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    apsp_status_t rc = device_state(&st);
    if (rc != APSP_OK) return rc;
    return solve_locked<T>(d, n, ld, s, *st);
}

template <typename T>
apsp_status_t solve_host(T* h, int n, int ld, cudaStream_t s) {
    if (!args_ok(h, n, ld)) return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    apsp_status_t rc = device_state(&st);
    if (rc != APSP_OK) return rc;
    const int ldd = (n + 3) & ~3;  // vector-friendly device pitch
    rc = ensure_buffer(*st, &st->stage, &st->stage_bytes, (size_t)n * ldd * sizeof(T));
    if (rc != APSP_OK) return rc;
    T* dd = static_cast<T*>(st->stage);
    cudaError_t e;
    if (ld == ldd)
        e = cudaMemcpyAsync(dd, h, (size_t)n * ld * sizeof(T), cudaMemcpyHostToDevice, s);
    else
        e = cudaMemcpy2DAsync(dd, (size_t)ldd * sizeof(T), h, (size_t)ld * sizeof(T),
                              (size_t)n * sizeof(T), n, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    rc = solve_locked<T>(dd, n, ldd, s, *st);
    if (rc != APSP_OK) return rc;
    if (ld == ldd)
        e = cudaMemcpyAsync(h, dd, (size_t)n * ld * sizeof(T), cudaMemcpyDeviceToHost, s);
    else
        e = cudaMemcpy2DAsync(h, (size_t)ld * sizeof(T), dd, (size_t)ldd * sizeof(T),
                              (size_t)n * sizeof(T), n, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return APSP_OK;
}

// Batched host solves: matrix b is uploaded into staging buffer b % 2 on a
// copy stream, solved on s, and downloaded on the copy stream, so the copies
// of matrices b - 1 and b + 1 overlap the solve of matrix b.  On the copy
// stream, the upload of matrix b + 2 follows the download of matrix b, which
// used the same buffer; the solve of matrix b waits for its upload.
template <typename T>
apsp_status_t solve_host_batch(const T* const* in, T* const* out, int count, int n, int ld, cudaStream_t s) {
    if (count < 0 || n < 0 || n > APSP_MAX_N || ld < n) return APSP_EINVAL;
    if (count == 0 || n == 0) return APSP_OK;
    if (in == nullptr || out == nullptr) return APSP_EINVAL;
    for (int b = 0; b < count; ++b)
        if (in[b] == nullptr || out[b] == nullptr) return APSP_EINVAL;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    apsp_status_t rc = device_state(&st);
    if (rc != APSP_OK) return rc;
    const int ldd = (n + 3) & ~3;  // vector-friendly device pitch
    const size_t bytes = (size_t)n * ldd * sizeof(T);
    rc = ensure_buffer(*st, &st->stage, &st->stage_bytes, bytes);
    if (rc == APSP_OK && count > 1) rc = ensure_buffer(*st, &st->stage2, &st->stage2_bytes, bytes);
    if (rc != APSP_OK) return rc;
    cudaError_t e = cudaSuccess;
    if (!st->copy) e = cudaStreamCreateWithFlags(&st->copy, cudaStreamNonBlocking);
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
        if (!st->bev[i]) e = cudaEventCreateWithFlags(&st->bev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e);
    T* buf[2] = {static_cast<T*>(st->stage), static_cast<T*>(st->stage2)};
    cudaStream_t c = st->copy;
    auto copy = [&](T* dst, size_t dpitch, const T* src, size_t spitch, cudaMemcpyKind kind) {
        if (dpitch == spitch) return cudaMemcpyAsync(dst, src, (size_t)n * dpitch * sizeof(T), kind, c);
        return cudaMemcpy2DAsync(dst, dpitch * sizeof(T), src, spitch * sizeof(T), (size_t)n * sizeof(T), n,
                                 kind, c);
    };
    auto upload = [&](int b) {
        cudaError_t x = copy(buf[b & 1], ldd, in[b], ld, cudaMemcpyHostToDevice);
        if (x == cudaSuccess) x = cudaEventRecord(st->bev[1 + (b & 1)], c);
        return x;
    };
    // the staging buffers may still be in use by earlier work on s
    e = cudaEventRecord(st->bev[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c, st->bev[0], 0);
    if (e == cudaSuccess) e = upload(0);
    if (e == cudaSuccess && count > 1) e = upload(1);
    for (int b = 0; b < count && e == cudaSuccess; ++b) {
        const int k = b & 1;
        e = cudaStreamWaitEvent(s, st->bev[1 + k], 0);
        if (e != cudaSuccess) break;
        rc = solve_locked<T>(buf[k], n, ldd, s, *st);
        if (rc != APSP_OK) break;
        e = cudaEventRecord(st->bev[3 + k], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c, st->bev[3 + k], 0);
        if (e == cudaSuccess) e = copy(out[b], ld, buf[k], ldd, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess && b + 2 < count) e = upload(b + 2);
    }
    // wait for everything enqueued, even after an error
    const cudaError_t e1 = cudaStreamSynchronize(c);
    const cudaError_t e2 = cudaStreamSynchronize(s);
    if (rc != APSP_OK) return rc;
    if (e == cudaSuccess) e = e1 != cudaSuccess ? e1 : e2;
    if (e != cudaSuccess) return cuda_fail(e);
    return APSP_OK;
}

// ------------------------------------------------------------- validator

template <typename T>
__device__ __forceinline__ int entry_flags(T v, bool diag);
template <>
__device__ __forceinline__ int entry_flags<int32_t>(int32_t v, bool diag) {
    return ((diag && v != 0) ? 1 : 0) | (v < 0 ? 2 : 0);
}
template <>
__device__ __forceinline__ int entry_flags<float>(float v, bool diag) {
    return ((diag && v != 0.0f) ? 1 : 0) | (v < 0.0f ? 2 : 0) | (isnan(v) ? 4 : 0);
}

template <typename T>
__global__ void validate_kernel(const T* __restrict__ d, long long ld, int n, int* flags) {
    const long long total = (long long)n * n;
    int f = 0;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / n, j = idx - i * n;
        f |= entry_flags<T>(d[i * ld + j], i == j);
    }
    f = __reduce_or_sync(0xffffffffu, f);
    if (f && (threadIdx.x & 31) == 0) atomicOr(flags, f);
}

template <typename T>
apsp_status_t validate(const T* d, int n, int ld, cudaStream_t s, int* flags) {
    if (!args_ok(d, n, ld) || flags == nullptr) return APSP_EINVAL;
    if (n == 0) return APSP_OK;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* st = nullptr;
        apsp_status_t rc = device_state(&st);
        if (rc != APSP_OK) return rc;
    }
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)n * n;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    validate_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(d, ld, n, flags);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return APSP_OK;
}

}  // namespace

namespace apsp {
// Lets the sparse entry points report through apsp_last_cuda_error().
void set_last_cuda_error(int e) { g_last_cuda_error = e; }

size_t workspace_bytes(int n) {
    const size_t nb = (size_t)(n + kTB - 1) / kTB;
    const size_t npad = nb * kTB;
    const size_t base = kErrBytes + (2 * (size_t)kTB * npad + 2 * (size_t)kTB * kTB) * 4;
    const size_t panels2 = 2 * (size_t)kTB * npad * 4;       // second row/column panel buffers
    const size_t flags = ((5 * nb + 4) * 4 + 255) / 256 * 256;  // flags, item counters, part counts
    return base + panels2 + flags;
}
}  // namespace apsp

extern "C" {

apsp_status_t apsp_solve(int32_t* dist, int n, int ld, apsp_stream_t stream) {
    return solve_device<int32_t>(dist, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_i32(int32_t* dist, int n, int ld, apsp_stream_t stream) {
    return solve_device<int32_t>(dist, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_f32(float* dist, int n, int ld, apsp_stream_t stream) {
    return solve_device<float>(dist, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_host_i32(int32_t* host, int n, int ld, apsp_stream_t stream) {
    return solve_host<int32_t>(host, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_host_f32(float* host, int n, int ld, apsp_stream_t stream) {
    return solve_host<float>(host, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_host_batch_i32(const int32_t* const* in, int32_t* const* out, int count, int n,
                                        int ld, apsp_stream_t stream) {
    return solve_host_batch<int32_t>(in, out, count, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_solve_host_batch_f32(const float* const* in, float* const* out, int count, int n, int ld,
                                        apsp_stream_t stream) {
    return solve_host_batch<float>(in, out, count, n, ld, (cudaStream_t)stream);
}

apsp_status_t apsp_validate_i32(const int32_t* dist, int n, int ld, apsp_stream_t stream,
                                int* flags_dev) {
    return validate<int32_t>(dist, n, ld, (cudaStream_t)stream, flags_dev);
}

apsp_status_t apsp_validate_f32(const float* dist, int n, int ld, apsp_stream_t stream,
                                int* flags_dev) {
    return validate<float>(dist, n, ld, (cudaStream_t)stream, flags_dev);
}

apsp_status_t apsp_stream_check(apsp_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    // Device error word of the current device's workspace: a bounded wait
    // that ran out recorded itself there.  Read it, then clear it.
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= (int)g_dev.size() || !g_dev[dev].ws) return APSP_OK;
    DeviceState& st = g_dev[dev];
    int* errp = static_cast<int*>(st.ws);
    int flags = 0;
    e = cudaMemcpy(&flags, errp, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (flags != 0) {
        cudaMemset(errp, 0, sizeof(int));
        return APSP_ETIMEOUT;
    }
    return APSP_OK;
}

int apsp_last_cuda_error(void) { return g_last_cuda_error; }

const char* apsp_status_string(apsp_status_t status) {
    switch (status) {
        case APSP_OK: return "APSP_OK";
        case APSP_EINVAL: return "APSP_EINVAL: invalid argument";
        case APSP_ECUDA: return "APSP_ECUDA: CUDA error";
        case APSP_ETIMEOUT: return "APSP_ETIMEOUT: device-side wait timed out";
        case APSP_EUNSUPPORTED: return "APSP_EUNSUPPORTED: device is not sm_103";
        case APSP_ENOMEM: return "APSP_ENOMEM: device allocation failed";
        case APSP_ENEGCYCLE: return "APSP_ENEGCYCLE: negative cycle";
    }
    return "unknown apsp status";
}

int apsp_version(void) { return 100; }  // 0.1.0

apsp_status_t apsp_release(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    apsp_status_t rc = APSP_OK;
    for (size_t dev = 0; dev < g_dev.size(); ++dev) {
        DeviceState& st = g_dev[dev];
        if (!st.ws && !st.stage && !st.stage2 && !st.copy && !st.done) continue;
        if (cudaSetDevice((int)dev) != cudaSuccess) { rc = APSP_ECUDA; continue; }
        if (st.done) cudaEventSynchronize(st.done);
        if (st.copy) cudaStreamSynchronize(st.copy);
        if (st.ws) cudaFree(st.ws);
        if (st.stage) cudaFree(st.stage);
        if (st.stage2) cudaFree(st.stage2);
        if (st.done) cudaEventDestroy(st.done);
        for (cudaEvent_t& ev : st.bev) {
            if (ev) cudaEventDestroy(ev);
            ev = nullptr;
        }
        if (st.copy) cudaStreamDestroy(st.copy);
        st.ws = st.stage = st.stage2 = nullptr;
        st.ws_bytes = st.stage_bytes = st.stage2_bytes = 0;
        st.copy = nullptr;
        st.done = nullptr;
    }
    cudaSetDevice(cur);
    return rc;
}

int apsp_debug_small_cluster_size(int is_float) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    if (device_state(&st) != APSP_OK) return -1;
    int& c = is_float ? st->small_f32 : st->small_i32;
    if (c < 0) c = is_float ? apsp::small_cluster_size<float>() : apsp::small_cluster_size<int32_t>();
    return c;
}

apsp_status_t apsp_debug_fail_next_allocations(int count) {
    if (count < 0 || count > 1000) return APSP_EINVAL;
    std::lock_guard<std::mutex> lock(g_mu);
    g_fail_allocs = count;
    return APSP_OK;
}

apsp_status_t apsp_debug_inject_phase3_timeout(unsigned long long timeout_ns) {
    if (timeout_ns == 0 || timeout_ns > kDefaultTimeoutNs) return APSP_EINVAL;
    std::lock_guard<std::mutex> lock(g_mu);
    g_inject = 1;
    g_inject_timeout_ns = timeout_ns;
    return APSP_OK;
}

apsp_status_t apsp_phase_timing_enable(int enable) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_timing.enabled = (enable != 0);
    return APSP_OK;
}

apsp_status_t apsp_phase_timing_read(double ms_out[3], long long launches_out[3]) {
    std::lock_guard<std::mutex> lock(g_mu);
    apsp_status_t rc = APSP_OK;
    for (int p = 0; p < 3; ++p) {
        for (auto& pr : g_timing.pending[p]) {
            float ms = 0.f;
            cudaError_t e = cudaEventSynchronize(pr.second);
            if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, pr.first, pr.second);
            if (e != cudaSuccess) {
                g_last_cuda_error = (int)e;
                rc = APSP_ECUDA;
            } else {
                g_timing.ms[p] += ms;
                g_timing.launches[p] += 1;
            }
            g_timing.pool.push_back(pr.first);
            g_timing.pool.push_back(pr.second);
        }
        g_timing.pending[p].clear();
        if (ms_out) ms_out[p] = g_timing.ms[p];
        if (launches_out) launches_out[p] = g_timing.launches[p];
        g_timing.ms[p] = 0;
        g_timing.launches[p] = 0;
    }
    return rc;
}

}  // extern "C"
