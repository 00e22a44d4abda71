// apsp_solve_noalloc: the int32 solve for callers that may not allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they want shortest
// paths.  Their GPU memory may be owned by another allocator (a framework's
// caching pool, or a process capped at a fixed budget that it has already
// spent), or the call may sit in a latency-critical loop where an allocation,
// which can synchronise the whole device, is not acceptable.  The default
// entry points allocate their workspace lazily.  This one uses a fixed
// scratch array compiled into the library's device image instead.  It calls
// no cudaMalloc, cudaFree or other allocating routine, on the device or on
// the host.
//
// The scratch has the same layout as the default workspace: [error word]
// [row panel][transposed column panel][primary tile][its transpose], sized
// for n <= APSP_NOALLOC_MAX_N.  The kernels are the library's own, unchanged.
// Only the workspace pointer differs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/apsp.h"
#include "fw_launch.h"

namespace {

constexpr int kTB = APSP_TILE;
constexpr size_t kErrBytes = 256;
constexpr size_t kNpadMax = (size_t)APSP_NOALLOC_MAX_N;  // a multiple of the tile
constexpr size_t kScratchBytes =
    kErrBytes + (2 * (size_t)kTB * kNpadMax + 2 * (size_t)kTB * kTB) * sizeof(int32_t);
static_assert(kNpadMax % APSP_TILE == 0, "maximum n must be a multiple of the tile");
static_assert(kScratchBytes == APSP_NOALLOC_SCRATCH_BYTES, "header size out of date");

// The scratch itself.  Every GPU that loads the library holds it until the
// process exits.  In host code `g_scratch` only names the symbol: its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;  // fixed table: the set-up allocates nothing either
struct Slot {
    bool ready = false;
    void* scratch = nullptr;     // device address of g_scratch on this device
    int sms = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};
Slot g_slots[kMaxDevices];
std::mutex g_slot_mu;

// One-time set-up for the current device (with that device current): look
// up the scratch's device address, opt the kernels into their shared-memory
// sizes, fetch the tensor-map encoder.
apsp_status_t setup_current_device(int dev, Slot** out) {
    std::lock_guard<std::mutex> lock(g_slot_mu);
    Slot& s = g_slots[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return APSP_ECUDA;
        if (!(major == 10 && minor == 3)) return APSP_EUNSUPPORTED;
        if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return APSP_ECUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return APSP_ECUDA;
        if (apsp::kernels_init<int32_t>() != cudaSuccess) return APSP_ECUDA;
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            s.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
        s.scratch = p;
        s.ready = true;
    }
    *out = &s;
    return APSP_OK;
}

bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, void* base,
               unsigned long long cols, unsigned long long rows, unsigned long long pitch_bytes,
               unsigned box_cols, unsigned box_rows) {
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" apsp_status_t apsp_solve_noalloc(int32_t* dist, int n, int ld, apsp_stream_t stream,
                                            int* err_dev) {
    if (n < 0 || ld < n || (n > 0 && dist == nullptr)) return APSP_EINVAL;
    if (n > APSP_NOALLOC_MAX_N) return APSP_EINVAL;  // beyond the fixed scratch
    if (n == 0) return APSP_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return APSP_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return APSP_EUNSUPPORTED;
    Slot* slot = nullptr;
    apsp_status_t rc = setup_current_device(dev, &slot);
    if (rc != APSP_OK) return rc;

    cudaStream_t s = (cudaStream_t)stream;
    const int nb = (n + kTB - 1) / kTB;
    const int npad = nb * kTB;
    char* w = static_cast<char*>(slot->scratch);
    apsp::RoundArgs a;
    a.d = dist;
    a.ld = ld;
    a.n = n;
    a.nb = nb;
    a.vec = ((reinterpret_cast<uintptr_t>(dist) & 15u) == 0 && (ld % 4) == 0) ? 1 : 0;
    a.npad = npad;
    a.err = reinterpret_cast<int*>(w);
    a.rowp = w + kErrBytes;
    a.colpT = w + kErrBytes + (size_t)kTB * npad * sizeof(int32_t);
    a.prim = w + kErrBytes + 2 * (size_t)kTB * npad * sizeof(int32_t);
    a.primT = w + kErrBytes + 2 * (size_t)kTB * npad * sizeof(int32_t) +
              (size_t)kTB * kTB * sizeof(int32_t);
    a.sms = slot->sms;
    a.inject = 0;
    a.timeout_ns = 2000000000ull;
    a.p3_cols = 8;
    a.p3_stages = 4;
    a.tma = 0;
    if (a.vec && nb > 1) {
        const int ks = apsp::phase3_slab_rows();
        a.tma = encode_2d(slot->encode, &a.tm_c, dist, n, n, (unsigned long long)ld * 4, kTB, kTB) &&
                encode_2d(slot->encode, &a.tm_a, a.colpT, npad, kTB, (unsigned long long)npad * 4, kTB, ks) &&
                encode_2d(slot->encode, &a.tm_b, a.rowp, npad, kTB, (unsigned long long)npad * 4, kTB, ks);
    }

    // The scratch keeps the previous call's contents.  Only the error word
    // must start at zero: every panel entry a round reads is written earlier
    // in that round.
    cudaError_t e = cudaMemsetAsync(a.err, 0, sizeof(int), s);
    for (int r = 0; r < nb && e == cudaSuccess; ++r) {
        e = apsp::launch_phase1<int32_t>(a, r, s);
        if (e == cudaSuccess && nb > 1) e = apsp::launch_phase2<int32_t>(a, r, s);
        if (e == cudaSuccess && nb > 1) e = apsp::launch_phase3<int32_t>(a, r, s);
    }
    if (e == cudaSuccess && err_dev != nullptr)
        e = cudaMemcpyAsync(err_dev, a.err, sizeof(int), cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? APSP_OK : APSP_ECUDA;
}
