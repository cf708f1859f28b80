// kla_chunk_fwd_noalloc: the fixed-length chunkwise prefill for callers that
// cannot hand the library a workspace buffer.
//
// Some callers cannot allocate device memory at the point where they run the
// prefill: a host framework that owns every device byte through its own
// pool and forbids out-of-band cudaMalloc, a plugin or custom-op interface
// that receives only input and output pointers, or a latency-critical serving
// loop where cudaMalloc's implicit device-wide synchronisation is not
// acceptable.  For them the workspace of the tensor-core path lives in a
// fixed, file-scope device array of kNoallocScratchBytes that every GPU which
// loads this library holds until the process exits.
//
// Host code may not use the array's name as a device address (on the host it
// is only a stand-in symbol): the first call on each device, with that device
// current, looks the address up with cudaGetSymbolAddress and caches it.  That
// first call should therefore come before any stream capture.  The cache is
// keyed on the device's current context as well: after a device reset the
// module is loaded again, possibly at another address, and the next call
// looks the address up anew.
//
// The kernels record a bounded wait that gave up, or another device-side
// error, in the status word at the start of the array;
// kla_chunk_fwd_noalloc_status reads it (the array's address is not exposed
// otherwise).
//
// All calls share the one array, and it keeps the contents of the last call.
// The only part that must start at zero, the status word, is cleared on the
// stream by every call before any kernel reads it.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array; callers must serialise them.

#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "../../include/kla.h"
#include "kla_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)KLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct ScratchEntry {
    void *addr;
    unsigned long long ctx_id;   // context the address belongs to (0: unknown)
};

std::mutex g_setup_lock;
ScratchEntry g_scratch[kMaxDevices] = {};

// Identifier of the calling thread's current context (0 when the driver
// cannot tell; the cache then keys on the device alone).
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(fn);
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
        ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device, looked up once
// per device and context.  Returns nullptr and fills `err` on failure.
void *scratch_for_current_device(cudaError_t &err) {
    int dev = -1;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> guard(g_setup_lock);
    ScratchEntry &e = g_scratch[dev];
    if (e.addr == nullptr || e.ctx_id != current_context_id()) {
        void *ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);   // also makes the context current
        if (err != cudaSuccess) return nullptr;
        e.addr = ptr;
        e.ctx_id = current_context_id();
    }
    err = cudaSuccess;
    return e.addr;
}

}  // namespace

extern "C" int kla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                     const float *alpha, const float *eta, float eps,
                                     const float *S0, void *o, float *S_T, int B, int T, int H,
                                     int dk, int dv, int chunk, int dtype, void *stream) {
    // The size check comes first and touches no device state.
    const size_t need = kla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype);
    if (need > kNoallocScratchBytes) {
        char msg[256];
        std::snprintf(msg, sizeof msg,
                      "kla_chunk_fwd_noalloc: these sizes need %zu bytes of scratch; the "
                      "built-in array holds %zu (use kla_chunk_fwd with a workspace)",
                      need, kNoallocScratchBytes);
        kla::set_error_message(msg);
        return KLA_ERR_WORKSPACE;
    }
    cudaError_t err = cudaSuccess;
    void *scratch = scratch_for_current_device(err);
    if (scratch == nullptr) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "kla_chunk_fwd_noalloc: scratch set-up failed: %s",
                      cudaGetErrorString(err));
        kla::set_error_message(msg);
        return KLA_ERR_CUDA;
    }
    return kla_chunk_fwd(q, k, v, alpha, eta, eps, S0, o, S_T, B, T, H, dk, dv, chunk, dtype,
                         scratch, kNoallocScratchBytes, stream);
}

extern "C" int kla_chunk_fwd_noalloc_status(void *stream) {
    cudaError_t err = cudaSuccess;
    void *scratch = scratch_for_current_device(err);
    if (scratch == nullptr) {
        char msg[256];
        std::snprintf(msg, sizeof msg, "kla_chunk_fwd_noalloc_status: scratch set-up failed: %s",
                      cudaGetErrorString(err));
        kla::set_error_message(msg);
        return KLA_ERR_CUDA;
    }
    return kla_workspace_status(scratch, kNoallocScratchBytes, stream);
}
