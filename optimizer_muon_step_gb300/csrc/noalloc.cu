// The Muon step without any device allocation by anyone: its scratch
// memory is a file-scope device array that the library's module owns.
//
// Who needs this: callers that only hand over the parameter, gradient and
// momentum buffers and cannot obtain device memory for a workspace -- for
// example an optimizer plug-in running inside a host framework that owns
// all device memory through its own pool, where an out-of-band cudaMalloc
// would bypass the pool's accounting or fail under its hard memory cap, or
// a plain C caller with no device allocator at hand.
//
// Cost: every GPU on which this library's device code is loaded holds the
// array (MUON_STATIC_SCRATCH_BYTES) until the process exits.
#include <mutex>

#include "internal.h"

namespace {

// Device scratch shared by every call of muon_step_batched_noalloc on a
// device.  In host code `g_scratch` is only a host-side stand-in for the
// symbol, never a usable address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[MUON_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Resolves the device address of g_scratch for the current device, once per
// device, with that device current, and keeps it for the life of the
// process.  The address belongs to the device's primary context: after a
// cudaDeviceReset (or anything else that destroys that context) the kept
// address is stale, so this entry point must not be called again in that
// process.
muon_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MUON_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MUON_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MUON_OK;
}

}  // namespace

extern "C" muon_status_t muon_step_batched_noalloc(const muon_matrix_t* mats, int64_t count,
                                                   const muon_hparams_t* hp, void* stream) {
    if (count < 0 || (count > 0 && !mats)) return MUON_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i) {
        const size_t need = muon_workspace_bytes_per_matrix(mats[i].rows, mats[i].cols);
        if (need == 0) return MUON_ERR_INVALID_ARG;
        if (need > static_cast<size_t>(MUON_STATIC_SCRATCH_BYTES)) return MUON_ERR_WORKSPACE_TOO_SMALL;
    }
    if (count == 0) return muon_step_batched(mats, 0, hp, nullptr, 0, stream);
    void* scratch = nullptr;
    muon_status_t s = scratch_address(&scratch);
    if (s != MUON_OK) return s;
    return muon_step_batched(mats, count, hp, scratch, static_cast<size_t>(MUON_STATIC_SCRATCH_BYTES), stream);
}
