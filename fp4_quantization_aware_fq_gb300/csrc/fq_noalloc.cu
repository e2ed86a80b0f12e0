// fq_noalloc.cu -- fq_osci_update_noalloc: the OsciReset optimizer step
// without a caller-provided workspace.
//
// fq_osci_update keeps one float per tensor (the tensor amax of the freshly
// updated master weights) in a workspace the caller allocates.  Some callers
// cannot allocate device memory at the point where they run the step: code
// that lives inside a framework whose caching allocator owns all device
// memory and offers it no handle, a plugin that is handed only its input and
// output tensors, or a process that forbids cudaMalloc/cudaFree after start-up
// (allocation there can synchronise the device or fail under a memory cap).
// For them this file holds that scratch in a file-scope device array of
// FQ_NOALLOC_MAX_TENSORS floats, which every GPU that loads the library keeps
// until the process exits.
#include <mutex>

#include "fq.h"
#include "fq_internal.h"

namespace {

constexpr int kMaxTensors = FQ_NOALLOC_MAX_TENSORS;
static_assert(kMaxTensors <= fqk::kOsciMaxTensors, "one grouped launch per call");

// The scratch itself.  Host code must not use this name as an address: on the
// host it is only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_osci_amax[kMaxTensors];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
float *g_scratch[kMaxDevices];  // device address of g_osci_amax per device; NULL: not set up

// Set-up, once per device, with that device current.
fq_status scratch_on_current_device(float **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_osci_amax) != cudaSuccess || !p)
            return FQ_ERR_CUDA;
        g_scratch[dev] = static_cast<float *>(p);
    }
    *out = g_scratch[dev];
    return FQ_OK;
}

}  // namespace

extern "C" FQ_API fq_status fq_osci_update_noalloc(
    const fq_config *cfg, int32_t ntensors, const int64_t *rows, const int64_t *cols,
    float *const *master, const float *const *delta, float *const *dist_q, float *const *dist_m,
    const fq_qtensor *prev, const fq_qtensor *next, void *const *xhat, int32_t xhat_dtype,
    uint8_t *const *mask, void *stream)
{
    if (ntensors > kMaxTensors)
        return FQ_ERR_WORKSPACE;
    if (ntensors <= 0)
        return ntensors == 0 ? FQ_OK : FQ_ERR_INVALID_ARG;
    float *scratch = nullptr;
    fq_status st = scratch_on_current_device(&scratch);
    if (st != FQ_OK)
        return st;
    // fq_osci_update clears the amax slots on the stream before its first
    // pass, so whatever an earlier call left in the array does not leak in.
    return fq_osci_update(cfg, ntensors, rows, cols, master, delta, dist_q, dist_m, prev, next,
                          xhat, xhat_dtype, mask, scratch, sizeof(g_osci_amax), stream);
}
