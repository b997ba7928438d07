// ce_noalloc.cu -- ce_fwd_bwd_noalloc: the forward + backward call for
// callers that cannot allocate device memory.
//
// Some hosts give their extensions no allocator: an inference or training
// runtime that reserves all device memory up front for its own pool, or a
// plugin interface whose entry points receive only the input and output
// buffers. Such callers cannot provide the workspace ce_fwd_bwd needs. This
// entry point takes its scratch from a fixed array in the library's own
// device memory instead (the array exists on every GPU that loads the
// library, until the process exits), and allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "ce.h"
#include "ce_device.cuh"
#include "ce_host.h"

namespace {

// Scratch for up to CE_NOALLOC_MAX_ROWS rows: control block, per-row loss,
// per-row statistics (the same layout as a caller-provided workspace).
constexpr size_t kNoallocBytes =
    ce::kWsCtlBytes + ((static_cast<size_t>(CE_NOALLOC_MAX_ROWS) * sizeof(float) + 255) & ~static_cast<size_t>(255)) +
    static_cast<size_t>(CE_NOALLOC_MAX_ROWS) * 4 * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

// The array's device address, looked up once per CUDA context. A context's
// id is never reused within a process, so after cudaDeviceReset (a new
// primary context, the module loaded again at a possibly different address)
// the next call looks the address up again instead of using the old one.
constexpr int kMaxDevices = 64;
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the current device's context. In
// host code the array's name is only a host-side stand-in, so the address is
// asked from the runtime (cudaGetSymbolAddress), with that device current.
ce_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    unsigned long long id = ce::current_context_id();
    if (id == 0 || g_scratch[dev].ctx_id != id || g_scratch[dev].ptr == nullptr) {
        // also makes the device's primary context current on this thread
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CE_ERR_CUDA;
        id = ce::current_context_id();
        if (id == 0) return CE_ERR_CUDA;
        g_scratch[dev].ctx_id = id;
        g_scratch[dev].ptr = p;
    }
    *out = g_scratch[dev].ptr;
    return CE_OK;
}

}  // namespace

extern "C" {

ce_status ce_fwd_bwd_noalloc(const ce_params *p, void *logits_inout, const void *target, float *loss,
                             const float *grad_output, void *stream) {
    if (!p) return CE_ERR_INVALID_ARG;
    // The batch normalisers must come from this call's own kernel: a caller
    // has no way to run ce_prepare on the library's scratch.
    if (p->variant & CE_VARIANT_PREPARED) return CE_ERR_INVALID_ARG;
    if (p->n_rows > CE_NOALLOC_MAX_ROWS) return CE_ERR_WORKSPACE;  // more rows than the fixed scratch holds
    if (p->n_rows < 0) return CE_ERR_INVALID_ARG;
    size_t need = 0;
    ce_status st = ce_workspace_size(p, &need);
    if (st != CE_OK) return st;
    if (need > kNoallocBytes) return CE_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != CE_OK) return st;
    return ce_fwd_bwd(p, logits_inout, target, loss, grad_output, scratch, kNoallocBytes, stream);
}

}  // extern "C"
