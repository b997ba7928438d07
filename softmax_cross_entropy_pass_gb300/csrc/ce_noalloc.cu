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

namespace {

// Scratch for up to CE_NOALLOC_MAX_ROWS rows: control block, per-row loss,
// per-row statistics (the same layout as a caller-provided workspace).
constexpr size_t kNoallocBytes =
    ce::kWsCtlBytes + ((static_cast<size_t>(CE_NOALLOC_MAX_ROWS) * sizeof(float) + 255) & ~static_cast<size_t>(255)) +
    static_cast<size_t>(CE_NOALLOC_MAX_ROWS) * 4 * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is asked
// from the runtime, once per device, with that device current.
ce_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CE_OK;
}

}  // namespace

extern "C" {

ce_status ce_fwd_bwd_noalloc(const ce_params *p, void *logits_inout, const void *target, float *loss,
                             const float *grad_output, void *stream) {
    if (!p) return CE_ERR_INVALID_ARG;
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
