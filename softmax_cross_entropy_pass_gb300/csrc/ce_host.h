// ce_host.h -- host-side helpers shared by the launch code: the id of the
// current CUDA context, used to key per-context caches (a function's shared
// memory attribute, a symbol's device address). A context id is never reused
// within a process, so a cache keyed on it is not fooled by a device reset
// that replaces the primary context.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace ce {

// Id of the context current on this thread; 0 if there is none (the runtime
// makes the device's primary context current at its first call that needs
// one) or the CUDA driver entry points are unavailable.
inline unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *a = nullptr, *b = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace ce
