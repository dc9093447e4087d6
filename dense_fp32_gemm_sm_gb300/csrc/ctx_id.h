// ctx_id.h -- identity of the CUDA context current on the calling host thread.
//
// Addresses of __device__ variables (cudaGetSymbolAddress) and kernel attributes
// (cudaFuncSetAttribute) belong to a context, not to a device ordinal: after
// cudaDeviceReset, or when the primary context is released and created again, the
// library's module is loaded anew, its variables may sit at other addresses and its
// kernels have lost their attributes.  Host-side caches of those are therefore keyed
// on the context's id (cuCtxGetId: unique for the life of the process, never reused),
// and a cache entry whose id differs from the current context's is looked up again.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>

namespace fgemm {

// Id of the context current on this thread; 0 when none is current (the runtime
// binds the device's primary context lazily, at the first call that needs it) or
// when the driver offers no id query.  Callers treat 0 as "do not trust a cache".
inline unsigned long long current_context_id()
{
    static std::atomic<void *> get_current{nullptr}, get_id{nullptr};
    static std::atomic<int> looked_up{0};
    if (!looked_up.load(std::memory_order_acquire)) {
        void *f = nullptr, *g = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q1) !=
                cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess)
            f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess)
            g = nullptr;
        (void)cudaGetLastError();
        get_current.store(f, std::memory_order_relaxed);
        get_id.store(g, std::memory_order_relaxed);
        looked_up.store(1, std::memory_order_release);
    }
    auto cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(get_current.load(std::memory_order_relaxed));
    auto gid = reinterpret_cast<PFN_cuCtxGetId_v12000>(get_id.load(std::memory_order_relaxed));
    if (!cur || !gid) return 0;
    CUcontext ctx = nullptr;
    if (cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (gid(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace fgemm
