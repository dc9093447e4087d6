// splitk_noalloc.cu -- split-K GEMM for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: a plugin or callback running
// inside a host program that owns all GPU memory through its own pool, a
// latency-critical loop where the synchronisation and unpredictable cost of
// cudaMalloc/cudaFree are not acceptable, or a process whose memory budget is fixed
// up front.  For them, fgemm_sgemm_splitk_noalloc runs the split-K GEMM with its
// partial products in a fixed array that lives in every GPU's global memory from the
// moment the library is loaded until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "fgemm.h"

namespace {

// The shared scratch array (FGEMM_NOALLOC_SCRATCH_BYTES on every device that loads
// the library).  Host code must not use this name as an address: it only stands for
// the symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[FGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (with that device current) and cached.  nullptr if the lookup fails.
float *scratch_on_current_device()
{
    static std::atomic<float *> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    float *p = cache[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        p = static_cast<float *>(addr);
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" fgemm_status fgemm_sgemm_splitk_noalloc(fgemm_op transa, fgemm_op transb, int M, int N,
                                                   int K, float alpha, const float *A, int lda,
                                                   const float *B, int ldb, float beta, float *C,
                                                   int ldc, const float *bias, int apply_relu,
                                                   int splits, cudaStream_t stream)
{
    // Reject, before anything else, a problem whose partial products do not fit.
    const size_t need = fgemm_splitk_workspace_size(M, N, K, splits);
    if (need > (size_t)FGEMM_NOALLOC_SCRATCH_BYTES) return FGEMM_ERR_NOT_SUPPORTED;
    float *scratch = scratch_on_current_device();
    if (scratch == nullptr) return FGEMM_ERR_LAUNCH;
    // Every partial product is written before it is read, so nothing has to start
    // at zero.  No allocation happens below: the split-K path only launches kernels.
    return fgemm_sgemm_splitk(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                              apply_relu, splits, scratch, (size_t)FGEMM_NOALLOC_SCRATCH_BYTES,
                              stream);
}
