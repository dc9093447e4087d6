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

#include <mutex>

#include "ctx_id.h"
#include "fgemm.h"
#include "fgemm_internal.h"

namespace {

// The shared scratch array (FGEMM_NOALLOC_SCRATCH_BYTES on every device that loads
// the library).  Host code must not use this name as an address: it only stands for
// the symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[FGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of g_noalloc_scratch in the context current on this thread.  It is
// looked up (cudaGetSymbolAddress, with the device current) at the first call in a
// context and cached with that context's id: after cudaDeviceReset the module is
// loaded again, the array may sit elsewhere, and the id no longer matches, so the
// address is looked up anew.  nullptr if the lookup fails.
float *scratch_in_current_context()
{
    struct Entry {
        unsigned long long ctx;
        float *addr;
    };
    static Entry cache[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return nullptr;
    }
    const unsigned long long ctx = fgemm::current_context_id();
    if (ctx != 0) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev].ctx == ctx) return cache[dev].addr;
    }
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    // The lookup made the device's primary context current if none was.
    std::lock_guard<std::mutex> lock(mu);
    cache[dev] = Entry{fgemm::current_context_id(), static_cast<float *>(addr)};
    return static_cast<float *>(addr);
}

}  // namespace

extern "C" fgemm_status fgemm_sgemm_splitk_noalloc(fgemm_op transa, fgemm_op transb, int M, int N,
                                                   int K, float alpha, const float *A, int lda,
                                                   const float *B, int ldb, float beta, float *C,
                                                   int ldc, const float *bias, int apply_relu,
                                                   int splits, cudaStream_t stream)
{
    // The argument rules of fgemm_sgemm_splitk come first; then the scratch the call
    // will use (none for splits == 1, alpha == 0 or K == 0) is checked against the array.
    size_t need = 0;
    const fgemm_status st = fgemm::splitk_plan((int)transa, (int)transb, M, N, K, alpha, A, lda, B,
                                               ldb, beta, C, ldc, splits, &need);
    if (st != FGEMM_OK) return st;
    if (need == 0)
        return fgemm_sgemm_splitk(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                                  apply_relu, splits, nullptr, 0, stream);
    if (need > (size_t)FGEMM_NOALLOC_SCRATCH_BYTES) return FGEMM_ERR_NOT_SUPPORTED;
    float *scratch = scratch_in_current_context();
    if (scratch == nullptr) return FGEMM_ERR_LAUNCH;
    // Every partial product is written before it is read, so nothing has to start
    // at zero.  No allocation happens below: the split-K path only launches kernels.
    return fgemm_sgemm_splitk(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                              apply_relu, splits, scratch, (size_t)FGEMM_NOALLOC_SCRATCH_BYTES,
                              stream);
}
