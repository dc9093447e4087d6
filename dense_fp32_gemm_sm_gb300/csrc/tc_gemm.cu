// tc_gemm.cu -- host side of the tensor-core path: TMA tensor maps, launch, and the
// device error word that bounded waits report into.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ctx_id.h"
#include "fgemm_internal.h"
#include "tc_gemm.cuh"

namespace fgemm {

// Bits set by a tensor-core kernel whose mbarrier wait ran out (see tc::ERR_*).
__device__ unsigned g_tc_error;

namespace {

// Testing hook (fgemm_debug_withhold_tensor_core): k-block the producer withholds,
// and the wait bound to use meanwhile.
std::atomic<int> g_withhold_kb{-1};
std::atomic<unsigned long long> g_wait_limit_ns{tc::kWaitLimitNs};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// One operand as a 3-D tensor map (inner, outer, batch), `batch` problems `stride`
// elements apart.  K-major storage (rows x K, K contiguous): inner = K, boxes of
// 32 x box_rows with the 128-byte swizzle (the canonical UMMA layout).  MN-major
// storage (K x rows, rows contiguous): inner = rows, plain box_rows x 32 boxes that
// the kernel transposes on chip.
bool make_operand_map(CUtensorMap *map, const float *base, bool kmajor, long long rows, long long K,
                      long long ld, long long batch, long long stride, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const long long outer = kmajor ? rows : K;
    if (batch <= 1) stride = ld * outer;  // unused extent-1 dimension; any legal stride
    const cuuint64_t dims[3] = {(cuuint64_t)(kmajor ? K : rows), (cuuint64_t)outer,
                                (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)stride * 4};
    const cuuint32_t box[3] = {kmajor ? (cuuint32_t)tc::BK : (cuuint32_t)box_rows,
                               kmajor ? (cuuint32_t)box_rows : (cuuint32_t)tc::BK, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r =
        enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            kmajor ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C as the 3-D tensor map (N, M, batch) of the TMA-store epilogue: 32 x 32 boxes
// with the 128-byte swizzle.
bool make_output_map(CUtensorMap *map, float *base, long long M, long long N, long long ldc,
                     long long batch, long long stride)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    if (batch <= 1) stride = ldc * M;
    const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ldc * 4, (cuuint64_t)stride * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_device(int *dev) { return cudaGetDevice(dev) == cudaSuccess ? 0 : -1; }

// Device address of g_tc_error in the current context, looked up once per context
// (a device reset loads the module again, and the variable may move).
unsigned *error_word()
{
    struct Entry {
        unsigned long long ctx;
        unsigned *addr;
    };
    static Entry cache[64];
    static std::mutex mu;
    int dev = 0;
    if (current_device(&dev) != 0) return nullptr;
    const unsigned long long ctx = current_context_id();
    if (ctx != 0) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev & 63].ctx == ctx) return cache[dev & 63].addr;
    }
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_tc_error) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[dev & 63] = Entry{current_context_id(), static_cast<unsigned *>(addr)};
    return static_cast<unsigned *>(addr);
}

// The kernel's dynamic shared memory attribute, set once per context.
template <int MODE, int TA, int TB>
cudaError_t prepare_tc()
{
    static std::atomic<unsigned long long> ready_ctx[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<unsigned long long> &ready = ready_ctx[dev & 63];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ready.load(std::memory_order_acquire) == ctx) return cudaSuccess;
    e = cudaFuncSetAttribute(tc::tc_gemm_kernel<MODE, TA, TB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::TcShape<MODE, TA, TB>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    ready.store(current_context_id(), std::memory_order_release);
    return cudaSuccess;
}

template <int MODE, int TA, int TB>
fgemm_status launch_tc_mode(const TcProblem &q, tc::TcParams &p, cudaStream_t stream)
{
    using Shape = tc::TcShape<MODE, TA, TB>;
    if (!make_operand_map(&p.tmA, q.A, TA == 0, q.M, q.K, q.lda, q.batch, q.sA, Shape::TILE_M) ||
        !make_operand_map(&p.tmB, q.B, TB == 1, q.N, q.K, q.ldb, q.batch, q.sB, Shape::TILE_N))
        return FGEMM_ERR_NOT_SUPPORTED;
    p.tiles_m = (q.M + Shape::TILE_M - 1) / Shape::TILE_M;
    p.tiles_n = (q.N + Shape::TILE_N - 1) / Shape::TILE_N;
    unsigned *err = error_word();
    int sms = 0;
    if (!err || prepare_tc<MODE, TA, TB>() != cudaSuccess || device_sm_count(&sms) != 0) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    // Persistent: one CTA per SM (or per tile, if there are fewer tiles).
    const long long tiles = (long long)p.tiles_m * p.tiles_n * p.batch;
    const long long grid = tiles < sms ? tiles : sms;
    // With 256-wide MMAs, a last partial wave of at most half the grid is run as twice
    // as many 128-wide half tiles, so it takes half as long.
    const long long rem = tiles % grid;
    p.full_items = tiles;
    p.total_items = tiles;
    if (Shape::MMA_N == 2 * tc::MMA_M && rem > 0 && 2 * rem <= grid) {
        p.full_items = tiles - rem;
        p.total_items = tiles + rem;
    }
    tc::tc_gemm_kernel<MODE, TA, TB><<<(unsigned)grid, tc::THREADS, Shape::SMEM_BYTES, stream>>>(p, err);
    return cudaGetLastError() == cudaSuccess ? FGEMM_OK : FGEMM_ERR_LAUNCH;
}

}  // namespace

bool tc_supported(const TcProblem &q)
{
    if (q.K <= 0 || q.alpha == 0.0f || q.M <= 0 || q.N <= 0 || q.batch <= 0) return false;
    if ((q.ta != 0 && q.ta != 1) || (q.tb != 0 && q.tb != 1)) return false;
    auto ok16 = [](const void *ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
    if (!ok16(q.A) || !ok16(q.B) || q.lda % 4 || q.ldb % 4) return false;
    if (q.batch > 1 && (q.sA % 4 || q.sB % 4)) return false;
    const long long lim = 1ll << 38;  // tensor-map strides are below 2^40 bytes
    if (q.lda >= lim || q.ldb >= lim || q.sA >= lim || q.sB >= lim) return false;
    // (the smallest tile of any instance is 128 x 128)
    if ((long long)((q.M + 127) / 128) * ((q.N + 127) / 128) > INT_MAX) return false;
    return encode_fn() != nullptr;
}

fgemm_status launch_tc(int mode, const TcProblem &q, cudaStream_t stream)
{
    tc::TcParams p;
    std::memset(&p, 0, sizeof(p));
    p.C = q.C;
    p.bias = q.bias;
    p.ldc = q.ldc;
    p.strideC = q.batch > 1 ? q.sC : 0;
    p.M = q.M;
    p.N = q.N;
    p.K = q.K;
    p.alpha = q.alpha;
    p.beta = q.beta;
    p.relu = q.relu ? 1 : 0;
    p.c_vec = (reinterpret_cast<uintptr_t>(q.C) % 16 == 0 && q.ldc % 4 == 0 &&
               (q.batch <= 1 || q.sC % 4 == 0))
                  ? 1
                  : 0;
    // TMA stores clip a box at the tensor's edge in whole 16-byte chunks (measured: with
    // N = 31 the store wrote column 31 of a padded C), so they are used only when the
    // last column ends a chunk.
    p.c_tma = (q.beta == 0.0f && p.c_vec && q.N % 4 == 0 && q.ldc < (1ll << 38) &&
               q.sC < (1ll << 38) && make_output_map(&p.tmC, q.C, q.M, q.N, q.ldc, q.batch, q.sC))
                  ? 1
                  : 0;
    p.batch = q.batch;
    p.withhold_kb = g_withhold_kb.load(std::memory_order_relaxed);
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    const int layout = q.ta * 2 + q.tb;  // 0: NN, 1: NT, 2: TN, 3: TT
    if (mode == tc::MODE_3XTF32) {
        switch (layout) {
        case 0: return launch_tc_mode<tc::MODE_3XTF32, 0, 0>(q, p, stream);
        case 1: return launch_tc_mode<tc::MODE_3XTF32, 0, 1>(q, p, stream);
        case 2: return launch_tc_mode<tc::MODE_3XTF32, 1, 0>(q, p, stream);
        default: return launch_tc_mode<tc::MODE_3XTF32, 1, 1>(q, p, stream);
        }
    }
    switch (layout) {
    case 0: return launch_tc_mode<tc::MODE_TF32, 0, 0>(q, p, stream);
    case 1: return launch_tc_mode<tc::MODE_TF32, 0, 1>(q, p, stream);
    case 2: return launch_tc_mode<tc::MODE_TF32, 1, 0>(q, p, stream);
    default: return launch_tc_mode<tc::MODE_TF32, 1, 1>(q, p, stream);
    }
}

void tc_debug_withhold(int k_block, long long wait_limit_ns)
{
    if (k_block < 0) {
        g_withhold_kb.store(-1);
        g_wait_limit_ns.store(tc::kWaitLimitNs);
    } else {
        g_withhold_kb.store(k_block);
        g_wait_limit_ns.store(wait_limit_ns > 0 ? (unsigned long long)wait_limit_ns
                                                : tc::kWaitLimitNs);
    }
}

fgemm_status tc_device_status(int clear)
{
    int dev = 0;
    if (current_device(&dev) != 0) return FGEMM_ERR_LAUNCH;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    if (v != 0 && clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
    }
    return v ? FGEMM_ERR_TIMEOUT : FGEMM_OK;
}

}  // namespace fgemm
