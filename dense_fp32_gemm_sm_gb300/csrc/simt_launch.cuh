// simt_launch.cuh -- host launchers for the SIMT kernel configurations.
#pragma once

#include <atomic>
#include <climits>

#include "ctx_id.h"
#include "fgemm_internal.h"
#include "simt_gemm.cuh"

namespace fgemm {

// The tile shapes behind each ConfigId.  Every configuration uses warps of
// 8 x 4 lanes; each thread owns groups of 4 consecutive rows and columns.
template <int ID, int TA, int TB>
struct ConfigOf;

// 256 threads, two CTAs per SM.  When both operands are stored with k contiguous (NT)
// the copies transpose both (32 element copies per thread per stage); with
// unpredicated interior copies that still fits 128 registers, and 32-deep stages
// measured faster than 16-deep ones there (QK^T 128 x 2048 x 2048 x 128: 56.4 against
// 52.7 TFLOP/s with 5 stages of 16; 4096^3 NT 56.3 against 54.4).
template <int TA, int TB>
struct ConfigOf<CFG_128x128, TA, TB> {
    using type = SimtCfg<128, 128, 32, 64, 32, 8, 8, 3, 2, TA, TB, true>;
};
template <int TA, int TB>
struct ConfigOf<CFG_128x64, TA, TB> {  // 128 threads, three CTAs per SM
    // (the unpredicated copy path measured 3.6 % slower on this tile at 1024^3)
    using type = SimtCfg<128, 64, 16, 64, 32, 8, 8, 4, 3, TA, TB, true, 1, false>;
};
template <int TA, int TB>
struct ConfigOf<CFG_64x64, TA, TB> {  // 256 threads, 4 x 4 per thread
    using type = SimtCfg<64, 64, 16, 32, 16, 4, 4, 4, 2, TA, TB, true>;
};
// The 128 x 128 tile with element-wise copies: any alignment.  A k-contiguous operand
// is copied element by element in every configuration (transposed on the way), so this
// differs from CFG_128x128 only for operands that config moves in 16-byte vectors.
template <int TA, int TB>
struct ConfigOf<CFG_128x128_SCALAR, TA, TB> {
    using type = SimtCfg<128, 128, 32, 64, 32, 8, 8, 3, 2, TA, TB, false>;
};

template <int TA, int TB>
struct ConfigOf<CFG_64x64_SCALAR, TA, TB> {  // element-wise copies: any alignment
    using type = SimtCfg<64, 64, 16, 32, 16, 4, 4, 4, 2, TA, TB, false>;
};

template <int TA, int TB>
struct ConfigOf<CFG_32x32, TA, TB> {  // 64 threads, 4 x 4 per thread: tiny problems
    using type = SimtCfg<32, 32, 16, 32, 16, 4, 4, 4, 8, TA, TB, true>;
};

// Four k-groups of two warps share each 32 x 32 tile (each group takes 8 of every
// stage's 32 k), and 8 stages keep 256 k in flight: for grids of a few hundred tiles
// or fewer, where the serial k-steps per thread and the load latency set the time.
// Measured on GB300 (L2 flushed, one call): 256^3 8.9 us against 10.9 us for the
// one-group 32 x 32 tile, 384^3 10.9 against 13.0; no gain from k-groups on larger
// tiles (128 x 64 at 1024^3: 68 us against 58 us).
template <int TA, int TB>
struct ConfigOf<CFG_32x32_K4, TA, TB> {
    using type = SimtCfg<32, 32, 32, 32, 16, 4, 4, 8, 2, TA, TB, true, 4>;
};

// The quarter tiles of the last-wave split: 64 x 64 with four k-groups of two
// warps (8 x 8 per thread), so a quarter tile has the CTA size, register budget and
// per-thread tile of a 128 x 128 tile and a quarter of its serial k-steps.  64-deep
// stages give each k-group 16 k per stage; when B is transposed on copy (NT, TT),
// 32-deep stages keep its element copies per thread at 16 (at 64 deep the TT instance
// needed 8 B of spill space).
template <int TA, int TB>
struct SplitTailOf {
    static constexpr bool B_T = TB == 1;
    using type = SimtCfg<64, 64, B_T ? 32 : 64, 64, 32, 8, 8, B_T ? 4 : 3, 2, TA, TB, true, 4>;
};

// Opt a kernel in to its dynamic shared memory once per context (attributes belong to
// the context's copy of the kernel; a device reset drops them).  Tag makes the
// per-context record distinct per kernel.
template <class Tag, class KernelFn>
static cudaError_t prepare_kernel_fn(KernelFn kernel, int smem_bytes)
{
    static std::atomic<unsigned long long> ready_ctx[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<unsigned long long> &ready = ready_ctx[dev & 63];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ready.load(std::memory_order_acquire) == ctx) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    // the calls above made the device's primary context current if none was
    ready.store(current_context_id(), std::memory_order_release);
    return cudaSuccess;
}

template <class Cfg>
static cudaError_t prepare_kernel()
{
    return prepare_kernel_fn<Cfg>(simt_gemm_kernel<Cfg>, Cfg::SMEM_BYTES);
}

// Whole 128 x 128 tiles of TT problems always run in the one-dimensional linear tile
// order (the same grouped order within each problem as TILE_GRID): with TILE_GRID's
// index arithmetic that instance needs 12 B of spill space at its 128-register budget,
// with TILE_LINEAR's none (ptxas; register allocation at the budget moves with small
// code changes).
template <class Cfg>
constexpr bool kLinearWhole = Cfg::TA == 1 && Cfg::TB == 1 && Cfg::BM == 128 &&
                              Cfg::BN == 128 && Cfg::KS == 1;

template <class Cfg>
static fgemm_status launch_simt(const GemmParams &p0, int batch, cudaStream_t stream)
{
    GemmParams p = p0;
    p.tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    p.tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const long long tiles = (long long)p.tiles_m * p.tiles_n;
    if (tiles > INT_MAX) return FGEMM_ERR_NOT_SUPPORTED;
    if constexpr (kLinearWhole<Cfg>) {
        struct LinearTag {};
        if (prepare_kernel_fn<LinearTag>(simt_gemm_kernel<Cfg, TILE_LINEAR>, Cfg::SMEM_BYTES) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
        // One launch of tiles x batch CTAs, in chunks of problems when that exceeds a grid.
        const long long per_launch = INT_MAX / tiles;
        for (long long b0 = 0; b0 < batch; b0 += per_launch) {
            const long long nb = batch - b0 < per_launch ? batch - b0 : per_launch;
            GemmParams q = p;
            if (b0) {
                if (q.A) q.A += b0 * q.strideA;
                if (q.B) q.B += b0 * q.strideB;
                q.C += b0 * q.strideC;
            }
            simt_gemm_kernel<Cfg, TILE_LINEAR><<<(unsigned)(tiles * nb), Cfg::THREADS,
                                                 Cfg::SMEM_BYTES, stream>>>(q);
            if (cudaGetLastError() != cudaSuccess) return FGEMM_ERR_LAUNCH;
        }
        return FGEMM_OK;
    } else {
        if (prepare_kernel<Cfg>() != cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
        const int kMaxZ = 65535;
        for (int b0 = 0; b0 < batch; b0 += kMaxZ) {
            const int nb = batch - b0 < kMaxZ ? batch - b0 : kMaxZ;
            GemmParams q = p;
            if (b0) {
                if (q.A) q.A += (long long)b0 * q.strideA;
                if (q.B) q.B += (long long)b0 * q.strideB;
                q.C += (long long)b0 * q.strideC;
            }
            simt_gemm_kernel<Cfg><<<dim3((unsigned)tiles, 1, (unsigned)nb), Cfg::THREADS,
                                    Cfg::SMEM_BYTES, stream>>>(q);
            if (cudaGetLastError() != cudaSuccess) return FGEMM_ERR_LAUNCH;
        }
        return FGEMM_OK;
    }
}

// Plan of a last-wave split over Main-sized tiles: tile counts, the whole tiles of
// all problems (p.full_units) and the remainder r = tiles mod SMs, whose tiles then
// run as tail_ctas CTAs each.
template <class Main>
static fgemm_status plan_split(GemmParams &p, int batch, int tail_ctas, long long *rem)
{
    p.tiles_m = (p.M + Main::BM - 1) / Main::BM;
    p.tiles_n = (p.N + Main::BN - 1) / Main::BN;
    const long long total = (long long)p.tiles_m * p.tiles_n * batch;
    int sms = 0;
    if (device_sm_count(&sms) != 0 || sms < 1) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    *rem = total % sms;
    if (total - *rem > INT_MAX || (long long)tail_ctas * *rem > INT_MAX)
        return FGEMM_ERR_NOT_SUPPORTED;
    p.full_units = (int)(total - *rem);
    return FGEMM_OK;
}

// The first launch of a split: the whole tiles.  One problem: the per-problem kernel
// over the first full_units tiles.  A batch: the linear-order kernel, whose whole
// tiles may end inside a problem.
template <class Main>
static fgemm_status launch_whole_tiles(const GemmParams &p, int batch, cudaStream_t stream)
{
    struct LinearTag {};
    if constexpr (!kLinearWhole<Main>) {
        if (prepare_kernel<Main>() != cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
    }
    if (prepare_kernel_fn<LinearTag>(simt_gemm_kernel<Main, TILE_LINEAR>, Main::SMEM_BYTES) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    if (p.full_units <= 0) return FGEMM_OK;
    if constexpr (!kLinearWhole<Main>) {
        if (batch == 1) {
            simt_gemm_kernel<Main><<<(unsigned)p.full_units, Main::THREADS, Main::SMEM_BYTES,
                                     stream>>>(p);
            return cudaGetLastError() == cudaSuccess ? FGEMM_OK : FGEMM_ERR_LAUNCH;
        }
    }
    simt_gemm_kernel<Main, TILE_LINEAR><<<(unsigned)p.full_units, Main::THREADS,
                                         Main::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FGEMM_OK : FGEMM_ERR_LAUNCH;
}

// Last-wave split: the first (tiles - r) tiles of all problems whole, then the
// last r = tiles mod SMs as quarter tiles (TILE_QUARTER), two launches on
// the stream.
template <class Main, class Tail>
static fgemm_status launch_simt_split(const GemmParams &p0, int batch, cudaStream_t stream)
{
    struct TailTag {};
    static_assert(Tail::THREADS == Main::THREADS, "tail CTAs fill the slots of main CTAs");
    GemmParams p = p0;
    long long rem = 0;
    fgemm_status st = plan_split<Main>(p, batch, 4, &rem);
    if (st != FGEMM_OK) return st;
    if (prepare_kernel_fn<TailTag>(simt_gemm_kernel<Tail, TILE_QUARTER, Main>, Tail::SMEM_BYTES) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    st = launch_whole_tiles<Main>(p, batch, stream);
    if (st != FGEMM_OK) return st;
    if (rem > 0) {
        // A programmatic dependent of the whole tiles when there are any (it starts on
        // the SMs they leave and waits for them before its stores); otherwise the call's
        // first launch, in plain stream order.
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(4 * rem), 1, 1);
        cfg.blockDim = dim3(Tail::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Tail::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = p.full_units > 0 ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, simt_gemm_kernel<Tail, TILE_QUARTER, Main>, p, 0) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
    }
    return FGEMM_OK;
}

// Last-wave k-split: the first (tiles - r) tiles whole, then each of the last
// r = tiles mod SMs tiles as a cluster of KSPLIT CTAs, one k-slice each, reduced
// through distributed shared memory (TILE_KSPLIT); two launches on the stream.
template <class Main>
static fgemm_status launch_simt_ksplit(const GemmParams &p0, int batch, cudaStream_t stream)
{
    struct KsplitTag {};
    GemmParams p = p0;
    long long rem = 0;
    fgemm_status st = plan_split<Main>(p, batch, KSPLIT, &rem);
    if (st != FGEMM_OK) return st;
    if (prepare_kernel_fn<KsplitTag>(simt_gemm_kernel<Main, TILE_KSPLIT>, Main::SMEM_BYTES) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    st = launch_whole_tiles<Main>(p, batch, stream);
    if (st != FGEMM_OK) return st;
    if (rem > 0) {
        // Clusters of KSPLIT; a programmatic dependent of the whole tiles when there are
        // any (see launch_simt_split).
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = KSPLIT;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(KSPLIT * rem), 1, 1);
        cfg.blockDim = dim3(Main::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Main::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = p.full_units > 0 ? 2 : 1;
        if (cudaLaunchKernelEx(&cfg, simt_gemm_kernel<Main, TILE_KSPLIT>, p, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
    }
    return FGEMM_OK;
}

// Last-wave k-chain: the first (tiles - r) tiles whole, then the last r = tiles mod SMs
// tiles in S k-slices (S = kchain_slices, from the launch-time model: 4 for the 112
// tiles of 4096^3), one launch per slice (TILE_KCHAIN).  Every slice's launch is a
// programmatic dependent of the launch before it (it may start while that one runs and
// waits for it only before writing C), so the slices' products run side by side over
// r * S CTAs and on SMs the whole tiles have left; the additions into C happen in slice
// order.  The first launch of the call is never a dependent: it follows the stream's
// earlier work, which may have written A or B.

template <class Main>
static fgemm_status launch_simt_kchain(const GemmParams &p0, int batch, cudaStream_t stream)
{
    struct KchainTag {};
    GemmParams p = p0;
    long long rem = 0;
    fgemm_status st = plan_split<Main>(p, batch, 1, &rem);
    if (st != FGEMM_OK) return st;
    if (prepare_kernel_fn<KchainTag>(simt_gemm_kernel<Main, TILE_KCHAIN>, Main::SMEM_BYTES) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    int sms = 0;
    if (device_sm_count(&sms) != 0) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    const int slices = kchain_slices(Main::TA, Main::TB, rem, p.K, sms);
    st = launch_whole_tiles<Main>(p, batch, stream);
    if (st != FGEMM_OK) return st;
    for (int s = 0; rem > 0 && s < slices; ++s) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)rem, 1, 1);
        cfg.blockDim = dim3(Main::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Main::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        // Slice 0 may start while the whole tiles of this call finish (they trigger their
        // dependents at once); with no whole tiles it is the call's first launch and
        // follows the stream's earlier work in plain stream order.
        cfg.numAttrs = (s > 0 || p.full_units > 0) ? 1 : 0;
        const int chain = s | (slices << 8);
        if (cudaLaunchKernelEx(&cfg, simt_gemm_kernel<Main, TILE_KCHAIN>, p, chain) != cudaSuccess) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
    }
    return FGEMM_OK;
}

#define FGEMM_LAUNCH_TABLE(NAME, TA, TB)                                   \
    const LaunchFn NAME[NUM_CONFIGS] = {                                   \
        &launch_simt<ConfigOf<CFG_128x128, TA, TB>::type>,                 \
        &launch_simt<ConfigOf<CFG_128x64, TA, TB>::type>,                  \
        &launch_simt<ConfigOf<CFG_64x64, TA, TB>::type>,                   \
        &launch_simt<ConfigOf<CFG_64x64_SCALAR, TA, TB>::type>,            \
        &launch_simt<ConfigOf<CFG_32x32, TA, TB>::type>,                   \
        &launch_simt<ConfigOf<CFG_32x32_K4, TA, TB>::type>,                \
        &launch_simt_split<ConfigOf<CFG_128x128, TA, TB>::type,            \
                           SplitTailOf<TA, TB>::type>,                     \
        &launch_simt_ksplit<ConfigOf<CFG_128x128, TA, TB>::type>,          \
        &launch_simt_kchain<ConfigOf<CFG_128x128, TA, TB>::type>,          \
        &launch_simt<ConfigOf<CFG_128x128_SCALAR, TA, TB>::type>,          \
    };                                                                     \
    static_assert(NUM_CONFIGS == 10, "one launcher per configuration");

}  // namespace fgemm
