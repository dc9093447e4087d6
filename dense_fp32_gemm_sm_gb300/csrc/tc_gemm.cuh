// tc_gemm.cuh -- the same GEMM on the 5th-generation tensor cores of sm_103a
// (tcgen05), in TF32 or in 3xTF32.
//
// The pages name tensor cores as the next step after the CUDA-core ladder
// (GEMM 优化详解, "进一步优化方向 / Tensor Core"; GPU架构下的矩阵乘法深入优化,
// "6. fp32 + tensor core" uses FP16 WMMA on V100).  Here the contraction stays FP32
// in, FP32 out:
//
//   TF32   : D += A * B with each FP32 operand read as TF32 (10 explicit mantissa bits).
//   3xTF32 : every operand x is split on chip into hi = x with the low 13 mantissa
//            bits cleared (exactly representable in TF32) and lo = x - hi (exact in
//            FP32), and D += A_lo*B_hi + A_hi*B_lo + A_hi*B_hi.  (The MMA itself reads
//            an FP32 operand as hi, so an operand kept in shared memory stays as loaded
//            and only its lo is written.)  The dropped term
//            A_lo*B_lo and the TF32 rounding of lo are about 2^-21 relative to |a||b|:
//            close to FP32 accuracy (the split of Ootomo & Yokota, "Recovering single
//            precision accuracy from Tensor Cores while surpassing the FP32 theoretical
//            peak performance", 2022).
//
// Structure: a persistent kernel, one CTA per SM, each CTA walking work items (C
// tiles, item = blockIdx.x, + gridDim.x, ...; a last partial wave of 256-wide tiles
// runs as 128-wide halves), ten warps:
//   warp 0     TMA producer: one lane streams the operand tiles of every k-block (32
//              deep; 128-byte swizzled boxes for K-major operands, plain boxes for
//              MN-major ones) into a ring of stages, running ahead across items.
//   warp 1     allocates tensor memory; one lane issues tcgen05.mma (M=128, N=MMA_N,
//              K=8) into one or two FP32 accumulators and commits each stage back to
//              the producer through an mbarrier.
//   warps 2-5  (every layout but TF32 NT) move one operand of each stage from shared
//              memory through registers into tensor memory, where the MMA reads it as
//              its A operand -- transposed on the way when stored MN-major, split into
//              hi and lo in 3xTF32 -- and write the lo part of the other operand beside
//              it (3xTF32) or transpose it (both operands MN-major) in shared memory.
//   warps 6-9  epilogue of the previous item while the next one is being multiplied
//              (warps 2-5 join them when there is nothing to convert): tcgen05.ld of
//              their 32 accumulator lanes, alpha, beta*C, bias, ReLU; with beta == 0
//              (and N a multiple of 4) the tile is staged in shared memory and written by
//              TMA stores, otherwise stored directly; then the accumulator is handed
//              back to the MMA warp.
// TcShape below fixes, per layout and mode, which operand goes through tensor memory,
// the MMA's N (256 in TF32 when one operand is K-major, else 128) and the number of
// accumulators.  In NN the tensor-memory operand is B, so the MMA computes C^T and the
// epilogue reads accumulator lanes as columns of C.  Every mbarrier wait is bounded by
// a wall-clock limit: on expiry the kernel records the failure in a device error word,
// drains its own copies and MMAs, frees its tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fgemm {
namespace tc {

constexpr int MMA_M = 128;  // rows of the MMA = tensor-memory lanes
constexpr int BK = 32;      // k per stage: 32 FP32 values = one 128-byte swizzle row
constexpr int UMMA_K = 8;   // K of one kind::tf32 MMA (32 bytes)
constexpr int THREADS = 320;  // 10 warps, see the kernel
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // default: 4 s per wait

// Error bits recorded in the device error word.
constexpr unsigned ERR_PRODUCER = 1u, ERR_MMA_WAIT = 2u, ERR_SPLIT_WAIT = 4u, ERR_EPILOGUE = 8u,
                   ERR_DRAIN = 16u;

enum Mode { MODE_TF32 = 1, MODE_3XTF32 = 3 };

// Shapes of one kernel instance.  The MMA is 128 x MMA_N x 8; MMA_N = 256 halves the
// MMA instructions and the operand traffic per FLOP against 128 (measured, TF32 NT:
// 549 -> 659 TFLOP/s at 4096^3, 599 -> 820 at 8192^3), and is used in TF32 whenever one
// operand is K-major.  3xTF32 keeps MMA_N = 128: its extra lo tile leaves room for only
// two stages at 256 (measured 190 against 240 TFLOP/s at 4096^3).  The operand that goes through tensor memory (see the
// kernel) is always the 128-row side; with MMA_N = 256 there is room in tensor memory
// for it or for a second accumulator, not both, so those layouts use one accumulator.
template <int MODE, int TA, int TB>
struct TcShape {
    static constexpr bool A_K = TA == 0, B_K = TB == 1;  // operand stored K-major
    static constexpr bool THREE = MODE == MODE_3XTF32;
    // Which operand reaches the MMA through tensor memory (as its A operand):
    // B when A is K-major and B is not (NN: the MMA then computes C^T), else A in
    // 3xTF32 or when A is stored K x M; TF32 NT uses none.
    static constexpr bool B_VIA_TMEM = A_K && !B_K;
    static constexpr bool A_VIA_TMEM = !B_VIA_TMEM && (THREE || !A_K);
    static constexpr bool TMEM_OP = A_VIA_TMEM || B_VIA_TMEM;
    static constexpr bool TRANS_OUT = B_VIA_TMEM;
    static constexpr bool WIDE = !THREE && (A_K || B_K);
    static constexpr int MMA_N = WIDE ? 256 : 128;
    static constexpr int NACC = (TMEM_OP && WIDE) ? 1 : 2;  // accumulators in tensor memory
    // The C tile of one MMA sequence: MMA rows are C rows, or C columns when TRANS_OUT.
    static constexpr int TILE_M = TRANS_OUT ? MMA_N : MMA_M;
    static constexpr int TILE_N = TRANS_OUT ? MMA_M : MMA_N;
    static constexpr int A_BYTES = TILE_M * BK * 4;
    static constexpr int B_BYTES = TILE_N * BK * 4;
    // 3xTF32: the lo part of the operand that stays in shared memory (128 rows).
    static constexpr int LO_BYTES = THREE ? MMA_M * BK * 4 : 0;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + LO_BYTES;
    static constexpr int STAGES = STAGE_BYTES > 32768 ? 4 : 6;
    // Tensor-memory columns: the accumulators, then per stage 32 columns of the MMA's
    // A operand (64 in 3xTF32: hi, lo).
    static constexpr uint32_t ACC_COLS = NACC * MMA_N;
    static constexpr uint32_t OP_COLS = THREE ? 64 : 32;
    static constexpr uint32_t TMEM_COLS = TMEM_OP ? 512 : ACC_COLS;
    static_assert(!TMEM_OP || ACC_COLS + STAGES * OP_COLS <= TMEM_COLS, "tensor-memory columns");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "allocation: a power of two");
    // Epilogue staging: 32 KB, two 4 KB chunk buffers per epilogue warp (four warps),
    // or one per warp when eight warps share the epilogue.
    static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = 4 * 8192;
    static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_BYTES;
    // full[S], split[S], empty[S], acc_full[2], acc_empty[2], drain, read_done, TMEM slot
    static constexpr int BAR_BYTES = (3 * STAGES + 6) * 8 + 8;
    static constexpr int SMEM_BYTES = 1024 + BAR_OFFSET + BAR_BYTES;  // + alignment slack
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

struct TcParams {
    // K-major operand: dims (K, rows, batch), box (32, tile rows, 1), 128-byte swizzle.
    // MN-major operand: dims (rows, K, batch), box (128, 32, 1), no swizzle.
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmC;  // C: dims (N, M, batch), box (32, 32, 1), 128-byte swizzle (stores)
    float *C;
    const float *bias;
    long long ldc, strideC;
    int M, N, K;
    float alpha, beta;
    int relu;
    int c_vec;
    int c_tma;  // beta == 0 and C allows TMA stores: stage rows in shared memory
    int tiles_m, tiles_n;
    int batch;   // problems in the strided batch; tiles run over (batch, tile-row, tile-col)
    // Work items: items [0, full_items) are whole tiles; items from full_items on split
    // each remaining tile into two halves of 128 along the MMA's N (the last partial
    // wave then takes half as long).  total_items = full_items when nothing is split.
    long long full_items, total_items;
    unsigned long long wait_limit_ns;  // bound of every mbarrier wait
    int withhold_kb;  // testing: the producer never issues this k-block (-1: none)
};

// ---- PTX wrappers ----------------------------------------------------------------

__device__ __forceinline__ uint32_t cvta_smem(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the phase with the given parity has completed, for at most
// limit_ns.  With `give_up_on_error`, stop early once any CTA has recorded an
// error (drain waits must not: they guard copies still landing in shared memory).
// On expiry, record `code` and return false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *err,
                                          unsigned code, unsigned long long limit_ns,
                                          bool give_up_on_error = true)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 0) {
            if (give_up_on_error && *(volatile unsigned *)err != 0u) return false;
            if (global_timer() - t0 > limit_ns) {
                atomicOr(err, code);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the canonical 128-byte
// swizzled layout: rows of 128 bytes (32 FP32 along K), groups of 8 rows 1024 bytes
// apart (stride byte offset), 1024-byte aligned base, descriptor version 1.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t smem_addr)
{
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::tf32: D FP32, A and B TF32, both K-major, M x N.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA with the A operand read from tensor memory (128 lanes = rows of A,
// one 32-bit column per element along K) instead of shared memory.
__device__ __forceinline__ void umma_tf32_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 32 consecutive columns of this thread's tensor-memory lane (warp-wide: lane i
// of the warp writes lane base + i); complete before return.
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// hi = x with the 13 low mantissa bits cleared (a TF32 value); lo = x - hi, exact.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo)
{
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    lo = x - hi;
}

// ---- Split / transpose of one stage (warps 2-5, thread t in 0..127) --------------

// K-major operand tile (already in the canonical swizzled layout): lo goes to the same
// offsets of the lo tile; the tile itself stays as TMA wrote it.  The MMA reads an FP32
// operand as TF32 by dropping its 13 low mantissa bits -- measured on GB300 for operands
// in shared and in tensor memory: 1 + 3/4 ulp and 1 + 1/2 ulp read as 1, 2 + 7/4 ulp as
// 2 + 1 ulp -- so the raw tile is read as exactly hi, and writing hi back is not needed.
__device__ __forceinline__ void split_kmajor(const float4 *tile, float4 *lo, int t)
{
#pragma unroll 4
    for (int c = t; c < MMA_M * BK * 4 / 16; c += 128) {
        const float4 v = tile[c];
        float4 h, l;
        split_tf32(v.x, h.x, l.x);
        split_tf32(v.y, h.y, l.y);
        split_tf32(v.z, h.z, l.z);
        split_tf32(v.w, h.w, l.w);
        lo[c] = l;
    }
}

// Byte offset of element (row r, k) in a 128-row K-major tile with 128-byte rows and
// the 128-byte swizzle (16-byte chunk index XOR row % 8, 8-row groups of 1024 bytes).
__device__ __forceinline__ int kmajor_offset(int r, int kq)
{
    return (r >> 3) * 1024 + (r & 7) * 128 + ((kq ^ (r & 7)) << 4);
}

// MN-major tile: 32 rows of k, each 128 floats along m (or n), as TMA wrote it.  Each
// thread reads 8 (row, k-quad) pairs -- rows lane + 32j, k-quads 2*wq + i -- so a warp
// reads 32 consecutive floats of one k row per load; after every converter thread has
// read (bounded wait on read_done), it writes its values back K-major (swizzled
// 16-byte chunks, conflict-free per quarter warp), and the lo parts for 3xTF32.
template <bool SPLIT>
__device__ __forceinline__ bool transpose_mnmajor(uint8_t *tile, uint8_t *lo, int t, uint32_t read_done,
                                                  uint32_t parity, unsigned *err,
                                                  unsigned long long limit_ns)
{
    const int lane = t & 31, wq = t >> 5;
    const float *src = reinterpret_cast<const float *>(tile);
    float v[8][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = lane + 32 * j, kq = 2 * wq + i;
#pragma unroll
            for (int e = 0; e < 4; ++e) v[2 * j + i][e] = src[(4 * kq + e) * 128 + r];
        }
    mbar_arrive(read_done);
    if (!mbar_wait(read_done, parity, err, ERR_SPLIT_WAIT, limit_ns)) return false;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = lane + 32 * j, kq = 2 * wq + i;
            const float *x = v[2 * j + i];
            float4 h, l;
            if constexpr (SPLIT) {
                split_tf32(x[0], h.x, l.x);
                split_tf32(x[1], h.y, l.y);
                split_tf32(x[2], h.z, l.z);
                split_tf32(x[3], h.w, l.w);
                *reinterpret_cast<float4 *>(lo + kmajor_offset(r, kq)) = l;
            } else {
                h = make_float4(x[0], x[1], x[2], x[3]);
            }
            *reinterpret_cast<float4 *>(tile + kmajor_offset(r, kq)) = h;
        }
    return true;
}

// MN-major tile -> tensor memory, for the A operand of the MMA: tile row r (one m,
// or one n) becomes tensor-memory lane r, k its column.  TMA wrote the tile as 32 rows
// of k, 128 floats each; thread r (lane r of the tile, in the 32-lane quarter its warp
// may access) reads column r of that -- a warp reads 128 consecutive bytes per k, no
// bank conflict -- so the transpose happens in registers, and shared memory sees one
// read of the tile instead of a read and a write.  3xTF32: hi and lo go to two
// column ranges.
template <bool SPLIT>
__device__ __forceinline__ void mnmajor_to_tmem(const uint8_t *tile, int r, uint32_t t_hi,
                                                uint32_t t_lo)
{
    const float *src = reinterpret_cast<const float *>(tile) + r;
    uint32_t h[32];
    if constexpr (SPLIT) {
        uint32_t l[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float hi, lo;
            split_tf32(src[k * 128], hi, lo);
            h[k] = __float_as_uint(hi);
            l[k] = __float_as_uint(lo);
        }
        tmem_st_32cols(t_hi, h);
        tmem_st_32cols(t_lo, l);
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) h[k] = __float_as_uint(src[k * 128]);
        tmem_st_32cols(t_hi, h);
    }
    tmem_st_wait();
}

// K-major tile (canonical 128-byte swizzled layout) -> tensor memory: thread r reads
// row r (eight 16-byte chunks; a warp's loads of one chunk index cover all 32 banks)
// into tensor-memory lane r, k as its column.  3xTF32: hi and lo go to two column
// ranges.
template <bool SPLIT>
__device__ __forceinline__ void kmajor_to_tmem(const uint8_t *tile, int r, uint32_t t_hi,
                                               uint32_t t_lo)
{
    uint32_t h[32];
    uint32_t l[SPLIT ? 32 : 1];
#pragma unroll
    for (int kq = 0; kq < 8; ++kq) {
        const float4 v = *reinterpret_cast<const float4 *>(tile + kmajor_offset(r, kq));
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (SPLIT) {
                float hi, lo;
                split_tf32(x[e], hi, lo);
                h[4 * kq + e] = __float_as_uint(hi);
                l[4 * kq + e] = __float_as_uint(lo);
            } else {
                h[4 * kq + e] = __float_as_uint(x[e]);
            }
        }
    }
    tmem_st_32cols(t_hi, h);
    if constexpr (SPLIT) tmem_st_32cols(t_lo, reinterpret_cast<const uint32_t (&)[32]>(l));
    tmem_st_wait();
}

// ---- The kernel ------------------------------------------------------------------

// MODE: MODE_TF32 or MODE_3XTF32.  TA = 0: A stored M x K (K-major), 1: K x M.
// TB = 1: B stored N x K (K-major), 0: K x N.
template <int MODE, int TA, int TB>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p, unsigned *err)
{
    using L = TcShape<MODE, TA, TB>;
    constexpr int S = L::STAGES;
    constexpr bool A_K = L::A_K, B_K = L::B_K, THREE = L::THREE;
    constexpr bool CONVERT = THREE || !A_K || !B_K;  // warps 2-5 touch each stage
    // One operand goes to tensor memory as the MMA's A operand, written there from
    // registers by warps 2-5 (transposed on the way when it is stored MN-major, split
    // into hi and lo in 3xTF32), so the tensor core reads only the other operand from
    // shared memory; in NN that is A, and the MMA computes the transposed tile D = C^T
    // (tensor-memory lanes are columns of C).  See TcShape for which goes where.
    constexpr bool B_VIA_TMEM = L::B_VIA_TMEM, TMEM_OP = L::TMEM_OP, TRANS_OUT = L::TRANS_OUT;
    constexpr int MMA_N = L::MMA_N, NACC = L::NACC;
    constexpr uint32_t ACC_COLS = L::ACC_COLS, OP_COLS = L::OP_COLS, TMEM_COLS = L::TMEM_COLS;
    // Without a split or transpose, warps 2-5 share the epilogue with warps 6-9.
    constexpr int EPI_WARPS = CONVERT ? 4 : 8;
    constexpr int EPI_COLS = MMA_N * 4 / EPI_WARPS;  // accumulator columns per epilogue warp
    constexpr int EPI_BUFS = 8 / (EPI_WARPS / 4) / 4;  // 4 KB buffers per epilogue warp
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment of the operand tiles (the swizzle atom).
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = cvta_smem(smem);
    const uint32_t bar0 = sbase + L::BAR_OFFSET;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto split_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto acc_full_bar = [&](int a) { return bar0 + 8u * (3 * S + a); };
    auto acc_empty_bar = [&](int a) { return bar0 + 8u * (3 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (3 * S + 4);
    const uint32_t read_bar = bar0 + 8u * (3 * S + 5);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::BAR_OFFSET + 8 * (3 * S + 6));

    auto a_off = [&](int s) { return s * L::STAGE_BYTES; };
    auto b_off = [&](int s) { return s * L::STAGE_BYTES + L::A_BYTES; };
    auto lo_off = [&](int s) { return s * L::STAGE_BYTES + L::A_BYTES + L::B_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = (p.K + BK - 1) / BK;
    const int tiles_per_problem = p.tiles_m * p.tiles_n;
    const long long total_items = p.total_items;
    const unsigned long long lim = p.wait_limit_ns;
    // The j-th tile of this CTA: problem bz, rows m0.., columns n0.. (grouped order:
    // 8 tile-rows swept column by column, so resident CTAs share panels in L2).
    auto tile_coords = [&](long long t, int &m0, int &n0, int &bz) {
        bz = (int)(t / tiles_per_problem);
        const int r = (int)(t - (long long)bz * tiles_per_problem);
        const int per_group = 8 * p.tiles_n;
        const int group = r / per_group;
        const int first_m = group * 8;
        const int rows_in_group = min(p.tiles_m - first_m, 8);
        const int in_group = r - group * per_group;
        m0 = (first_m + in_group % rows_in_group) * L::TILE_M;
        n0 = (in_group / rows_in_group) * L::TILE_N;
    };
    // Work item w: its tile's origin, moved to the second half for the odd half-item;
    // `narrow` items multiply 128 instead of MMA_N columns of the accumulator.
    auto item_coords = [&](long long w, int &m0, int &n0, int &bz, bool &narrow) {
        narrow = w >= p.full_items;
        const long long h = w - p.full_items;
        tile_coords(narrow ? p.full_items + h / 2 : w, m0, n0, bz);
        if (narrow && (h & 1)) {
            if constexpr (TRANS_OUT)
                m0 += MMA_M;
            else
                n0 += MMA_M;
        }
    };

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(split_bar(s), 128);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full_bar(a), 1);
            mbar_init(acc_empty_bar(a), EPI_WARPS);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        mbar_init(read_bar, 128);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         cvta_smem(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    if (warp == 0) {
        // ---- TMA producer: every k-block of every tile of this CTA, in order ----
        if (lane == 0) {
            int g = 0;  // k-blocks issued so far (runs across tiles)
            bool ok = true;
            for (long long t = blockIdx.x; ok && t < total_items; t += gridDim.x) {
                int m0, n0, bz;
                bool narrow;
                item_coords(t, m0, n0, bz, narrow);
                for (int kb = 0; kb < KT; ++kb) {
                    const int s = g % S, round = g / S;
                    if (round > 0 && !mbar_wait(empty_bar(s), (round - 1) & 1, err, ERR_PRODUCER, lim)) {
                        ok = false;
                        break;
                    }
                    if (g == p.withhold_kb) {  // testing: as if this copy never arrived
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), L::A_BYTES + L::B_BYTES);
                    if constexpr (A_K)
                        tma_load_3d(sbase + a_off(s), &p.tmA, full_bar(s), kb * BK, m0, bz);
                    else
                        tma_load_3d(sbase + a_off(s), &p.tmA, full_bar(s), m0, kb * BK, bz);
                    if constexpr (B_K)
                        tma_load_3d(sbase + b_off(s), &p.tmB, full_bar(s), kb * BK, n0, bz);
                    else
                        tma_load_3d(sbase + b_off(s), &p.tmB, full_bar(s), n0, kb * BK, bz);
                    ++g;
                }
            }
            // Never leave with copies in flight into this CTA's shared memory.
            for (int k = g - S < 0 ? 0 : g - S; k < g; ++k)
                mbar_wait(full_bar(k % S), (k / S) & 1, err, ERR_DRAIN, lim, false);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: accumulator j % NACC for this CTA's j-th tile ----
        if (lane == 0) {
            constexpr uint32_t idesc_full = make_idesc(MMA_M, MMA_N);
            constexpr uint32_t idesc_narrow = make_idesc(MMA_M, MMA_M);
            int g = 0;
            bool ok = true;
            int j = 0;
            for (long long t = blockIdx.x; ok && t < total_items; t += gridDim.x, ++j) {
                const uint32_t idesc = t >= p.full_items ? idesc_narrow : idesc_full;
                const int acc = j % NACC, use = j / NACC;
                // The epilogue must have drained this accumulator (tile j - NACC).
                if (use > 0 && !mbar_wait(acc_empty_bar(acc), (use - 1) & 1, err, ERR_MMA_WAIT, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * MMA_N);
                for (int kb = 0; kb < KT; ++kb, ++g) {
                    const int s = g % S, round = g / S;
                    ok = CONVERT ? mbar_wait(split_bar(s), round & 1, err, ERR_MMA_WAIT, lim)
                                 : mbar_wait(full_bar(s), round & 1, err, ERR_MMA_WAIT, lim);
                    if (!ok) break;
                    tc_fence_after();
                    if constexpr (TMEM_OP) {
                        // A operand in tensor memory; B operand = the other (K-major) tile.
                        const uint32_t at = tmem + ACC_COLS + (uint32_t)s * OP_COLS;
                        const int kop = B_VIA_TMEM ? a_off(s) : b_off(s);
                        const int kop_lo = lo_off(s);
                        const uint64_t bd = kmajor_sw128_desc(sbase + kop);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t koff = (uint64_t)((k * UMMA_K * 4) >> 4);
                            const uint32_t ak = at + (uint32_t)(k * UMMA_K);
                            if constexpr (THREE) {
                                const uint64_t bld = kmajor_sw128_desc(sbase + kop_lo);
                                umma_tf32_tmem_a(d, ak + 32u, bd + koff, idesc, (kb | k) != 0);
                                umma_tf32_tmem_a(d, ak, bld + koff, idesc, 1u);
                                umma_tf32_tmem_a(d, ak, bd + koff, idesc, 1u);
                            } else {
                                umma_tf32_tmem_a(d, ak, bd + koff, idesc, (kb | k) != 0);
                            }
                        }
                        umma_commit(empty_bar(s));
                        continue;
                    }
                    // TF32 with both operands K-major: the TMA tiles feed the MMA.
                    const uint64_t ad = kmajor_sw128_desc(sbase + a_off(s));
                    const uint64_t bd = kmajor_sw128_desc(sbase + b_off(s));
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t koff = (uint64_t)((k * UMMA_K * 4) >> 4);  // 32 bytes per step
                        umma_tf32(d, ad + koff, bd + koff, idesc, (kb | k) != 0);
                    }
                    umma_commit(empty_bar(s));  // the stage is free once these MMAs have read it
                }
                if (ok) umma_commit(acc_full_bar(acc));  // accumulator j is complete
            }
            if (!ok) {
                // Give up: make sure nothing issued is still running before teardown.
                umma_commit(drain_bar);
                mbar_wait(drain_bar, 0, err, ERR_DRAIN, lim, false);
            }
        }
    } else if (CONVERT && warp < 6) {
        // ---- warps 2..5: each stage's tensor-memory operand, and the split or
        // transpose of the shared-memory operand ----
        if constexpr (CONVERT) {
            static_assert(TMEM_OP, "every converted layout routes one operand through tensor memory");
            const int t = threadIdx.x - 64;  // 0..127
            const int r = 32 * (warp & 3) + lane;  // the tensor-memory lane this thread writes
            int g = 0, transposes = 0;
            bool ok = true;
            for (long long tl = blockIdx.x; ok && tl < total_items; tl += gridDim.x) {
                for (int kb = 0; kb < KT; ++kb, ++g) {
                    const int s = g % S, round = g / S;
                    ok = mbar_wait(full_bar(s), round & 1, err, ERR_SPLIT_WAIT, lim);
                    if (!ok) break;
                    // The tensor-memory operand (this stage's columns are free: the copy
                    // that just landed was issued only after the MMAs of the stage's
                    // previous round had completed) ...
                    const uint32_t t_hi = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + ACC_COLS +
                                          (uint32_t)s * OP_COLS;
                    if constexpr (B_VIA_TMEM)
                        mnmajor_to_tmem<THREE>(smem + b_off(s), r, t_hi, t_hi + 32u);
                    else if constexpr (A_K)
                        kmajor_to_tmem<THREE>(smem + a_off(s), r, t_hi, t_hi + 32u);
                    else
                        mnmajor_to_tmem<THREE>(smem + a_off(s), r, t_hi, t_hi + 32u);
                    // ... and the shared-memory operand: split, or transpose (and split).
                    if constexpr (B_VIA_TMEM) {
                        if constexpr (THREE)
                            split_kmajor(reinterpret_cast<float4 *>(smem + a_off(s)),
                                         reinterpret_cast<float4 *>(smem + lo_off(s)), t);
                    } else if constexpr (!B_K) {
                        ok = transpose_mnmajor<THREE>(smem + b_off(s), smem + lo_off(s), t,
                                                      read_bar, transposes & 1, err, lim);
                        ++transposes;
                        if (!ok) break;
                    } else if constexpr (THREE) {
                        split_kmajor(reinterpret_cast<float4 *>(smem + b_off(s)),
                                     reinterpret_cast<float4 *>(smem + lo_off(s)), t);
                    }
                    // Generic-proxy writes must be visible to the tensor core (async
                    // proxy); tensor-memory stores are ordered by the tcgen05 fence.
                    if constexpr (THREE || !B_K)
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    tc_fence_before();
                    mbar_arrive(split_bar(s));
                }
            }
        }
    } else {
        // ---- epilogue warps (6..9, or 2..9): tile j while tile j + 1 is multiplied ----
        // Warp w reads accumulator lanes 32*(w%4) .. +31 (rows of the tile) and columns
        // [c_first, c_first + EPI_COLS).
        const int q = warp & 3;
        const int ew = warp - (CONVERT ? 6 : 2);  // 0 .. EPI_WARPS-1
        const int c_first = (ew / 4) * EPI_COLS;
        const uint32_t stage0 = sbase + (uint32_t)(L::EPI_OFFSET + ew * EPI_BUFS * 4096);
        uint8_t *const ebuf = smem + L::EPI_OFFSET + ew * EPI_BUFS * 4096;
        int j = 0;
        for (long long t = blockIdx.x; t < total_items; t += gridDim.x, ++j) {
            int m0, n0, bz;
            bool narrow;
            item_coords(t, m0, n0, bz, narrow);
            const int c_end = narrow ? MMA_M : MMA_N;  // accumulator columns of this item
            const int acc = j % NACC, use = j / NACC;
            if (!mbar_wait(acc_full_bar(acc), use & 1, err, ERR_EPILOGUE, lim)) break;
            tc_fence_after();
            const uint32_t src = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * MMA_N);
            if constexpr (TRANS_OUT) {
                // D = C^T: this thread holds column n of C, rows m0 + c0 + i.
                const int n = n0 + q * 32 + lane;
                const float bn = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.0f;
                if (p.c_tma) {
                    // Stage 32 rows x 32 columns of C (row i: 128 bytes, 16-byte chunk index
                    // XOR i % 8; lane = column, so each row's stores hit 32 banks) and write
                    // them with one TMA store, as in the untransposed case.
#pragma unroll 1
                    for (int c0 = c_first; c0 < c_first + EPI_COLS && c0 < c_end; c0 += 32) {
                        const int buf = EPI_BUFS == 2 ? (c0 >> 5) & 1 : 0;
                        if (lane == 0) {
                            if constexpr (EPI_BUFS == 2)
                                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                            else
                                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                        }
                        __syncwarp();
                        uint32_t r[32];
                        tmem_ld_32cols(src + (uint32_t)c0, r);
                        uint8_t *const cbuf = ebuf + buf * 4096;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float o = p.alpha * __uint_as_float(r[i]) + bn;
                            if (p.relu) o = fmaxf(o, 0.0f);
                            *reinterpret_cast<float *>(cbuf + i * 128 +
                                                       ((((lane >> 2) ^ (i & 7)) << 4) | ((lane & 3) << 2))) = o;
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0 && n0 + q * 32 < p.N && m0 + c0 < p.M)
                            tma_store_3d(&p.tmC, stage0 + (uint32_t)buf * 4096u, n0 + q * 32, m0 + c0, bz);
                    }
                } else {
                    float *const C = p.C + (long long)bz * p.strideC;
#pragma unroll 1
                    for (int c0 = c_first; c0 < c_first + EPI_COLS && c0 < c_end; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld_32cols(src + (uint32_t)c0, r);
                        if (n < p.N) {
#pragma unroll 4
                            for (int i = 0; i < 32; ++i) {
                                const int m = m0 + c0 + i;
                                if (m >= p.M) break;
                                float *const cp = C + (long long)m * p.ldc + n;
                                float o = p.alpha * __uint_as_float(r[i]);
                                if (p.beta != 0.0f) o = fmaf(p.beta, *cp, o);
                                o += bn;
                                if (p.relu) o = fmaxf(o, 0.0f);
                                *cp = o;
                            }
                        }
                    }
                }
            } else {
                const int row = m0 + q * 32 + lane;
                if (p.c_tma) {
                    // beta == 0: alpha, bias, ReLU in registers; each 32 x 32 chunk is staged in
                    // shared memory (128-byte swizzle: lane = row, 16-byte chunk index XOR
                    // row % 8, conflict-free) and written by one TMA store, which clips the
                    // rows and columns outside C.  Two buffers per warp.
#pragma unroll 1
                    for (int c0 = c_first; c0 < c_first + EPI_COLS && c0 < c_end; c0 += 32) {
                        const int buf = EPI_BUFS == 2 ? (c0 >> 5) & 1 : 0;
                        // the store that last read this buffer must have finished reading it
                        if (lane == 0) {
                            if constexpr (EPI_BUFS == 2)
                                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                            else
                                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                        }
                        __syncwarp();
                        uint32_t r[32];
                        tmem_ld_32cols(src + (uint32_t)c0, r);
                        uint8_t *const rowbuf = ebuf + buf * 4096 + lane * 128;
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            float v[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int gc = n0 + c0 + 4 * g + e;
                                float o = p.alpha * __uint_as_float(r[4 * g + e]);
                                if (p.bias && gc < p.N) o += __ldg(p.bias + gc);
                                if (p.relu) o = fmaxf(o, 0.0f);
                                v[e] = o;
                            }
                            *reinterpret_cast<float4 *>(rowbuf + ((g ^ (lane & 7)) << 4)) =
                                make_float4(v[0], v[1], v[2], v[3]);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        // (a chunk entirely outside C is not stored at all)
                        if (lane == 0 && n0 + c0 < p.N && m0 + q * 32 < p.M)
                            tma_store_3d(&p.tmC, stage0 + (uint32_t)buf * 4096u, n0 + c0, m0 + q * 32, bz);
                    }
                } else {
                    float *const C = p.C + (long long)bz * p.strideC;
#pragma unroll 1
                    for (int c0 = c_first; c0 < c_first + EPI_COLS && c0 < c_end; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld_32cols(src + (uint32_t)c0, r);
                        if (row < p.M) {
                            float *const crow = C + (long long)row * p.ldc;
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const int gc = n0 + c0 + 4 * g;
                                float v[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) v[e] = p.alpha * __uint_as_float(r[4 * g + e]);
                                if (p.c_vec && gc + 3 < p.N) {
                                    if (p.beta != 0.0f) {
                                        const float4 c = *reinterpret_cast<const float4 *>(crow + gc);
                                        v[0] = fmaf(p.beta, c.x, v[0]);
                                        v[1] = fmaf(p.beta, c.y, v[1]);
                                        v[2] = fmaf(p.beta, c.z, v[2]);
                                        v[3] = fmaf(p.beta, c.w, v[3]);
                                    }
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        if (p.bias) v[e] += __ldg(p.bias + gc + e);
                                        if (p.relu) v[e] = fmaxf(v[e], 0.0f);
                                    }
                                    *reinterpret_cast<float4 *>(crow + gc) =
                                        make_float4(v[0], v[1], v[2], v[3]);
                                } else {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        if (gc + e >= p.N) break;
                                        float o = v[e];
                                        if (p.beta != 0.0f) o = fmaf(p.beta, crow[gc + e], o);
                                        if (p.bias) o += __ldg(p.bias + gc + e);
                                        if (p.relu) o = fmaxf(o, 0.0f);
                                        crow[gc + e] = o;
                                    }
                                }
                            }
                        }
                    }
                }
            }
            // Hand the accumulator back: all of this warp's tensor-memory reads are done.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_bar(acc));
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }

    // Teardown: the allocating warp frees the tensor memory once every thread is done.
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace tc
}  // namespace fgemm
