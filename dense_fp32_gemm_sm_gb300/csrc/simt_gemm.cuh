// simt_gemm.cuh -- register-blocked FP32 GEMM on the CUDA cores of sm_103a.
//
// One CTA computes a BM x BN tile of C = alpha*op(A)*op(B) + beta*C (then bias,
// ReLU).  Design, GB300-first:
//
//  * Staging (global -> shared): a STAGES-deep ring of shared tiles filled with
//    cp.async, replacing the two-buffer, register-staged ping-pong of
//    GPU架构下的矩阵乘法深入优化, "5. warp tiling + double buffer".  Both operands
//    are stored k-major in shared memory: sA[k][m] and sB[k][n].  An operand
//    whose rows already run along m (A stored K x M) or n (B stored K x N) is
//    copied with 16-byte vectors; an operand stored with k contiguous is
//    transposed by the copy itself (4-byte cp.async, one element per lane, a
//    warp covering 8 k x 4 rows: the global reads are whole 32-byte sectors and
//    the 32 shared addresses fall in 32 distinct banks; ncu nevertheless counts
//    about five shared wavefronts per such copy instruction, about one per
//    sector read, where a 16-byte copy of a row takes one per 128 bytes).
//    Out-of-range rows/columns and the K tail are zero-filled by the copy
//    (src-size 0), so the inner loop has no edge checks.
//
//  * k-major tiles let every thread read its A and B fragments for one k with
//    16-byte loads along m and n (the transposed-A idea of the same page, and the
//    row padding of GEMM 优化详解, "Level 3" / 第5章-基础Kernel, "Shared + Padding").
//    Fragments for k+1 are loaded while k is computed (register double buffer).
//    The lanes of a warp form 2 x 2 quads of the warp's lane grid, so both
//    fragment loads take 2 shared-memory wavefronts (see lane_coords).
//
//  * Register blocking (GEMM 优化详解, "Level 5: Register Blocking"): each thread
//    owns TM x TN accumulators (8 x 8), held as pairs along n and updated with the
//    packed FP32 FMA of sm_100+ (__ffma2_rn): one instruction does two FMAs, so
//    the FMA pipe stays busy while the issue slots left over carry the shared
//    loads.  Each a[i] is paired with itself once per k.
//
//  * Epilogue in registers (GEMM 优化详解, "Level 6: Kernel Fusion" and "Level 7:
//    Vectorized Loads"): v = alpha*acc (+ beta*C) (+ bias[col]) (+ row_bias[row]),
//    ReLU, then float4 stores when C is 16-byte aligned, scalar stores otherwise.
//
//  * K-groups (KS > 1, for the smallest grids): several warp groups split each
//    stage's k and add their sums through shared memory before the epilogue.
//
//  * Tiles are visited in groups of GROUP_M (16) tile-rows so that concurrently
//    resident CTAs share panels of A and B in L2.
//
//  * Last-wave split (TILE_QUARTER launches): with two CTAs per SM an SM retires
//    tile-pairs at the same rate as lone tiles, so a grid whose tile count leaves a
//    remainder r = tiles mod SMs spends a whole extra lone-tile period on those r
//    tiles while the other SMs idle.  A split launch runs the first tiles whole and
//    then cuts each of the last r into four quarter tiles with four k-groups each,
//    so the remainder's work spreads over the SMs in quarter-tile steps.
//
//  * Last-wave k-split (TILE_KSPLIT launches): the last r tiles stay whole, each
//    computed by a thread-block cluster of four CTAs that multiply one k-slice each;
//    the partial tiles are added in slice order through distributed shared memory
//    (no workspace, no atomics, the same result on every run).
//
//  * Last-wave k-chain (TILE_KCHAIN launches): the last r tiles stay whole, each in
//    two to eight k-slices (as many as the launch-time model finds fastest), one
//    launch per slice; each launch adds its slice's products into C in slice order,
//    the later ones as programmatic dependent launches that run alongside the earlier
//    ones and wait for them only before adding into C.
//
//  * The copy of a later stage is issued at k-step COPY_K of the current stage.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fgemm {

struct GemmParams {
    const float *A;
    const float *B;
    float *C;
    const float *bias;      // one value per column (length N), or null
    const float *row_bias;  // one value per row (length M), or null
    long long lda, ldb, ldc;
    long long strideA, strideB, strideC;
    int M, N, K;  // K is 0 when no products are formed (K == 0 or alpha == 0)
    float alpha, beta;
    int relu;
    int tiles_m, tiles_n;
    int c_vec;  // C pointer, ldc and strideC allow 16-byte accesses
    // Last-wave split: the tiles of the linear tile order (all problems of the
    // batch, problem-major) before full_units run whole, the rest as quarter tiles.
    int full_units;
};

// ---- PTX helpers ---------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; bytes [src_bytes, 16) of the destination are zeroed.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 4-byte global->shared copy; src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Thread-block cluster helpers (sm_90+): this CTA's rank, a cluster-wide barrier
// with release/acquire ordering of shared-memory writes, and a 16-byte load from
// the shared memory of CTA `rank` at the address a local variable has there.
__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local_addr, unsigned rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ int clamp_bytes(long long remaining_elems)
{
    return remaining_elems >= 4 ? 16 : (remaining_elems > 0 ? int(remaining_elems) * 4 : 0);
}

// d += a * b on two packed FP32 lanes: the sm_100+ packed FMA (round-to-nearest, no
// flush), through the compiler's builtin so that it schedules the packed FMAs itself.
__device__ __forceinline__ void ffma2(float2 &d, float2 a, float2 b) { d = __ffma2_rn(a, b, d); }

// ---- Configuration -------------------------------------------------------------

template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_, int STAGES_, int MINB_,
          int TA_, int TB_, bool VEC_, int KS_ = 1, bool FASTCOPY_ = true>
struct SimtCfg {
    // Interior stages issue their copies without per-copy bounds predicates.
    static constexpr bool FASTCOPY = FASTCOPY_;
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
    static constexpr int STAGES = STAGES_, MINB = MINB_;
    static constexpr int TA = TA_, TB = TB_;
    static constexpr bool VEC = VEC_;
    // KS groups of warps share the CTA tile: group g multiplies k-columns
    // [g*KB, (g+1)*KB) of every stage into its own accumulators, and the groups'
    // sums are added through shared memory before the epilogue.  More warps per
    // tile, fewer serial k-steps per thread: for problems with too few tiles to
    // keep every SM busy.
    static constexpr int KS = KS_;
    static constexpr int KB = BK / KS;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int GROUP_THREADS = 32 * WARPS_M * WARPS_N;
    static constexpr int THREADS = GROUP_THREADS * KS;
    static constexpr int LR = WM / TM;  // lanes along M
    static constexpr int LC = WN / TN;  // lanes along N
    static constexpr int A_LD = BM + 4;  // sA[k][m]; +4 floats keeps transposed writes conflict-free
    static constexpr int B_LD = BN + 4;  // sB[k][n]
    static constexpr int A_STAGE = BK * A_LD;
    static constexpr int B_STAGE = BK * B_LD;
    static constexpr int STAGE_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int RED_BYTES = (KS - 1) * GROUP_THREADS * TM * TN * 4;
    static constexpr int SMEM_BYTES = STAGE_BYTES > RED_BYTES ? STAGE_BYTES : RED_BYTES;
    // Tile-rows per group of the grouped tile order.  Measured on GB300 (ncu DRAM bytes,
    // one call, L2 flushed by the profiler): FC 8192 x 4096 x 11008 reads 1.73 GB with 8,
    // 1.13 GB with 16, 1.32 / 1.48 / 2.57 GB with 20 / 24 / 32 (larger groups no longer
    // keep their rows of A in L2 while the columns stream past); 4096^3 reads 0.35 GB
    // with 8 and 0.30 GB with 16.  The time is the same within 0.1 % for all of them.
    static constexpr int GROUP_M = 16;
    // k-step of each stage at which the copy of a later stage is issued.  NN tiles of
    // 128 rows: halfway through the stage, away from the barrier where every warp also
    // reloads its fragments (measured about 1 % faster at 4096^3, on the FC and PV
    // workloads and at 2048^3).  Otherwise right after the barrier: NT measured 8 %
    // faster so on QK^T, TN and TT spill registers with the later copy, and the small
    // tiles lose latency hiding (256^3 on 32 x 32 tiles: 11 against 13 us).  At most
    // KB - 2: the slot written is the one freed by the previous stage's barrier, and
    // the slot index advances at KB - 1.
    static constexpr int COPY_K = (TA == 0 && TB == 0 && BM >= 128) ? KB / 2 : 0;
    static_assert(COPY_K <= KB - 2, "the copy is issued before the slot index advances");

    static_assert(BK % KS == 0 && KB % 2 == 0, "each k-group takes an even number of k per stage");
    static_assert(LR * LC == 32, "a warp is LR x LC lanes");
    static_assert(LR % 2 == 0 && LC % 2 == 0, "lane quads are 2 x 2");
    static_assert(BM % WM == 0 && BN % WN == 0, "warp tiles must cover the CTA tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "16-byte fragments");
    static_assert(BK % 8 == 0, "transposing copies move 8 k per warp row");
    static_assert(BM % 4 == 0 && BN % 4 == 0, "transposing copies move 4 rows per warp");
    static_assert((BM * BK) % THREADS == 0 && (BN * BK) % THREADS == 0,
                  "element copies divide evenly over the threads");
    static_assert((BM * BK / 4) % THREADS == 0 && (BN * BK / 4) % THREADS == 0,
                  "vector copies divide evenly over the threads");
    static_assert(STAGES >= 2, "at least double buffering");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// ---- Tile loaders --------------------------------------------------------------
//
// Each loader is set up once per tile (base pointer, edge masks) and then issues
// one stage per call, advancing its pointer by BK along k.  Elements outside the
// matrix are zero-filled (src-size 0, with an in-bounds dummy address).

// Stored block whose rows run along k (K x MN storage, MN contiguous): rows
// [k0, k0+BK) x columns [c0, c0+COLS) -> s[k][c] with row stride S_LD.  Thread t
// always copies the same column chunk, in rows r_base + it * RSTEP.
template <int BK, int COLS, int S_LD, int THREADS, bool VEC, bool FAST>
struct KRowsCopy {
    static constexpr int W = VEC ? 4 : 1;          // elements per copy
    static constexpr int CPR = COLS / W;           // copies per row
    static constexpr int RSTEP = THREADS / CPR;    // rows between a thread's copies
    static constexpr int ITERS = BK / RSTEP;
    static_assert(THREADS % CPR == 0 && BK % RSTEP == 0, "copies divide evenly over the threads");

    const float *p;  // this thread's element in row (k0 + r_base) of the next stage
    int bytes_c;     // bytes of the chunk inside the matrix along the columns (0 .. 4*W)
    int r_base;

    __device__ __forceinline__ void init(const float *g, long long ld, int c0, int Ccount, int tid)
    {
        r_base = tid / CPR;
        const int c = c0 + (tid % CPR) * W;
        bytes_c = VEC ? clamp_bytes((long long)Ccount - c) : (c < Ccount ? 4 : 0);
        p = g + (long long)r_base * ld + c;
    }

    __device__ __forceinline__ void issue(uint32_t s_tile, const float *g, long long ld, int k0,
                                          int K, int tid)
    {
        const uint32_t s0 = s_tile + (r_base * S_LD + (tid % CPR) * W) * 4;
        if (FAST && k0 + BK <= K && bytes_c == 4 * W) {
            // Every copy of this stage is inside the matrix: no per-copy predicates.
#pragma unroll
            for (int it = 0; it < ITERS; ++it) {
                if constexpr (VEC)
                    cp_async_16(s0 + it * RSTEP * S_LD * 4, p + (long long)(it * RSTEP) * ld, 16);
                else
                    cp_async_4(s0 + it * RSTEP * S_LD * 4, p + (long long)(it * RSTEP) * ld, 4);
            }
            p += (long long)BK * ld;
            return;
        }
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const bool ok = k0 + r_base + it * RSTEP < K && bytes_c > 0;
            const float *src = ok ? p + (long long)(it * RSTEP) * ld : g;
            if constexpr (VEC)
                cp_async_16(s0 + it * RSTEP * S_LD * 4, src, ok ? bytes_c : 0);
            else
                cp_async_4(s0 + it * RSTEP * S_LD * 4, src, ok ? 4 : 0);
        }
        p += (long long)BK * ld;
    }
};

// Stored block whose rows run along m (or n) with k contiguous (MN x K storage):
// rows [r0, r0+ROWS) x k [k0, k0+BK) -> s[k][r] (a transpose).  Each warp moves
// 8 (k) x 4 (rows) patches: lane&7 picks k, lane>>3 picks the row, so a warp reads
// four full 32-byte sectors and writes 32 distinct banks (measured: about five
// shared wavefronts per instruction all the same, see the file header).  A thread
// keeps one k and copies rows r_base + it * RSTEP.
template <int BK, int ROWS, int S_LD, int THREADS, bool FAST>
struct KColsCopy {
    static constexpr int WARPS = THREADS / 32;
    static constexpr int PATCHES_K = BK / 8;
    static constexpr int RSTEP = 4 * WARPS / PATCHES_K;
    static constexpr int ITERS = ROWS / RSTEP;
    static_assert(WARPS % PATCHES_K == 0 && ROWS % RSTEP == 0 && ITERS <= 32,
                  "patches divide evenly over the warps");

    static constexpr unsigned kFullMask = ITERS == 32 ? 0xFFFFFFFFu : (1u << ITERS) - 1u;
    const float *p;  // this thread's element (row r0 + r_base, column k_local) of the next stage
    unsigned rmask;  // bit it: row r0 + r_base + it * RSTEP is inside the matrix

    __device__ __forceinline__ static int k_local(int tid) { return ((tid >> 5) % PATCHES_K) * 8 + (tid & 7); }
    __device__ __forceinline__ static int r_base(int tid)
    {
        return ((tid >> 5) / PATCHES_K) * 4 + ((tid & 31) >> 3);
    }

    __device__ __forceinline__ void init(const float *g, long long ld, int r0, int R, int tid)
    {
        const int rb = r0 + r_base(tid);
        rmask = 0;
#pragma unroll
        for (int it = 0; it < ITERS; ++it)
            if (rb + it * RSTEP < R) rmask |= 1u << it;
        p = g + (long long)rb * ld + k_local(tid);
    }

    __device__ __forceinline__ void issue(uint32_t s_tile, const float *g, long long ld, int k0,
                                          int K, int tid)
    {
        const uint32_t s0 = s_tile + (k_local(tid) * S_LD + r_base(tid)) * 4;
        if (FAST && k0 + BK <= K && rmask == kFullMask) {
            // Every copy of this stage is inside the matrix: no per-copy predicates.
#pragma unroll
            for (int it = 0; it < ITERS; ++it)
                cp_async_4(s0 + it * RSTEP * 4, p + (long long)(it * RSTEP) * ld, 4);
            p += BK;
            return;
        }
        const bool kok = k0 + k_local(tid) < K;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const bool ok = kok && ((rmask >> it) & 1u);
            cp_async_4(s0 + it * RSTEP * 4, ok ? p + (long long)(it * RSTEP) * ld : g, ok ? 4 : 0);
        }
        p += BK;
    }
};

// The two loaders of a configuration: A into sA[k][m], B into sB[k][n].
template <class Cfg>
struct StageCopy {
    using ACopy = typename std::conditional<
        Cfg::TA == 1, KRowsCopy<Cfg::BK, Cfg::BM, Cfg::A_LD, Cfg::THREADS, Cfg::VEC, Cfg::FASTCOPY>,
        KColsCopy<Cfg::BK, Cfg::BM, Cfg::A_LD, Cfg::THREADS, Cfg::FASTCOPY>>::type;
    using BCopy = typename std::conditional<
        Cfg::TB == 0, KRowsCopy<Cfg::BK, Cfg::BN, Cfg::B_LD, Cfg::THREADS, Cfg::VEC, Cfg::FASTCOPY>,
        KColsCopy<Cfg::BK, Cfg::BN, Cfg::B_LD, Cfg::THREADS, Cfg::FASTCOPY>>::type;
    ACopy a;
    BCopy b;

    __device__ __forceinline__ void init(const GemmParams &p, const float *A, const float *B, int m0,
                                         int n0, int tid)
    {
        if constexpr (Cfg::TA == 1)
            a.init(A, p.lda, m0, p.M, tid);
        else
            a.init(A, p.lda, m0, p.M, tid);
        if constexpr (Cfg::TB == 0)
            b.init(B, p.ldb, n0, p.N, tid);
        else
            b.init(B, p.ldb, n0, p.N, tid);
    }

    __device__ __forceinline__ void issue(uint32_t sA, uint32_t sB, const GemmParams &p,
                                          const float *A, const float *B, int k0, int K, int tid)
    {
        a.issue(sA, A, p.lda, k0, K, tid);
        b.issue(sB, B, p.ldb, k0, K, tid);
    }
};

// Row (within the CTA tile) of the thread's i-th accumulator row, and column of
// its j-th accumulator column: groups of 4 consecutive rows/columns, one 16-byte
// fragment load each.
// Lane -> (lr, lc) position in the warp's LR x LC lane grid.  Every 4 consecutive
// lanes form a 2 x 2 block (bit 0 picks the column, bit 1 the row).  Measured on
// GB300: a warp-wide 16-byte shared load costs 2 wavefronts when each group of 4
// consecutive lanes reads at most 2 distinct 16-byte chunks, and 4 otherwise.  The A
// fragment address depends on lr only and the B fragment address on lc only, so with
// 2 x 2 quads both loads take 2 wavefronts (8 per k-step for 8 x 8 per thread); a
// row-major lane order (quads along one row) makes the B loads take 4 (12 per k).
template <class Cfg>
__device__ __forceinline__ void lane_coords(int lane, int &lr, int &lc)
{
    constexpr int HC = Cfg::LC / 2;  // 2 x 2 quads across the lane grid's columns
    const int quad = lane >> 2;
    lc = (lane & 1) + 2 * (quad % HC);
    lr = ((lane >> 1) & 1) + 2 * (quad / HC);
}

template <class Cfg>
__device__ __forceinline__ int frag_row(int wm0, int lr, int i)
{
    return wm0 + (i / 4) * (Cfg::LR * 4) + lr * 4 + (i % 4);
}

template <class Cfg>
__device__ __forceinline__ int frag_col(int wn0, int lc, int j)
{
    return wn0 + (j / 4) * (Cfg::LC * 4) + lc * 4 + (j % 4);
}

// ---- The kernel ----------------------------------------------------------------

// How a CTA finds its tile.
enum TileMap {
    // blockIdx.x walks the grouped tile order of problem blockIdx.z.
    TILE_GRID = 0,
    // One-dimensional grid: CTA t takes tile t of the linear tile order (problem-
    // major, each problem in grouped order); the whole tiles of a split batch.
    TILE_LINEAR = 1,
    // One-dimensional grid: CTA 4 t' + q takes quarter q (row half q / 2, column
    // half q % 2) of Parent-sized tile full_units + t' of the linear tile order;
    // quarters wholly outside C do nothing.
    TILE_QUARTER = 2,
    // One-dimensional grid in clusters of KSPLIT CTAs: the CTAs of cluster t' each
    // multiply one k-slice of tile full_units + t' of the linear tile order, then
    // add their partial sums through distributed shared memory in slice order and
    // write the tile, a 1/KSPLIT band of rows each.
    TILE_KSPLIT = 3,
    // One-dimensional grid, one launch per k-slice (argument `chain` = slice | slices
    // << 8): CTA t multiplies that k-slice of tile full_units + t of the linear tile
    // order.  The slices of a tile are added in C itself, in slice order: slice 0
    // writes alpha * P_0 (+ beta * C), slice s > 0 waits for the launch of slice s - 1
    // to complete (griddepcontrol.wait: programmatic dependent launch), adds alpha * P_s
    // to what is in C and writes it back, and the last slice applies bias and ReLU.
    // Each launch (and the whole-tile launch before slice 0) lets the next one start as
    // soon as all of its CTAs are running (griddepcontrol.launch_dependents), so the
    // slices' products overlap the launches before them and only the additions into C
    // are ordered.
    TILE_KCHAIN = 4,
};
constexpr int KSPLIT = 4;

// griddepcontrol (programmatic dependent launch, sm_90+): let the next kernel of the
// stream start launching; wait until the preceding kernel has completed and its
// memory operations are visible.  Both are no-ops without a programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_prerequisite()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// MAP and Parent select the tile of each CTA; the body is the same for every map.
// (Moving the body into a function called from three kernels measured 1 % slower
// at 4096^3, so the maps live here as compile-time branches.)
template <class Cfg, int MAP = TILE_GRID, class Parent = Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
    simt_gemm_kernel(const GemmParams p, int chain = 0)
{
    // Let a programmatic dependent launch of this call (the k-chain slices after the
    // whole tiles, each slice after the one before) start as soon as every CTA of this
    // launch is running.  Without such a dependent this does nothing.
    if constexpr (MAP == TILE_KCHAIN || MAP == TILE_GRID || MAP == TILE_LINEAR)
        pdl_launch_dependents();
    extern __shared__ __align__(128) float smem[];
    float *const sA_all = smem;
    float *const sB_all = smem + Cfg::STAGES * Cfg::A_STAGE;
    constexpr int TM = Cfg::TM, TN = Cfg::TN;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int kg = warp / (Cfg::WARPS_M * Cfg::WARPS_N);  // k-group of this warp
    const int wg = warp % (Cfg::WARPS_M * Cfg::WARPS_N);  // warp within its group
    int lr, lc;
    lane_coords<Cfg>(lane, lr, lc);
    const int wm0 = (wg / Cfg::WARPS_N) * Cfg::WM, wn0 = (wg % Cfg::WARPS_N) * Cfg::WN;
    const int kb0 = kg * Cfg::KB;  // first k of a stage this group multiplies

    // Grouped tile order: GROUP_M consecutive tile-rows are swept column by column.
    int tile_m, tile_n;
    int m0, n0;
    long long bz;
    if constexpr (MAP == TILE_GRID) {
        const int pid = blockIdx.x;
        const int per_group = Cfg::GROUP_M * p.tiles_n;
        const int group = pid / per_group;
        const int first_m = group * Cfg::GROUP_M;
        const int rows_in_group = min(p.tiles_m - first_m, Cfg::GROUP_M);
        const int in_group = pid - group * per_group;
        tile_m = first_m + in_group % rows_in_group;
        tile_n = in_group / rows_in_group;
        m0 = tile_m * Cfg::BM;
        n0 = tile_n * Cfg::BN;
        bz = blockIdx.z;
    } else {
        static_assert(MAP != TILE_QUARTER || (Parent::BM == 2 * Cfg::BM && Parent::BN == 2 * Cfg::BN),
                      "a quarter CTA computes one quarter of a parent tile");
        const long long tiles = (long long)p.tiles_m * p.tiles_n;
        const long long t = MAP == TILE_LINEAR ? (long long)blockIdx.x
                            : MAP == TILE_KCHAIN ? (long long)p.full_units + blockIdx.x
                                                 : (long long)p.full_units + (blockIdx.x >> 2);
        static_assert(MAP != TILE_KSPLIT || KSPLIT == 4, "k-slice CTAs are numbered 4 t' + slice");
        bz = t / tiles;
        const int pid = (int)(t - bz * tiles);
        const int per_group = Parent::GROUP_M * p.tiles_n;
        const int group = pid / per_group;
        const int first_m = group * Parent::GROUP_M;
        const int rows_in_group = min(p.tiles_m - first_m, Parent::GROUP_M);
        const int in_group = pid - group * per_group;
        tile_m = first_m + in_group % rows_in_group;
        tile_n = in_group / rows_in_group;
        m0 = tile_m * Parent::BM;
        n0 = tile_n * Parent::BN;
        if constexpr (MAP == TILE_QUARTER) {
            const int q = blockIdx.x & 3;
            m0 += (q >> 1) * Cfg::BM;
            n0 += (q & 1) * Cfg::BN;
            if (m0 >= p.M || n0 >= p.N) return;  // the same for the whole CTA
        }
    }
    // k range of this CTA: all of K, or one k-slice (whole stages) of a k-split tile.
    int k_len = p.K;
    long long a_koff = 0, b_koff = 0;
    if constexpr (MAP == TILE_KSPLIT || MAP == TILE_KCHAIN) {
        const int slice = MAP == TILE_KSPLIT ? (int)cluster_rank() : (chain & 0xFF);
        const int slices = MAP == TILE_KSPLIT ? KSPLIT : (chain >> 8);
        const int per = ((p.K + slices - 1) / slices + Cfg::BK - 1) / Cfg::BK * Cfg::BK;
        const int kb = min(p.K, slice * per);
        k_len = min(p.K - kb, per);
        a_koff = Cfg::TA ? (long long)kb * p.lda : kb;
        b_koff = Cfg::TB ? kb : (long long)kb * p.ldb;
    }
    const float *const A = p.A + bz * p.strideA + a_koff;
    const float *const B = p.B + bz * p.strideB + b_koff;
    // The quarter tiles form their C pointer after the main loop (measured: it frees
    // the 24 B of spill space the TN instance needed); the other maps here.
    float *const C_early = MAP == TILE_QUARTER ? nullptr : p.C + bz * p.strideC;

    float2 acc[TM][TN / 2];  // acc[i][j] = (c[i][2j], c[i][2j+1])
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    const uint32_t sA_base = smem_addr(sA_all), sB_base = smem_addr(sB_all);
    const int KT = (k_len + Cfg::BK - 1) / Cfg::BK;

    if (KT > 0) {
        StageCopy<Cfg> copy;
        copy.init(p, A, B, m0, n0, tid);
        // Prologue: fill STAGES-1 slots, then wait for the first.
#pragma unroll
        for (int s = 0; s < Cfg::STAGES - 1; ++s) {
            if (s < KT)
                copy.issue(sA_base + s * Cfg::A_STAGE * 4, sB_base + s * Cfg::B_STAGE * 4, p, A, B,
                           s * Cfg::BK, k_len, tid);
            cp_async_commit();
        }
        cp_async_wait<Cfg::STAGES - 2>();
        __syncthreads();

        float4 fa[2][TM / 4], fb[2][TN / 4];
        auto load_frag = [&](int buf, int slot, int k) {
            const float *a = sA_all + slot * Cfg::A_STAGE + k * Cfg::A_LD;
            const float *b = sB_all + slot * Cfg::B_STAGE + k * Cfg::B_LD;
#pragma unroll
            for (int g = 0; g < TM / 4; ++g)
                fa[buf][g] = *reinterpret_cast<const float4 *>(a + frag_row<Cfg>(wm0, lr, 4 * g));
#pragma unroll
            for (int g = 0; g < TN / 4; ++g)
                fb[buf][g] = *reinterpret_cast<const float4 *>(b + frag_col<Cfg>(wn0, lc, 4 * g));
        };
        load_frag(0, 0, kb0);

        int slot = 0;
        for (int kt = 0; kt < KT; ++kt) {
#pragma unroll
            for (int k = 0; k < Cfg::KB; ++k) {
                const int cur = k & 1;
                if (k == Cfg::KB - 1) {
                    // Stage kt+1 must have landed, and every thread must be done with
                    // the slot the next copy overwrites.
                    cp_async_wait<Cfg::STAGES - 2>();
                    __syncthreads();
                    slot = (slot + 1 == Cfg::STAGES) ? 0 : slot + 1;
                    if (kt + 1 < KT) load_frag(cur ^ 1, slot, kb0);
                } else {
                    load_frag(cur ^ 1, slot, kb0 + k + 1);
                }
                if (k == Cfg::COPY_K) {
                    const int nk = kt + Cfg::STAGES - 1;
                    if (nk < KT) {
                        int ws = slot + Cfg::STAGES - 1;
                        if (ws >= Cfg::STAGES) ws -= Cfg::STAGES;
                        copy.issue(sA_base + ws * Cfg::A_STAGE * 4, sB_base + ws * Cfg::B_STAGE * 4,
                                   p, A, B, nk * Cfg::BK, k_len, tid);
                    }
                    cp_async_commit();
                }
                // Duplicate all of a[] first, then sweep the b pairs: each duplicate is
                // produced well before its first use.
                const float *a = reinterpret_cast<const float *>(&fa[cur][0]);
                const float2 *b2 = reinterpret_cast<const float2 *>(&fb[cur][0]);
                float2 ad[TM];
#pragma unroll
                for (int i = 0; i < TM; ++i) ad[i] = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < TN / 2; ++j)
#pragma unroll
                    for (int i = 0; i < TM; ++i) ffma2(acc[i][j], ad[i], b2[j]);
            }
        }
        cp_async_wait<0>();
    }

    float *const C = MAP == TILE_QUARTER ? p.C + bz * p.strideC : C_early;

    // ---- K-groups: groups 1.. hand their sums to group 0 through shared memory
    // (the stage buffers are free once every warp has passed the barrier), in
    // group order, so the result does not depend on timing.
    if constexpr (Cfg::KS > 1) {
        if (KT > 0) {
            constexpr int E = TM * TN / 2;  // accumulator pairs per thread
            float2 *const red = reinterpret_cast<float2 *>(smem);
            const int gt = tid - kg * Cfg::GROUP_THREADS;
            __syncthreads();
            if (kg > 0) {
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN / 2; ++j)
                        red[((kg - 1) * E + i * (TN / 2) + j) * Cfg::GROUP_THREADS + gt] = acc[i][j];
            }
            __syncthreads();
            if (kg == 0) {
#pragma unroll
                for (int g = 1; g < Cfg::KS; ++g)
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int j = 0; j < TN / 2; ++j) {
                            const float2 r =
                                red[((g - 1) * E + i * (TN / 2) + j) * Cfg::GROUP_THREADS + gt];
                            acc[i][j] = make_float2(acc[i][j].x + r.x, acc[i][j].y + r.y);
                        }
            }
        }
        if (kg != 0) return;
    }

    // ---- k-split tiles: partial sums through distributed shared memory.  Every CTA
    // of the cluster stores its slice's sums in its own shared memory (the stage
    // buffers are free once every warp is past the barrier); after a cluster barrier
    // CTA `slice` adds the four partials of its band of rows in slice order, so the
    // result does not depend on timing, and applies the epilogue of the whole tile.
    if constexpr (MAP == TILE_KSPLIT) {
        constexpr int P_LD = Cfg::BN + 4;
        constexpr int BAND = Cfg::BM / KSPLIT;  // rows each CTA reduces and writes
        constexpr int C4 = Cfg::BN / 4;         // 16-byte chunks per row
        constexpr int ITER = BAND * C4 / Cfg::THREADS;
        static_assert(Cfg::KS == 1, "one k-group per slice");
        static_assert(Cfg::BM * P_LD * 4 <= Cfg::SMEM_BYTES, "the partial tile fits the stages");
        static_assert(Cfg::BM % KSPLIT == 0 && (BAND * C4) % Cfg::THREADS == 0,
                      "the bands divide over the threads");
        __syncthreads();
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = frag_row<Cfg>(wm0, lr, i);
#pragma unroll
            for (int g = 0; g < TN / 4; ++g)
                *reinterpret_cast<float4 *>(smem + r * P_LD + frag_col<Cfg>(wn0, lc, 4 * g)) =
                    make_float4(acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x,
                                acc[i][2 * g + 1].y);
        }
        cluster_sync();
        // This launch may have started while the call's whole tiles were finishing;
        // it completes only after them.
        pdl_wait_prerequisite();
        const int band0 = (int)cluster_rank() * BAND;
        const bool products = p.K > 0;
        const bool has_bias = p.bias != nullptr, has_row_bias = p.row_bias != nullptr;
        const uint32_t base = smem_addr(smem);
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int e = it * Cfg::THREADS + tid;
            const int r = band0 + e / C4, c = (e % C4) * 4;
            const uint32_t la = base + (uint32_t)(r * P_LD + c) * 4u;
            float4 sum = ld_cluster_f4(la, 0);
#pragma unroll
            for (unsigned q = 1; q < (unsigned)KSPLIT; ++q) {
                const float4 w = ld_cluster_f4(la, q);
                sum.x += w.x;
                sum.y += w.y;
                sum.z += w.z;
                sum.w += w.w;
            }
            const int gr = m0 + r, gc = n0 + c;
            if (gr >= p.M || gc >= p.N) continue;
            float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = products ? p.alpha * v[q] : 0.0f;
            float *const dst = C + (long long)gr * p.ldc + gc;
            const float rb = has_row_bias ? __ldg(p.row_bias + gr) : 0.0f;
            if (p.c_vec && gc + 3 < p.N) {
                if (p.beta != 0.0f) {
                    const float4 c0 = *reinterpret_cast<const float4 *>(dst);
                    v[0] = fmaf(p.beta, c0.x, v[0]);
                    v[1] = fmaf(p.beta, c0.y, v[1]);
                    v[2] = fmaf(p.beta, c0.z, v[2]);
                    v[3] = fmaf(p.beta, c0.w, v[3]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (has_bias) v[q] += __ldg(p.bias + gc + q);
                    if (has_row_bias) v[q] += rb;
                    if (p.relu) v[q] = fmaxf(v[q], 0.0f);
                }
                *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (gc + q >= p.N) break;
                    float o = v[q];
                    if (p.beta != 0.0f) o = fmaf(p.beta, dst[q], o);
                    if (has_bias) o += __ldg(p.bias + gc + q);
                    if (has_row_bias) o += rb;
                    if (p.relu) o = fmaxf(o, 0.0f);
                    dst[q] = o;
                }
            }
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
        return;
    }

    // ---- Epilogue: alpha, beta, bias, ReLU in registers; vector stores where possible.
    // (Quarter tiles may have started while the call's whole tiles were finishing;
    // they complete only after them.)
    if constexpr (MAP == TILE_QUARTER) pdl_wait_prerequisite();
    // k-chain slices: C holds the sum of the earlier slices once the launch before this
    // one is complete, so every slice waits for it here (slice 0 too: its products need
    // nothing from the whole tiles, but then every launch of the call has completed when
    // the last slice has).  Slice 0 weighs C's old value by beta; later slices add their
    // products to what C holds, read past L1 (.cg), which may hold lines an earlier slice
    // replaced; only the last slice applies bias and ReLU.
    bool last = true;
    float cw = p.beta;
    if constexpr (MAP == TILE_KCHAIN) {
        const int slice = chain & 0xFF;
        last = slice + 1 == (chain >> 8);
        if (slice != 0) cw = 1.0f;
        pdl_wait_prerequisite();
    }
    const bool products = KT > 0;
    const bool has_bias = last && p.bias != nullptr, has_row_bias = last && p.row_bias != nullptr;
    const bool relu = last && p.relu;
    float bias_v[TN];
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        const int gc = n0 + frag_col<Cfg>(wn0, lc, j);
        bias_v[j] = (has_bias && gc < p.N) ? __ldg(p.bias + gc) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gr = m0 + frag_row<Cfg>(wm0, lr, i);
        if (gr >= p.M) continue;
        float *const crow = C + (long long)gr * p.ldc;
        const float rb = has_row_bias ? __ldg(p.row_bias + gr) : 0.0f;
#pragma unroll
        for (int g = 0; g < TN / 4; ++g) {
            const int gc = n0 + frag_col<Cfg>(wn0, lc, 4 * g);
            float v[4] = {acc[i][2 * g].x, acc[i][2 * g].y, acc[i][2 * g + 1].x, acc[i][2 * g + 1].y};
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = products ? p.alpha * v[e] : 0.0f;
            float *const dst = crow + gc;
            if (p.c_vec && gc + 3 < p.N) {
                if (cw != 0.0f) {
                    const float4 c = MAP == TILE_KCHAIN
                                         ? __ldcg(reinterpret_cast<const float4 *>(dst))
                                         : *reinterpret_cast<const float4 *>(dst);
                    v[0] = fmaf(cw, c.x, v[0]);
                    v[1] = fmaf(cw, c.y, v[1]);
                    v[2] = fmaf(cw, c.z, v[2]);
                    v[3] = fmaf(cw, c.w, v[3]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (has_bias) v[e] += bias_v[4 * g + e];
                    if (has_row_bias) v[e] += rb;
                    if (relu) v[e] = fmaxf(v[e], 0.0f);
                }
                *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (gc + e >= p.N) break;
                    float o = v[e];
                    if (cw != 0.0f)
                        o = fmaf(cw, MAP == TILE_KCHAIN ? __ldcg(dst + e) : dst[e], o);
                    if (has_bias) o += bias_v[4 * g + e];
                    if (has_row_bias) o += rb;
                    if (relu) o = fmaxf(o, 0.0f);
                    dst[e] = o;
                }
            }
        }
    }
}

}  // namespace fgemm
