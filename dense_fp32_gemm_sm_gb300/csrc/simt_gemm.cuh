// simt_gemm.cuh -- register-blocked FP32 GEMM on the CUDA cores of sm_103a.
//
// One CTA computes a BM x BN tile of C = alpha*op(A)*op(B) + beta*C (then bias,
// ReLU).  Design, GB300-first:
//
//  * Staging (global -> shared): a STAGES-deep ring of shared-memory tiles filled
//    with cp.async (16-byte vectors, or single elements when the operand is not
//    16-byte aligned).  Out-of-range rows/columns and the K tail are zero-filled
//    by the copy itself (src-size < cp-size), so the inner loop has no edge
//    checks.  Each operand lands in the orientation it has in global memory:
//    no register-staged transpose.  This replaces the two-buffer, register-staged
//    ping-pong of GPU架构下的矩阵乘法深入优化, "5. warp tiling + double buffer".
//
//  * Shared-memory layouts ("MK" = rows of K for A stored M x K, "KM" = rows of
//    M for A stored K x M; likewise "KN"/"NK" for B).  K-contiguous tiles get a
//    4-float row pad, so the 8 (or 4) distinct rows a warp reads in one 16-byte
//    load fall in distinct bank quads (conflict-free; the padding idea of
//    GEMM 优化详解, "Level 3 / Bank Conflict" and 第5章-基础Kernel, "Shared + Padding").
//
//  * Register blocking (GEMM 优化详解, "Level 5: Register Blocking"): each thread
//    owns TM x TN accumulators; per k it reads TM values of op(A) and TN values of
//    op(B) from shared memory with 16-byte loads and issues TM*TN FFMAs.  The
//    thread's rows/columns are chosen so each 16-byte load is either 4
//    consecutive k (K-contiguous tiles) or 4 consecutive rows/columns.
//
//  * Epilogue in registers (GEMM 优化详解, "Level 6: Kernel Fusion" and
//    "Level 7: Vectorized Loads"): v = alpha*acc (+ beta*C) (+ bias[col]),
//    ReLU, then float4 stores where the thread owns 4 consecutive columns and
//    C is 16-byte aligned, scalar stores otherwise.
//
//  * Tiles are visited in groups of GROUP_M tile-rows so that concurrently
//    resident CTAs share panels of A and B in the 126 MB L2.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fgemm {

struct GemmParams {
    const float *A;
    const float *B;
    float *C;
    const float *bias;
    long long lda, ldb, ldc;
    long long strideA, strideB, strideC;
    int M, N, K;  // K is 0 when no products are formed (K == 0 or alpha == 0)
    float alpha, beta;
    int relu;
    int tiles_m, tiles_n;
    int c_vec;  // C pointer, ldc and strideC allow 16-byte accesses
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

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ int clamp_bytes(long long remaining_elems)
{
    return remaining_elems >= 4 ? 16 : (remaining_elems > 0 ? int(remaining_elems) * 4 : 0);
}

// ---- Configuration -------------------------------------------------------------

template <int BM_, int BN_, int BK_, int WM_, int WN_, int TM_, int TN_, int STAGES_, int MINB_,
          int TA_, int TB_, bool VEC_>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int WM = WM_, WN = WN_, TM = TM_, TN = TN_;
    static constexpr int STAGES = STAGES_, MINB = MINB_;
    static constexpr int TA = TA_, TB = TB_;
    static constexpr bool VEC = VEC_;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;
    static constexpr int LR = WM / TM;  // lanes along M
    static constexpr int LC = WN / TN;  // lanes along N
    static constexpr int PAD = 4;       // floats of row padding on K-contiguous tiles
    // Shared-memory tile shapes (floats): A_ROWS x A_LD and B_ROWS x B_LD per stage.
    static constexpr int A_ROWS = TA ? BK : BM;
    static constexpr int A_LD = TA ? BM : BK + PAD;
    static constexpr int B_ROWS = TB ? BN : BK;
    static constexpr int B_LD = TB ? BK + PAD : BN;
    static constexpr int A_STAGE = A_ROWS * A_LD;
    static constexpr int B_STAGE = B_ROWS * B_LD;
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int GROUP_M = 8;

    static_assert(LR * LC == 32, "a warp is LR x LC lanes");
    static_assert(BM % WM == 0 && BN % WN == 0, "warp tiles must cover the CTA tile");
    static_assert(TM % 4 == 0 && TN % 4 == 0 && BK % 4 == 0, "16-byte fragments");
    static_assert((BM * BK / 4) % THREADS == 0 && (BN * BK / 4) % THREADS == 0,
                  "vector copies divide evenly over the threads");
    static_assert((BM * BK) % THREADS == 0 && (BN * BK) % THREADS == 0,
                  "element copies divide evenly over the threads");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// ---- Tile loaders --------------------------------------------------------------

// Copy the (rows x cols) stored block starting at (r0, c0) of a row-major matrix
// with leading dimension ld into a shared tile with row stride S_LD.  Rows at or
// beyond R and columns at or beyond Ccount are zero-filled.
template <int ROWS, int COLS, int S_LD, int THREADS, bool VEC>
__device__ __forceinline__ void load_block(uint32_t s_tile, const float *g, long long ld, long long r0,
                                           long long c0, long long R, long long Ccount, int tid)
{
    if constexpr (VEC) {
        constexpr int CPR = COLS / 4;  // 16-byte chunks per row
        constexpr int ITERS = ROWS * CPR / THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int idx = tid + it * THREADS;
            const int r = idx / CPR, cc = (idx % CPR) * 4;
            const long long gr = r0 + r, gc = c0 + cc;
            const int bytes = gr < R ? clamp_bytes(Ccount - gc) : 0;
            const float *src = bytes ? g + gr * ld + gc : g;
            cp_async_16(s_tile + (r * S_LD + cc) * 4, src, bytes);
        }
    } else {
        constexpr int ITERS = ROWS * COLS / THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int idx = tid + it * THREADS;
            const int r = idx / COLS, cc = idx % COLS;
            const long long gr = r0 + r, gc = c0 + cc;
            const bool ok = gr < R && gc < Ccount;
            cp_async_4(s_tile + (r * S_LD + cc) * 4, ok ? g + gr * ld + gc : g, ok ? 4 : 0);
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void load_stage(uint32_t sA, uint32_t sB, const GemmParams &p,
                                           const float *A, const float *B, int m0, int n0, int k0,
                                           int tid)
{
    if constexpr (Cfg::TA == 0)  // A stored M x K: rows m, columns k
        load_block<Cfg::BM, Cfg::BK, Cfg::A_LD, Cfg::THREADS, Cfg::VEC>(sA, A, p.lda, m0, k0, p.M,
                                                                       p.K, tid);
    else  // A stored K x M: rows k, columns m
        load_block<Cfg::BK, Cfg::BM, Cfg::A_LD, Cfg::THREADS, Cfg::VEC>(sA, A, p.lda, k0, m0, p.K,
                                                                       p.M, tid);
    if constexpr (Cfg::TB == 0)  // B stored K x N
        load_block<Cfg::BK, Cfg::BN, Cfg::B_LD, Cfg::THREADS, Cfg::VEC>(sB, B, p.ldb, k0, n0, p.K,
                                                                       p.N, tid);
    else  // B stored N x K
        load_block<Cfg::BN, Cfg::BK, Cfg::B_LD, Cfg::THREADS, Cfg::VEC>(sB, B, p.ldb, n0, k0, p.N,
                                                                       p.K, tid);
}

// Row (within the CTA tile) of the thread's i-th accumulator row, and column of
// its j-th accumulator column.
template <class Cfg>
__device__ __forceinline__ int frag_row(int wm0, int lr, int i)
{
    if constexpr (Cfg::TA == 0)
        return wm0 + lr + i * Cfg::LR;  // K-contiguous tile: one row per 16-byte load
    else
        return wm0 + (i / 4) * (Cfg::LR * 4) + lr * 4 + (i % 4);  // 4 rows per load
}

template <class Cfg>
__device__ __forceinline__ int frag_col(int wn0, int lc, int j)
{
    if constexpr (Cfg::TB == 1)
        return wn0 + lc + j * Cfg::LC;
    else
        return wn0 + (j / 4) * (Cfg::LC * 4) + lc * 4 + (j % 4);
}

// ---- The kernel ----------------------------------------------------------------

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB) simt_gemm_kernel(const GemmParams p)
{
    extern __shared__ __align__(128) float smem[];
    float *const sA_all = smem;
    float *const sB_all = smem + Cfg::STAGES * Cfg::A_STAGE;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp / Cfg::WARPS_N, warp_n = warp % Cfg::WARPS_N;
    const int lr = lane / Cfg::LC, lc = lane % Cfg::LC;
    const int wm0 = warp_m * Cfg::WM, wn0 = warp_n * Cfg::WN;

    // Grouped tile order: GROUP_M consecutive tile-rows are swept column by column.
    int tile_m, tile_n;
    {
        const int pid = blockIdx.x;
        const int per_group = Cfg::GROUP_M * p.tiles_n;
        const int group = pid / per_group;
        const int first_m = group * Cfg::GROUP_M;
        const int rows_in_group = min(p.tiles_m - first_m, Cfg::GROUP_M);
        const int in_group = pid - group * per_group;
        tile_m = first_m + in_group % rows_in_group;
        tile_n = in_group / rows_in_group;
    }
    const int m0 = tile_m * Cfg::BM, n0 = tile_n * Cfg::BN;
    const long long bz = blockIdx.z;
    const float *const A = p.A + bz * p.strideA;
    const float *const B = p.B + bz * p.strideB;
    float *const C = p.C + bz * p.strideC;

    float acc[Cfg::TM][Cfg::TN];
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
        for (int j = 0; j < Cfg::TN; ++j) acc[i][j] = 0.0f;

    const uint32_t sA_base = smem_addr(sA_all), sB_base = smem_addr(sB_all);
    const int KT = (p.K + Cfg::BK - 1) / Cfg::BK;

    // Prologue: fill STAGES-1 slots.
#pragma unroll
    for (int s = 0; s < Cfg::STAGES - 1; ++s) {
        if (s < KT)
            load_stage<Cfg>(sA_base + s * Cfg::A_STAGE * 4, sB_base + s * Cfg::B_STAGE * 4, p, A, B,
                            m0, n0, s * Cfg::BK, tid);
        cp_async_commit();
    }

    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<Cfg::STAGES - 2>();
        __syncthreads();  // slot kt is visible to all; slot kt-1 is no longer read by anyone
        {
            const int nk = kt + Cfg::STAGES - 1;
            if (nk < KT) {
                const int slot = nk % Cfg::STAGES;
                load_stage<Cfg>(sA_base + slot * Cfg::A_STAGE * 4, sB_base + slot * Cfg::B_STAGE * 4,
                                p, A, B, m0, n0, nk * Cfg::BK, tid);
            }
            cp_async_commit();
        }
        const int slot = kt % Cfg::STAGES;
        const float *const sA = sA_all + slot * Cfg::A_STAGE;
        const float *const sB = sB_all + slot * Cfg::B_STAGE;

#pragma unroll
        for (int kg = 0; kg < Cfg::BK; kg += 4) {
            float a[4][Cfg::TM], b[4][Cfg::TN];
            if constexpr (Cfg::TA == 0) {
#pragma unroll
                for (int i = 0; i < Cfg::TM; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        sA + frag_row<Cfg>(wm0, lr, i) * Cfg::A_LD + kg);
                    a[0][i] = v.x;
                    a[1][i] = v.y;
                    a[2][i] = v.z;
                    a[3][i] = v.w;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int g = 0; g < Cfg::TM / 4; ++g) {
                        const float4 v = *reinterpret_cast<const float4 *>(
                            sA + (kg + kk) * Cfg::A_LD + frag_row<Cfg>(wm0, lr, 4 * g));
                        a[kk][4 * g + 0] = v.x;
                        a[kk][4 * g + 1] = v.y;
                        a[kk][4 * g + 2] = v.z;
                        a[kk][4 * g + 3] = v.w;
                    }
            }
            if constexpr (Cfg::TB == 1) {
#pragma unroll
                for (int j = 0; j < Cfg::TN; ++j) {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        sB + frag_col<Cfg>(wn0, lc, j) * Cfg::B_LD + kg);
                    b[0][j] = v.x;
                    b[1][j] = v.y;
                    b[2][j] = v.z;
                    b[3][j] = v.w;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int g = 0; g < Cfg::TN / 4; ++g) {
                        const float4 v = *reinterpret_cast<const float4 *>(
                            sB + (kg + kk) * Cfg::B_LD + frag_col<Cfg>(wn0, lc, 4 * g));
                        b[kk][4 * g + 0] = v.x;
                        b[kk][4 * g + 1] = v.y;
                        b[kk][4 * g + 2] = v.z;
                        b[kk][4 * g + 3] = v.w;
                    }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
                    for (int j = 0; j < Cfg::TN; ++j) acc[i][j] = fmaf(a[kk][i], b[kk][j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // ---- Epilogue: alpha, beta, bias, ReLU in registers; vector stores where possible.
    const bool products = p.K > 0;
    float bias_v[Cfg::TN];
#pragma unroll
    for (int j = 0; j < Cfg::TN; ++j) {
        const int gc = n0 + frag_col<Cfg>(wn0, lc, j);
        bias_v[j] = (p.bias != nullptr && gc < p.N) ? __ldg(p.bias + gc) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i) {
        const int gr = m0 + frag_row<Cfg>(wm0, lr, i);
        if (gr >= p.M) continue;
        float *const crow = C + (long long)gr * p.ldc;
        float v[Cfg::TN];
#pragma unroll
        for (int j = 0; j < Cfg::TN; ++j) v[j] = products ? p.alpha * acc[i][j] : 0.0f;
        if constexpr (Cfg::TB == 0) {
#pragma unroll
            for (int g = 0; g < Cfg::TN / 4; ++g) {
                const int gc = n0 + frag_col<Cfg>(wn0, lc, 4 * g);
                float *const dst = crow + gc;
                if (p.c_vec && gc + 3 < p.N) {
                    float4 o = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
                    if (p.beta != 0.0f) {
                        const float4 c = *reinterpret_cast<const float4 *>(dst);
                        o.x = fmaf(p.beta, c.x, o.x);
                        o.y = fmaf(p.beta, c.y, o.y);
                        o.z = fmaf(p.beta, c.z, o.z);
                        o.w = fmaf(p.beta, c.w, o.w);
                    }
                    o.x += bias_v[4 * g];
                    o.y += bias_v[4 * g + 1];
                    o.z += bias_v[4 * g + 2];
                    o.w += bias_v[4 * g + 3];
                    if (p.relu) {
                        o.x = fmaxf(o.x, 0.0f);
                        o.y = fmaxf(o.y, 0.0f);
                        o.z = fmaxf(o.z, 0.0f);
                        o.w = fmaxf(o.w, 0.0f);
                    }
                    *reinterpret_cast<float4 *>(dst) = o;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (gc + e >= p.N) break;
                        float o = v[4 * g + e];
                        if (p.beta != 0.0f) o = fmaf(p.beta, dst[e], o);
                        o += bias_v[4 * g + e];
                        if (p.relu) o = fmaxf(o, 0.0f);
                        dst[e] = o;
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < Cfg::TN; ++j) {
                const int gc = n0 + frag_col<Cfg>(wn0, lc, j);
                if (gc >= p.N) continue;
                float o = v[j];
                if (p.beta != 0.0f) o = fmaf(p.beta, crow[gc], o);
                o += bias_v[j];
                if (p.relu) o = fmaxf(o, 0.0f);
                crow[gc] = o;
            }
        }
    }
}

}  // namespace fgemm
