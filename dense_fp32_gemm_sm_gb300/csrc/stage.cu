// stage.cu -- re-store an operand whose k index is contiguous in memory as a k-major
// copy, so that the GEMM kernels read both operands with 16-byte copies.
//
// GEMM 优化详解, "Level 1: Naive 实现" (its table of bottlenecks) names the fix for an
// operand read across its stored rows: transpose it or change its layout.  The CUDA-core
// kernels need op(A) and op(B) k-major in shared memory (for each k, a run of m and a
// run of n: the [k][m] tile of GPU架构下的矩阵乘法深入优化, "5. warp tiling + double
// buffer kernel实现").  An operand stored with k contiguous (A for op N, B for op T)
// is transposed on its way into shared memory by 4-byte copies, one per element, in
// every tile that reads it; this pass transposes it once per call into a workspace
// instead, at HBM speed:
//
//     Y[c][r] = X[r][c]   for r < R, c < Cc, every problem of the batch
//
// X: R x Cc, row-major with leading dimension ldx, problems sx elements apart.
// Y: Cc x R, row-major with leading dimension ldy, problems sy elements apart.
//
// An operand that is already k-major but not 16-byte aligned (an odd leading dimension
// or pointer) is copied row by row into aligned rows instead (stage_repitch_kernel),
// so that the GEMM after the copies can use its 16-byte kernels.
//
// Each CTA moves a 64 x 64 block through shared memory.  Interior blocks of a
// 16-byte-aligned X (the common case) go by 16-byte loads and stores: a thread reads
// four 4-float chunks of X's rows and writes four 4-float chunks of Y's rows, with its
// addresses advanced by fixed strides -- a tenth of the instructions of the element-wise
// path, which spends about 40 a element on 64-bit index arithmetic and bounds checks.
// Both are bound by HBM in a timed call: 8 bytes moved per element at about 6 TB/s,
// with the copy's writes evicting whatever dirty lines the L2 holds.  Edge
// blocks and unaligned sources take the element-wise path: 256 threads read rows of 64
// consecutive floats (a warp reads 128 contiguous bytes) and write rows of the
// transpose, with a bounds check per element.  The shared tile has 65 floats per row,
// so the element-wise accesses hit 32 distinct banks and the vector path at most two
// per bank.  Each thread has all its loads in flight before its first store.  Loads of X
// are streaming (X is not read again); Y stays in L2 for the GEMM that follows.

#include <cuda_runtime.h>

#include <cstdint>

#include "fgemm_internal.h"

namespace fgemm {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;
constexpr int kRowsPerPass = kThreads / kTile;      // 4 rows of the block per pass
constexpr int kPasses = kTile / kRowsPerPass;       // 16 passes: 16 elements a thread

__global__ void __launch_bounds__(kThreads) stage_transpose_kernel(
    const float *__restrict__ X, long long ldx, long long sx, int R, int Cc,
    float *__restrict__ Y, long long ldy, long long sy, long long tiles_c, int batch0,
    int x_vec)
{
    __shared__ float tile[kTile][kTile + 1];
    const long long t = blockIdx.x;
    const long long r0 = (t / tiles_c) * kTile;
    const long long c0 = (t % tiles_c) * kTile;
    const long long b = (long long)batch0 + blockIdx.y;
    const float *const x = X + b * sx;
    float *const y = Y + b * sy;

    if (x_vec && r0 + kTile <= R && c0 + kTile <= Cc) {
        // Interior block, 16-byte aligned rows (ldx, ldy multiples of 4; c0, r0 of 64).
        constexpr int kChunks = kTile / 4;           // 16 chunks of 4 floats a row
        constexpr int kRowsV = kThreads / kChunks;   // 16 rows a pass
        constexpr int kPassesV = kTile / kRowsV;     // 4 passes
        const int q = threadIdx.x % kChunks;         // chunk of the row
        const int rr = threadIdx.x / kChunks;        // first row of the pass
        const float *src = x + (r0 + rr) * ldx + c0 + 4 * q;
        const long long src_step = (long long)kRowsV * ldx;
        float4 v[kPassesV];
#pragma unroll
        for (int i = 0; i < kPassesV; ++i)
            v[i] = __ldcs(reinterpret_cast<const float4 *>(src + i * src_step));
#pragma unroll
        for (int i = 0; i < kPassesV; ++i) {
            float *row = &tile[rr + i * kRowsV][4 * q];
            row[0] = v[i].x;
            row[1] = v[i].y;
            row[2] = v[i].z;
            row[3] = v[i].w;
        }
        __syncthreads();
        // Y row c0 + cc, columns r0 + 4 q .. + 3: column cc of tile rows 4 q .. 4 q + 3.
        float *dst = y + (c0 + rr) * ldy + r0 + 4 * q;
        const long long dst_step = (long long)kRowsV * ldy;
#pragma unroll
        for (int i = 0; i < kPassesV; ++i) {
            const int cc = rr + i * kRowsV;
            const float4 w = make_float4(tile[4 * q][cc], tile[4 * q + 1][cc], tile[4 * q + 2][cc],
                                         tile[4 * q + 3][cc]);
            *reinterpret_cast<float4 *>(dst + i * dst_step) = w;
        }
        return;
    }

    const int tc = threadIdx.x % kTile;  // column of X read, then column of Y written
    const int tr = threadIdx.x / kTile;  // first row of the pass
    float v[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const long long r = r0 + tr + i * kRowsPerPass;
        const long long c = c0 + tc;
        v[i] = (r < R && c < Cc) ? __ldcs(x + r * ldx + c) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) tile[tr + i * kRowsPerPass][tc] = v[i];
    __syncthreads();
    // Row c of Y takes column c of the block: thread (tc, tr) writes Y[c0 + tr + ...][r0 + tc].
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const long long c = c0 + tr + i * kRowsPerPass;
        const long long r = r0 + tc;
        if (c < Cc && r < R) y[c * ldy + r] = tile[tc][tr + i * kRowsPerPass];
    }
}

// Y = X row by row into rows of leading dimension ldy (a multiple of 4): an operand
// that is already k-major but whose rows do not start on 16 bytes gets aligned rows.
// Thread (x, y) copies column blockIdx.x * 256 + threadIdx.x of a group of kRepitchRows
// rows, all loads in flight before the stores; warps read and write 128 contiguous bytes.
constexpr int kRepitchRows = 8;

__global__ void __launch_bounds__(kThreads) stage_repitch_kernel(
    const float *__restrict__ X, long long ldx, long long sx, int R, int Cc,
    float *__restrict__ Y, long long ldy, long long sy, int batch0)
{
    const long long b = (long long)batch0 + blockIdx.z;
    const float *const x = X + b * sx;
    float *const y = Y + b * sy;
    const long long c = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (c >= Cc) return;
    for (long long r0 = (long long)blockIdx.y * kRepitchRows; r0 < R;
         r0 += (long long)gridDim.y * kRepitchRows) {
        float v[kRepitchRows];
#pragma unroll
        for (int i = 0; i < kRepitchRows; ++i)
            v[i] = r0 + i < R ? __ldcs(x + (r0 + i) * ldx + c) : 0.0f;
#pragma unroll
        for (int i = 0; i < kRepitchRows; ++i)
            if (r0 + i < R) y[(r0 + i) * ldy + c] = v[i];
    }
}

}  // namespace

fgemm_status launch_stage_repitch(const float *X, long long ldx, long long sx, int R, int Cc,
                                  int batch, float *Y, long long ldy, long long sy,
                                  cudaStream_t stream)
{
    if (R <= 0 || Cc <= 0 || batch <= 0) return FGEMM_OK;
    const long long gx = ((long long)Cc + kThreads - 1) / kThreads;
    const long long groups = ((long long)R + kRepitchRows - 1) / kRepitchRows;
    if (gx > 0x7FFFFFFFLL) return FGEMM_ERR_NOT_SUPPORTED;
    const unsigned gy = (unsigned)(groups < 65535 ? groups : 65535);
    for (int b0 = 0; b0 < batch; b0 += 65535) {
        const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
        stage_repitch_kernel<<<dim3((unsigned)gx, gy, (unsigned)nb), kThreads, 0, stream>>>(
            X, ldx, sx, R, Cc, Y, ldy, sy, b0);
        if (cudaGetLastError() != cudaSuccess) return FGEMM_ERR_LAUNCH;
    }
    return FGEMM_OK;
}

fgemm_status launch_stage_transpose(const float *X, long long ldx, long long sx, int R, int Cc,
                                    int batch, float *Y, long long ldy, long long sy,
                                    cudaStream_t stream)
{
    if (R <= 0 || Cc <= 0 || batch <= 0) return FGEMM_OK;
    const long long tiles_r = ((long long)R + kTile - 1) / kTile;
    const long long tiles_c = ((long long)Cc + kTile - 1) / kTile;
    const long long tiles = tiles_r * tiles_c;
    if (tiles > 0x7FFFFFFFLL) return FGEMM_ERR_NOT_SUPPORTED;
    // 16-byte vectors need every row of X and Y (and every problem) to start on 16 bytes.
    const bool x_vec = reinterpret_cast<uintptr_t>(X) % 16 == 0 && ldx % 4 == 0 &&
                       (batch == 1 || sx % 4 == 0) && reinterpret_cast<uintptr_t>(Y) % 16 == 0 &&
                       ldy % 4 == 0 && (batch == 1 || sy % 4 == 0);
    for (int b0 = 0; b0 < batch; b0 += 65535) {
        const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
        stage_transpose_kernel<<<dim3((unsigned)tiles, (unsigned)nb, 1), kThreads, 0, stream>>>(
            X, ldx, sx, R, Cc, Y, ldy, sy, tiles_c, b0, x_vec ? 1 : 0);
        if (cudaGetLastError() != cudaSuccess) return FGEMM_ERR_LAUNCH;
    }
    return FGEMM_OK;
}

}  // namespace fgemm
