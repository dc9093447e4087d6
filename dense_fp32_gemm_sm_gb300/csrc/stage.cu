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
// Each CTA moves a 64 x 64 block through shared memory: 256 threads read it as rows
// of 64 consecutive floats (a warp reads 128 contiguous bytes) and write it back as
// rows of the transpose (likewise contiguous).  The shared tile has 65 floats per row,
// so both the row-wise writes and the column-wise reads hit 32 distinct banks.  Each
// thread holds 16 loads in flight before its first store, which keeps enough bytes
// moving to saturate HBM.  Elements outside X are neither read nor written.
#include <cuda_runtime.h>

#include "fgemm_internal.h"

namespace fgemm {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;
constexpr int kRowsPerPass = kThreads / kTile;      // 4 rows of the block per pass
constexpr int kPasses = kTile / kRowsPerPass;       // 16 passes: 16 elements a thread

__global__ void __launch_bounds__(kThreads) stage_transpose_kernel(
    const float *__restrict__ X, long long ldx, long long sx, int R, int Cc,
    float *__restrict__ Y, long long ldy, long long sy, long long tiles_c, int batch0)
{
    __shared__ float tile[kTile][kTile + 1];
    const long long t = blockIdx.x;
    const long long r0 = (t / tiles_c) * kTile;
    const long long c0 = (t % tiles_c) * kTile;
    const long long b = (long long)batch0 + blockIdx.y;
    const float *const x = X + b * sx;
    float *const y = Y + b * sy;
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

}  // namespace

fgemm_status launch_stage_transpose(const float *X, long long ldx, long long sx, int R, int Cc,
                                    int batch, float *Y, long long ldy, long long sy,
                                    cudaStream_t stream)
{
    if (R <= 0 || Cc <= 0 || batch <= 0) return FGEMM_OK;
    const long long tiles_r = ((long long)R + kTile - 1) / kTile;
    const long long tiles_c = ((long long)Cc + kTile - 1) / kTile;
    const long long tiles = tiles_r * tiles_c;
    if (tiles > 0x7FFFFFFFLL) return FGEMM_ERR_NOT_SUPPORTED;
    for (int b0 = 0; b0 < batch; b0 += 65535) {
        const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
        stage_transpose_kernel<<<dim3((unsigned)tiles, (unsigned)nb, 1), kThreads, 0, stream>>>(
            X, ldx, sx, R, Cc, Y, ldy, sy, tiles_c, b0);
        if (cudaGetLastError() != cudaSuccess) return FGEMM_ERR_LAUNCH;
    }
    return FGEMM_OK;
}

}  // namespace fgemm
