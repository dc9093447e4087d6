// fgemm_internal.h -- declarations shared by the C-ABI layer and the kernel
// instantiation units (host code only; no device code here).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fgemm.h"

namespace fgemm {

struct GemmParams;

// A launcher runs one configuration over `batch` problems on a stream.
using LaunchFn = fgemm_status (*)(const GemmParams &p, int batch, cudaStream_t stream);

// Kernel configurations.  Ids are part of the test/bench interface.
enum ConfigId {
    CFG_128x128 = 0,        // 128x128 CTA tile, 8x8 per thread, 2 CTAs/SM; BK=32 x 3 stages
    CFG_128x64 = 1,         // 128x64x16, 8x8 per thread, 4 stages, 3 CTAs/SM (more CTAs for mid sizes)
    CFG_64x64 = 2,          // 64x64x16, 4x4 per thread, 4 stages (small problems)
    CFG_64x64_SCALAR = 3,   // 64x64x16 with element-wise copies: any alignment
    CFG_32x32 = 4,          // 32x32x16, 4x4 per thread, 64 threads (tiny problems)
    CFG_32x32_K4 = 5,       // 32x32x32, 4x4 per thread, four k-groups of 2 warps, 8 stages
                            // (the smallest grids: a quarter of the serial k-steps per thread)
    CFG_128x128_SPLIT = 6,  // CFG_128x128 for all but the last (tiles mod SMs) tiles, which
                            // then run as 64x64 quarters with four k-groups (second launch)
    CFG_128x128_KSPLIT = 7, // CFG_128x128 for all but the last (tiles mod SMs) tiles, which
                            // then run as clusters of four k-slices of whole tiles (second launch)
    CFG_128x128_KCHAIN = 8, // CFG_128x128 for all but the last (tiles mod SMs) tiles, which
                            // then run as 2..8 k-slices of whole tiles, one launch each,
                            // added into C in slice order (programmatic dependent launches)
    CFG_128x128_SCALAR = 9, // CFG_128x128 with element-wise copies: any alignment
    NUM_CONFIGS = 10,
};

struct ConfigInfo {
    const char *name;
    int bm, bn;
    bool needs_vec;  // requires 16-byte aligned A/B, lda/ldb and batch strides
};

extern const ConfigInfo kConfigs[NUM_CONFIGS];

// SM count of the current device (cached per device).  Returns 0 on success.
int device_sm_count(int *out);

// Number of k-slices (2..8) the k-chain configuration cuts the last r tiles into in the
// given transpose layout: the count with the shortest modelled time (S r whole-tile CTAs
// over K / S, plus the chaining of S launches), the smaller count on a tie.
int kchain_slices(int ta, int tb, long long r, long long K, int num_sms);

// The configuration for a problem (host-only; see fgemm_select_config).
int select_config(int ta, int tb, long long M, long long N, long long K, long long batch,
                  bool aligned, int num_sms);

// Saturating size arithmetic: sizes no allocation could hold come out as SIZE_MAX, so
// they never pass a workspace check by wrapping around.
inline size_t sat_mul(size_t a, size_t b) { return (b != 0 && a > SIZE_MAX / b) ? SIZE_MAX : a * b; }
inline size_t sat_add(size_t a, size_t b) { return a > SIZE_MAX - b ? SIZE_MAX : a + b; }

// Sizes the kernels can index: their 32-bit tile, row, column and k positions run up to
// 255 past the last row, column or k (a 256-row tensor-core tile, a 32-deep k-block), so
// M, N and K stay at or below 2^31 - 256.
inline bool dims_supported(long long M, long long N, long long K)
{
    return M <= FGEMM_MAX_DIM && N <= FGEMM_MAX_DIM && K <= FGEMM_MAX_DIM;
}

// Bytes of the workspace copies a staged call makes with `mask` (bit 0: A, bit 1: B): each
// copy is K x ld4(rows) floats a problem (ld4: rounded up to a multiple of 4), B's starting
// at the next multiple of 256 bytes after A's.  problems_a/_b: the problems each operand
// holds (1 when a batch shares it).
size_t stage_bytes(int mask, long long M, long long N, long long K, long long problems_a,
                   long long problems_b);

// Which operands a staged call copies into the workspace first (bit 0: A, bit 1: B; 0:
// none), by the launch-time model: an operand stored with k contiguous is transposed
// k-major, a k-major one that is not 16-byte aligned gets aligned rows; the copies' modelled
// time plus the GEMM in the layout they leave, against the GEMM as stored, among the copies
// that fit in `workspace_bytes`.  aligned_a/_b: whether the operand as stored allows the
// 16-byte copies.  Host-only.
int staging_choice(int ta, int tb, long long M, long long N, long long K, long long batch,
                   long long problems_a, long long problems_b, bool aligned_a, bool aligned_b,
                   size_t workspace_bytes, int num_sms);

// Y = X^T for each of `batch` problems (stage.cu): X is R x Cc (leading dimension ldx,
// problems sx elements apart), Y is Cc x R (ldy, sy).  Asynchronous on `stream`.
fgemm_status launch_stage_transpose(const float *X, long long ldx, long long sx, int R, int Cc,
                                    int batch, float *Y, long long ldy, long long sy,
                                    cudaStream_t stream);

// Y = X (R x Cc) into rows of leading dimension ldy for each of `batch` problems: the
// copy of a k-major operand whose rows are not 16-byte aligned (stage.cu).
fgemm_status launch_stage_repitch(const float *X, long long ldx, long long sx, int R, int Cc,
                                  int batch, float *Y, long long ldy, long long sy,
                                  cudaStream_t stream);

// A validated problem for the tensor-core path (tc_gemm.cu).
struct TcProblem {
    int ta, tb, M, N, K;
    float alpha, beta;
    const float *A;
    long long lda, sA;
    const float *B;
    long long ldb, sB;
    float *C;
    long long ldc, sC;
    int batch;
    const float *bias;
    int relu;
};

// Whether the tcgen05 kernels can run this problem (layout, alignment, sizes).
bool tc_supported(const TcProblem &q);
// Launch the tcgen05 kernel: mode 1 = TF32, 3 = 3xTF32.
fgemm_status launch_tc(int mode, const TcProblem &q, cudaStream_t stream);
// FGEMM_ERR_TIMEOUT if a tensor-core kernel on the current device recorded a wait
// that ran out (cleared when `clear`), FGEMM_OK otherwise.
fgemm_status tc_device_status(int clear);
// Testing: withhold one k-block in later tensor-core launches (k_block < 0: normal).
void tc_debug_withhold(int k_block, long long wait_limit_ns);

// Validates a split-K call (the rules of fgemm_sgemm_splitk without its workspace)
// and gives the workspace bytes it will use: 0 when it runs without one (splits == 1,
// no products, or nothing to do).
fgemm_status splitk_plan(int ta, int tb, int M, int N, int K, float alpha, const float *A, int lda,
                         const float *B, int ldb, float beta, float *C, int ldc, int splits,
                         size_t *workspace_bytes);

// C = act(alpha * sum_s W[s] + beta * C + bias), W: S slices of M x N (ld N).
fgemm_status launch_splitk_reduce(const float *W, int S, float *C, long long ldc, int M, int N,
                                  float alpha, float beta, const float *bias, int relu,
                                  cudaStream_t stream);

// Launch tables, one per transpose combination (defined in inst_<ta><tb>.cu).
extern const LaunchFn kLaunchNN[NUM_CONFIGS];
extern const LaunchFn kLaunchNT[NUM_CONFIGS];
extern const LaunchFn kLaunchTN[NUM_CONFIGS];
extern const LaunchFn kLaunchTT[NUM_CONFIGS];

}  // namespace fgemm
