/*
 * fgemm.h -- C ABI of a single-GPU FP32 GEMM library for NVIDIA GB300 (sm_103a).
 *
 * The operation (GEMM 优化详解, "GEMM 基础理论 / 数学定义"; 第5章-基础Kernel,
 * "1.1 什么是矩阵乘法"):
 *
 *     C = alpha * op(A) * op(B) + beta * C,   op(A) is M x K, op(B) is K x N, C is M x N,
 *     C[i][j] = alpha * sum_{k=0}^{K-1} op(A)[i][k] * op(B)[k][j] + beta * C[i][j]
 *
 * All matrices are ROW-MAJOR with an explicit leading dimension (the distance,
 * in elements, between the starts of two consecutive stored rows):
 *   transa == FGEMM_OP_N: A is stored M x K, element (i,k) at A[i*lda + k], lda >= max(1,K)
 *   transa == FGEMM_OP_T: A is stored K x M, element (i,k) at A[k*lda + i], lda >= max(1,M)
 *   transb == FGEMM_OP_N: B is stored K x N, element (k,j) at B[k*ldb + j], ldb >= max(1,N)
 *   transb == FGEMM_OP_T: B is stored N x K, element (k,j) at B[j*ldb + k], ldb >= max(1,K)
 *   C is stored M x N, element (i,j) at C[i*ldc + j], ldc >= max(1,N).
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers owned by the caller.  The library allocates
 *     nothing, frees nothing and keeps no workspace.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream)
 *     and never synchronises.  Results are valid once the stream has run.
 *   - C must not share memory with A, B or a bias vector (not checked; such a call
 *     gives undefined results).  A, B and the bias are only read and may overlap
 *     one another.
 *   - beta == 0: C is not read before it is written (it may hold NaN).
 *   - alpha == 0 or K == 0: no products are formed and A, B are not read
 *     (they may be NULL); the result is beta*C (then bias, ReLU).
 *   - M == 0, N == 0 or batch == 0: nothing happens and FGEMM_OK is returned.
 *   - Invalid arguments return FGEMM_ERR_INVALID_VALUE before anything is
 *     launched; C is left untouched.  A failed launch returns FGEMM_ERR_LAUNCH.
 *     Nothing aborts or exits the process.
 *   - Sizes: M, N and K up to FGEMM_MAX_DIM (2^31 - 256); a valid call with a larger
 *     one returns FGEMM_ERR_NOT_SUPPORTED before anything is launched.  Element
 *     offsets are 64-bit, so C, A and B may each hold more than 2^31 elements; tile,
 *     row, column and k positions are 32-bit and run up to 255 past the last row,
 *     column or k, which the limit keeps below 2^31.
 *   - Any alignment is accepted.  When the pointer, leading dimension or batch
 *     stride of a k-major operand (A for transa == T, B for transb == N) is not a
 *     multiple of 16 bytes, the call runs a kernel that moves single elements
 *     instead of 16-byte vectors (an operand stored with k contiguous is moved
 *     element by element in any case, so its alignment does not matter); C's
 *     alignment only decides between vector and element stores.
 *   - Arithmetic is IEEE FP32 fused multiply-add on the CUDA cores, summing k
 *     in an order that differs from the plain loop; results agree with an FP64
 *     evaluation to within 1e-5 * (|alpha| sum_k |a_ik||b_kj| + |beta||c_ij| + |bias_j|).
 *   - Thread safety: calls from several host threads are safe, with two
 *     exceptions: fgemm_sgemm_splitk_noalloc calls whose kernels overlap on the GPU
 *     share one scratch array and must be ordered (see there), and the test hook
 *     fgemm_debug_withhold_tensor_core must not run beside tensor-core calls.
 *   - Per-context state: the library caches a few per-context facts (the device
 *     address of its own __device__ variables, kernel attributes) keyed on the
 *     context's id, so they are looked up again after cudaDeviceReset.
 */
#ifndef FGEMM_H
#define FGEMM_H

#include <cuda_runtime_api.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fgemm_status {
    FGEMM_OK = 0,
    FGEMM_ERR_INVALID_VALUE = 1, /* an argument breaks the rules above; nothing launched */
    FGEMM_ERR_LAUNCH = 2,        /* the CUDA launch (or a CUDA query before it) failed */
    FGEMM_ERR_NOT_SUPPORTED = 3, /* e.g. no sm_103a device, a config that cannot run the call,
                                    or a size above FGEMM_MAX_DIM */
    FGEMM_ERR_TIMEOUT = 4,       /* a tensor-core kernel gave up waiting (fgemm_device_status) */
} fgemm_status;

typedef enum fgemm_op { FGEMM_OP_N = 0, FGEMM_OP_T = 1 } fgemm_op;

/* Largest M, N or K a call takes (see "Sizes" above). */
#define FGEMM_MAX_DIM 2147483392

/*
 * Plain GEMM: C = alpha*op(A)*op(B) + beta*C.
 * Defined by GEMM 优化详解, "数学定义" (C = alpha x A x B + beta x C) with the
 * 0-based sum of 第5章-基础Kernel, "1.1 什么是矩阵乘法".
 */
fgemm_status fgemm_sgemm(fgemm_op transa, fgemm_op transb, int M, int N, int K, float alpha,
                         const float *A, int lda, const float *B, int ldb, float beta, float *C,
                         int ldc, cudaStream_t stream);

/*
 * Fully-connected layer epilogue fused into the GEMM (GEMM 优化详解, "Level 6:
 * Kernel Fusion", and the layer Y = X x W + b of "为什么 GEMM 重要？"):
 *     C[i][j] = act( alpha * sum_k op(A)[i][k] op(B)[k][j] + beta * C[i][j] + bias[j] )
 * bias: device vector of N floats indexed by output column, or NULL for none.
 * apply_relu: nonzero applies act(x) = max(0, x) (a NaN becomes 0); zero applies none.
 * All four combinations of bias / ReLU are accepted.
 */
fgemm_status fgemm_sgemm_bias_relu(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                   float alpha, const float *A, int lda, const float *B, int ldb,
                                   float beta, float *C, int ldc, const float *bias,
                                   int apply_relu, cudaStream_t stream);

/*
 * The same fused epilogue with a bias per output ROW (row-broadcast bias):
 *     C[i][j] = act( alpha * sum_k op(A)[i][k] op(B)[k][j] + beta * C[i][j] + row_bias[i] )
 * (the per-column bias of GEMM 优化详解, "Level 6: Kernel Fusion", broadcast the other
 * way, e.g. a per-query term added to attention scores).  row_bias: device vector of
 * M floats, or NULL; apply_relu as above.  Runs on the CUDA cores.
 */
fgemm_status fgemm_sgemm_row_bias_relu(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                       float alpha, const float *A, int lda, const float *B,
                                       int ldb, float beta, float *C, int ldc,
                                       const float *row_bias, int apply_relu, cudaStream_t stream);

/*
 * Strided batch: for b in [0, batch), the plain GEMM on A + b*strideA,
 * B + b*strideB, C + b*strideC (strides in elements).  Used for batched
 * attention scores Q x K^T (GEMM 优化详解, "为什么 GEMM 重要？"; batching small
 * problems is the page's advice for small matrices in "矩阵大小选择策略").
 * strideA, strideB >= 0 (0 reuses one operand for every problem).
 * strideC >= 0, and no element of C may belong to two problems (checked
 * exactly, so interleaved layouts such as ldc = batch*N, strideC = N are
 * accepted); an overlap returns FGEMM_ERR_INVALID_VALUE.
 */
fgemm_status fgemm_sgemm_strided_batched(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                         float alpha, const float *A, int lda, long long strideA,
                                         const float *B, int ldb, long long strideB, float beta,
                                         float *C, int ldc, long long strideC, int batch,
                                         cudaStream_t stream);

/*
 * Split-K GEMM for problems with few output tiles and a long K (small squares,
 * skinny outputs): the small-matrix strategy of GEMM 优化详解, "矩阵大小选择策略",
 * where one tile per SM would leave most of the GPU idle.  The K range is cut into
 * `splits` slices (each a multiple of 32 deep); every slice's partial product is
 * written to `workspace` by the CUDA-core kernel, then one reduction kernel sums the
 * slices in a fixed order and applies the epilogue:
 *     C = act( alpha * sum_s P_s + beta * C + bias[col] )    (bias may be NULL)
 * The sum order is fixed, so results are the same on every run (they may differ in
 * the last bits from fgemm_sgemm, whose sum order differs).
 * workspace: caller-owned device memory of at least fgemm_splitk_workspace_size()
 * bytes, 16-byte aligned, not overlapping A, B, C or bias; its contents are
 * overwritten.  splits in [1, 64] (1 = fgemm_sgemm_bias_relu); a single problem
 * (no batch).  Other rules as for fgemm_sgemm_bias_relu; a missing or too small
 * workspace returns FGEMM_ERR_INVALID_VALUE before anything is launched.
 */
size_t fgemm_splitk_workspace_size(int M, int N, int K, int splits);

fgemm_status fgemm_sgemm_splitk(fgemm_op transa, fgemm_op transb, int M, int N, int K, float alpha,
                                const float *A, int lda, const float *B, int ldb, float beta,
                                float *C, int ldc, const float *bias, int apply_relu, int splits,
                                float *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Split-K without any device allocation, for callers that are not allowed to call
 * cudaMalloc (a plugin inside a program that owns all GPU memory through its own
 * pool, a latency-critical loop that cannot afford cudaMalloc's synchronisation and
 * cost, a process with a fixed memory budget).  The source pages have no
 * counterpart; this is a property of the library, not of the method.
 *
 * Same arguments and result as fgemm_sgemm_splitk, without the workspace: the
 * partial products go to one fixed array of FGEMM_NOALLOC_SCRATCH_BYTES in the
 * global memory of every GPU that loads the library, held until the process exits.
 *   - Order of checks: first the argument rules of fgemm_sgemm_splitk
 *     (FGEMM_ERR_INVALID_VALUE); then, for a call that uses partial products
 *     (splits > 1, K > 0, alpha != 0), their size: more than the array holds
 *     (fgemm_splitk_workspace_size(M, N, K, splits) > FGEMM_NOALLOC_SCRATCH_BYTES)
 *     returns FGEMM_ERR_NOT_SUPPORTED before anything is launched.  16 MiB holds,
 *     e.g., 4 slices of a 1024 x 1024 C.  A call that needs no partial products
 *     runs at any size, exactly as fgemm_sgemm_splitk runs it.
 *   - The first call in each CUDA context (per device, and again after
 *     cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - Every call uses the same array and leaves its contents behind; nothing in it has
 *     to start at zero (each partial product is written before it is read).  Calls
 *     whose kernels overlap on the GPU -- on different streams, or from different
 *     host threads -- race on the array and give wrong results: order them.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define FGEMM_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

fgemm_status fgemm_sgemm_splitk_noalloc(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                        float alpha, const float *A, int lda, const float *B,
                                        int ldb, float beta, float *C, int ldc, const float *bias,
                                        int apply_relu, int splits, cudaStream_t stream);

/*
 * GEMM with operand staging through a caller workspace.  GEMM 优化详解, "Level 1:
 * Naive 实现" (its table of bottlenecks), gives the remedy for an operand read across
 * its stored rows: transpose it or change its layout.  The CUDA-core kernels keep
 * op(A) and op(B) k-major in shared memory, so an operand stored with k contiguous
 * (A for transa == N, B for transb == T) is transposed on its way in, by 4-byte
 * copies in every tile that reads it, and an operand whose rows do not start on 16
 * bytes (an odd leading dimension, batch stride or pointer) makes the call take the
 * element-wise kernel.  This call can instead copy an operand once into `workspace`:
 * transposed k-major when it is stored with k contiguous, row by row into aligned rows
 * when it is already k-major (8 bytes moved per element at HBM speed).  The GEMM then
 * runs on the copies with 16-byte copies only.  On a 152-SM GB300 this pays for large
 * products (4096^3 NN, the 8192 x 4096 x 11008 FC layer, batched Q x K^T; any unaligned
 * problem beyond a few hundred per side) and not for small ones, so by default the
 * launch-time model decides per call.
 *
 * Result: that of fgemm_gemm_explicit with config -1 and the same arguments (strided
 * batch, bias (may be NULL), ReLU), within the same error bound; the sum order can
 * differ from the unstaged call, so the last bits may too.
 *   stage: -1 lets the model choose among the copies that fit in the workspace (none
 *     when workspace is NULL or too small for any); otherwise a mask of the copies to
 *     make -- bit 0 copies A, bit 1 copies B, 0 runs the plain kernels -- whose bytes
 *     must fit (else FGEMM_ERR_INVALID_VALUE).  Anything outside [-1, 3] returns
 *     FGEMM_ERR_INVALID_VALUE.
 *   workspace: caller-owned device memory, 16-byte aligned (else
 *     FGEMM_ERR_INVALID_VALUE), not overlapping A, B, C or bias; `workspace_bytes` of it
 *     may be overwritten.  fgemm_staged_workspace_size(transa, transb, M, N, K, batch)
 *     bytes hold every copy the call could make (both operands); less limits the
 *     model's choice.  An operand a batch shares (stride 0) is copied once.  Staged calls
 *     whose kernels may overlap on the GPU (other streams, other host threads) need
 *     workspaces of their own; calls on one stream may share one.
 *   Checks happen before anything is launched.
 * A staged call launches on `stream` one copy kernel per copied operand (and per 65535
 * problems of a batch), then the GEMM's launches (fgemm_launch_count of the layout the
 * copies leave); it may be captured in a CUDA graph.  Other rules as for
 * fgemm_gemm_explicit.
 */
size_t fgemm_staged_workspace_size(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                   int batch);

fgemm_status fgemm_sgemm_staged(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                float alpha, const float *A, int lda, long long strideA,
                                const float *B, int ldb, long long strideB, float beta, float *C,
                                int ldc, long long strideC, int batch, const float *bias,
                                int apply_relu, int stage, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * The mask fgemm_sgemm_staged(stage = -1) would use on a GPU with `num_sms` SMs and a
 * workspace of `workspace_bytes`: bit 0 set when it copies A, bit 1 when it copies B, 0
 * when it runs the plain kernels.  shared_a / shared_b: nonzero when the batch shares the
 * operand (its stride is 0); aligned_a / aligned_b: nonzero when the operand as stored
 * is 16-byte aligned (pointer, leading dimension and batch stride).  -1 for arguments
 * out of range.  Host-only: no CUDA call is made.
 */
int fgemm_staged_choice(fgemm_op transa, fgemm_op transb, int M, int N, int K, int batch,
                        int shared_a, int shared_b, int aligned_a, int aligned_b,
                        size_t workspace_bytes, int num_sms);

/*
 * Arithmetic of the contraction (GEMM 优化详解, "进一步优化方向": tensor cores are the
 * next step after the CUDA-core ladder):
 *   FGEMM_MATH_FP32    FP32 FMA on the CUDA cores (the plain entry points use this).
 *   FGEMM_MATH_TF32    tcgen05 tensor cores, each operand read as TF32 (10 mantissa
 *                      bits); error within 2e-3 * sum_k |a_ik||b_kj| per element.
 *   FGEMM_MATH_3XTF32  tensor cores with each operand split on chip into a TF32 high
 *                      part and a residual, three products per term (hi*hi, hi*lo,
 *                      lo*hi): near-FP32 accuracy.
 * Special values: FP32 and TF32 give IEEE results (NaN and infinities land where the
 * definition puts them; TF32 drops the 13 low mantissa bits, so a NaN whose payload
 * lies only there reads as an infinity).  In 3xTF32 an infinity in an operand makes
 * NaN of the outputs it reaches (a correction product multiplies it by the other
 * operand's residual, often 0); outputs the definition leaves finite are unaffected.
 */
typedef enum fgemm_math {
    FGEMM_MATH_FP32 = 0,
    FGEMM_MATH_TF32 = 1,
    FGEMM_MATH_3XTF32 = 2,
} fgemm_math;

/*
 * The general call with a choice of arithmetic.  Arguments, conventions and
 * validation are those of fgemm_gemm_explicit (bias may be NULL; batch = 1 with
 * zero strides is a single GEMM).  The tensor-core modes take every transpose
 * combination; they need 16-byte aligned A and B and lda, ldb, strideA, strideB
 * multiples of 4.  A call they cannot run (unaligned operands, K == 0, alpha == 0)
 * uses the FP32 CUDA-core kernel instead (at least as accurate);
 * fgemm_math_supported tells beforehand which one a call will use.  A tensor-core kernel bounds
 * every internal wait; if one runs out it stops, leaves C undefined and records it
 * for fgemm_device_status.
 */
fgemm_status fgemm_gemm_math(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N,
                             int K, float alpha, const float *A, int lda, long long strideA,
                             const float *B, int ldb, long long strideB, float beta, float *C,
                             int ldc, long long strideC, int batch, const float *bias,
                             int apply_relu, cudaStream_t stream);

/*
 * FGEMM_ERR_TIMEOUT if a tensor-core kernel on the current device recorded a wait
 * that ran out since the word was last cleared, FGEMM_OK if not.  Reads device
 * memory synchronously: call it after the streams that ran the kernels have
 * finished.  Nonzero `clear` resets the record.
 */
fgemm_status fgemm_device_status(int clear);

/*
 * Which arithmetic fgemm_gemm_math will use for a call with these operands: 1 when
 * it runs the requested one (always for FGEMM_MATH_FP32; for the tensor-core modes
 * when the layout, alignment and sizes suit the tcgen05 kernel), 0 when it would run
 * the FP32 CUDA-core kernel instead (unaligned operands, K == 0, alpha == 0, an empty
 * problem, or no driver) or nothing at all (a size above FGEMM_MAX_DIM), -1 when
 * `math` is not an fgemm_math value.  The arguments
 * mean what they mean for fgemm_gemm_math; the pointers are only tested for 16-byte
 * alignment, never dereferenced, and nothing else is validated.  Host-only: no
 * kernel runs and no device memory is touched (the first call looks up the driver's
 * tensor-map encoder).
 */
int fgemm_math_supported(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N, int K,
                         float alpha, const float *A, int lda, long long strideA, const float *B,
                         int ldb, long long strideB, int batch);

/*
 * fgemm_gemm_math with operand staging through a caller workspace: the tensor-core
 * counterpart of fgemm_sgemm_staged (with FGEMM_MATH_FP32 it is fgemm_sgemm_staged).
 * The tcgen05 kernel reads an operand stored K-major (A for transa == N, B for
 * transb == T) straight from its TMA tiles; with both operands MN-major (transa == T,
 * transb == N) it also transposes one of them in shared memory and runs at about half
 * the rate of the other layouts, and an operand whose pointer, leading dimension or
 * batch stride is not 16-byte aligned keeps the call off the tensor cores.  This call can
 * first copy operands K-major into `workspace` -- transposed when MN-major, into aligned
 * rows when already K-major -- and run the tensor-core kernel on the copies.
 * Result: that of fgemm_gemm_math on the same arguments (the copies are exact), except
 * that a call whose unaligned operands the copies make aligned runs on the tensor cores
 * (with their error bound) instead of the CUDA cores.
 *   stage: -1 lets the library choose among the copies that fit: every operand whose
 *     alignment keeps the call off the tensor cores (all of them or none), else in a TN
 *     call the copy of A (so that it runs as NN), or B's when only that fits; otherwise
 *     a mask of the copies to make -- bit 0 copies A, bit 1 copies B -- whose bytes must
 *     fit (else FGEMM_ERR_INVALID_VALUE).  Anything outside [-1, 3] returns
 *     FGEMM_ERR_INVALID_VALUE.
 *   workspace: as for fgemm_sgemm_staged; fgemm_math_staged_workspace_size(math, ...)
 *     bytes hold both copies (A as M x K rows, B as N x K rows, each row rounded up to
 *     a multiple of 4 floats); less limits the choice.  Concurrent calls need workspaces
 *     of their own.  Checks happen before anything is launched.
 * A staged call launches one copy kernel per copied operand (and per 65535 problems of
 * a batch) on `stream`, then the GEMM; it may be captured in a CUDA graph.
 * fgemm_math_staged_choice (host-only; arguments as for fgemm_staged_choice) gives the
 * mask stage = -1 would use, or -1 for arguments out of range.
 */
size_t fgemm_math_staged_workspace_size(fgemm_math math, fgemm_op transa, fgemm_op transb, int M,
                                        int N, int K, int batch);

int fgemm_math_staged_choice(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N,
                             int K, int batch, int shared_a, int shared_b, int aligned_a,
                             int aligned_b, size_t workspace_bytes, int num_sms);

fgemm_status fgemm_gemm_math_staged(fgemm_math math, fgemm_op transa, fgemm_op transb, int M,
                                    int N, int K, float alpha, const float *A, int lda,
                                    long long strideA, const float *B, int ldb, long long strideB,
                                    float beta, float *C, int ldc, long long strideC, int batch,
                                    const float *bias, int apply_relu, int stage, void *workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/*
 * Testing only (failure detection without a GPU fault).  Makes later tensor-core
 * launches of this process behave as if the copy of k-block `k_block` never arrived:
 * the producer withholds it, the kernel's bounded wait runs out after
 * `wait_limit_ns` (<= 0: the default 4 s), the kernel drains its own copies and
 * MMAs, frees its tensor memory, records FGEMM_ERR_TIMEOUT for fgemm_device_status
 * and returns with C undefined; the CUDA context stays usable.  k_block < 0 restores
 * normal operation.  Not thread-safe with concurrent tensor-core calls.
 */
void fgemm_debug_withhold_tensor_core(int k_block, long long wait_limit_ns);

/* Static, human-readable text for a status code (never NULL). */
const char *fgemm_status_string(fgemm_status status);

/* ----------------------------------------------------------------------------
 * Kernel configurations (for tests and benchmarks).
 *
 * The plain entry points pick a kernel configuration from the shape, the
 * transposes, 16-byte alignment and the SM count: the one with the least launch
 * time estimated by a model fitted to measurements (the number of CTAs the busiest
 * SM runs, times a per-k cost, with a latency floor).  The calls below expose that
 * choice so every configuration can be tested on edge shapes, and timed.
 *
 * Three configurations issue more than one kernel launch on the caller's stream:
 * whole 128 x 128 tiles first, then the last (tiles mod SMs) tiles either as 64 x 64
 * quarter tiles ("..._split", one more launch), as thread-block clusters of four CTAs
 * that each multiply one k-slice of a tile and add their partial sums through
 * distributed shared memory in a fixed order ("..._ksplit", one more launch), or as
 * two to eight k-slices of every tile, one launch per slice, each adding its products
 * into C in slice order ("..._kchain"; fgemm_launch_count gives the number).  Every
 * last-wave launch is a programmatic dependent of the launch before it: it may start
 * while that one runs and waits for it only before writing C.  All allocate nothing and
 * give the same result on every run.
 *
 * Calls with an unaligned k-major operand (see the alignment rule above) take one of
 * the two "..._scalar" configurations, which move single elements: the 128 x 128 tile
 * for large problems, the 64 x 64 tile for small ones (by the same model).  The
 * `aligned` argument of the queries below means the vector configurations may run.
 * ------------------------------------------------------------------------- */

/* Number of kernel configurations; valid ids are 0 .. fgemm_num_configs()-1. */
int fgemm_num_configs(void);

/* Static name of a configuration ("simt_128x128_t8x8", "simt_128x128_t8x8_ksplit", ...),
 * or NULL for a bad id. */
const char *fgemm_config_name(int config);

/*
 * The configuration the plain entry points would use for this problem on a
 * GPU with `num_sms` SMs.  `aligned` is nonzero when A, B, their leading
 * dimensions and batch strides are all multiples of 16 bytes.  Host-only: no
 * CUDA call is made.  Returns -1 for arguments the entry points would reject.
 */
int fgemm_select_config(fgemm_op transa, fgemm_op transb, int M, int N, int K, int batch,
                        int aligned, int num_sms);

/*
 * Kernel launches one call with this configuration (config < 0: the one the plain entry
 * points would select) makes on a GPU with `num_sms` SMs: 1 for most configurations (1
 * per 65535 problems of a batch; TT whole 128 x 128 tiles 1 per 2^31 - 1 tiles), and for the
 * last-wave configurations one for the
 * whole tiles (if any) plus one for the last (tiles mod SMs) tiles -- or, for
 * "..._kchain", one per k-slice (2 to 8, chosen from the remainder and K).  K is the
 * depth the kernels see: 0 when alpha == 0.  0 for an empty problem and for calls the
 * entry points refuse as FGEMM_ERR_NOT_SUPPORTED (a size above FGEMM_MAX_DIM, or more
 * tiles than one launch takes), -1 for arguments they reject as invalid.  Host-only: no
 * CUDA call is made.
 */
int fgemm_launch_count(int config, fgemm_op transa, fgemm_op transb, int M, int N, int K,
                       int batch, int aligned, int num_sms);

/*
 * The most general call, with an explicit configuration (config < 0 means
 * "select as the plain entry points do").  Argument meaning and validation are
 * those of the calls above (bias may be NULL; batch = 1 with zero strides is a
 * single GEMM).  A configuration that needs 16-byte alignment returns
 * FGEMM_ERR_NOT_SUPPORTED for unaligned operands.
 */
fgemm_status fgemm_gemm_explicit(int config, fgemm_op transa, fgemm_op transb, int M, int N,
                                 int K, float alpha, const float *A, int lda, long long strideA,
                                 const float *B, int ldb, long long strideB, float beta, float *C,
                                 int ldc, long long strideC, int batch, const float *bias,
                                 int apply_relu, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FGEMM_H */
