// fgemm_api.cu -- the C ABI: argument validation, kernel selection, dispatch.
//
// Validation and selection are plain host integer code and run before any CUDA
// call, so an invalid call never touches the device (and can be tested on a
// machine without a GPU).  The launcher pattern (build grid/block, launch on the
// caller's stream, then check the launch) is the host side of every listing in
// GPU架构下的矩阵乘法深入优化 ("CUDA_CHECK(cudaPeekAtLastError())"), turned into
// status codes because a library must not abort its caller.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>

#include "fgemm_internal.h"
#include "simt_gemm.cuh"

namespace fgemm {

const ConfigInfo kConfigs[NUM_CONFIGS] = {
    {"simt_128x128_t8x8", 128, 128, true},
    {"simt_128x64x16_t8x8_s4", 128, 64, true},
    {"simt_64x64x16_t4x4_s4", 64, 64, true},
    {"simt_64x64x16_t4x4_s4_scalar", 64, 64, false},
    {"simt_32x32x16_t4x4_s4", 32, 32, true},
    {"simt_32x32x32_t4x4_s8_k4", 32, 32, true},
    {"simt_128x128_t8x8_split", 128, 128, true},
    {"simt_128x128_t8x8_ksplit", 128, 128, true},
    {"simt_128x128_t8x8_kchain", 128, 128, true},
    {"simt_128x128_t8x8_scalar", 128, 128, false},
};

namespace {

struct Problem {
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
    cudaStream_t stream;
    const float *row_bias = nullptr;
};

long long floor_div(long long a, long long b)
{
    long long q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
    return q;
}

// True when two different problems of the batch would write the same element
// of C: (b - b') * sC == di * ldc + dj with |di| < M, |dj| < N for some b != b'.
bool c_batches_overlap(long long M, long long N, long long ldc, long long sC, long long batch)
{
    if (batch <= 1) return false;
    if (sC >= (M - 1) * ldc + N) return false;  // consecutive problems are disjoint ranges
    const long long reach = (M - 1) * ldc + N;  // |offset| of any two elements of one problem < reach
    for (long long d = 1; d < batch; ++d) {
        const long long x = d * sC;
        if (x >= reach) break;  // every later problem starts beyond this one's last element
        const long long q = floor_div(x, ldc);
        for (long long di = q; di <= q + 1; ++di) {
            const long long dj = x - di * ldc;
            if (di > -M && di < M && dj > -N && dj < N) return true;
        }
    }
    return false;
}

// Returns FGEMM_OK when the problem is valid.  Sets *noop when nothing has to run.
fgemm_status validate(const Problem &p, bool *noop)
{
    *noop = false;
    if (p.ta != 0 && p.ta != 1) return FGEMM_ERR_INVALID_VALUE;
    if (p.tb != 0 && p.tb != 1) return FGEMM_ERR_INVALID_VALUE;
    if (p.M < 0 || p.N < 0 || p.K < 0 || p.batch < 0) return FGEMM_ERR_INVALID_VALUE;
    const long long a_cols = p.ta ? p.M : p.K;  // stored row length of A
    const long long b_cols = p.tb ? p.K : p.N;
    if (p.lda < (a_cols > 1 ? a_cols : 1)) return FGEMM_ERR_INVALID_VALUE;
    if (p.ldb < (b_cols > 1 ? b_cols : 1)) return FGEMM_ERR_INVALID_VALUE;
    if (p.ldc < (p.N > 1 ? p.N : 1)) return FGEMM_ERR_INVALID_VALUE;
    if (p.sA < 0 || p.sB < 0 || p.sC < 0) return FGEMM_ERR_INVALID_VALUE;
    if (p.M == 0 || p.N == 0 || p.batch == 0) {
        *noop = true;
        return FGEMM_OK;
    }
    const bool products = p.K > 0 && p.alpha != 0.0f;
    if (products && (p.A == nullptr || p.B == nullptr)) return FGEMM_ERR_INVALID_VALUE;
    if (p.C == nullptr) return FGEMM_ERR_INVALID_VALUE;
    if (c_batches_overlap(p.M, p.N, p.ldc, p.sC, p.batch)) return FGEMM_ERR_INVALID_VALUE;
    // A valid call with a size the 32-bit tile and k positions cannot reach.
    if (!dims_supported(p.M, p.N, p.K)) return FGEMM_ERR_NOT_SUPPORTED;
    return FGEMM_OK;
}

bool aligned16(const void *ptr, long long ld, long long stride, int batch)
{
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    if (ld % 4 != 0) return false;
    if (batch > 1 && stride % 4 != 0) return false;
    return true;
}

fgemm_status run(int config, const Problem &p)
{
    bool noop = false;
    fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK || noop) return st;
    if (config >= NUM_CONFIGS) return FGEMM_ERR_INVALID_VALUE;

    const bool products = p.K > 0 && p.alpha != 0.0f;
    // Only operands moved by 16-byte copies need alignment: the k-major ones (A for op T,
    // B for op N).  An operand stored with k contiguous is copied element by element
    // (transposed on the way) in every configuration.
    const bool aligned = !products || ((p.ta == 0 || aligned16(p.A, p.lda, p.sA, p.batch)) &&
                                       (p.tb == 1 || aligned16(p.B, p.ldb, p.sB, p.batch)));
    if (config < 0) {
        int sms = 0;
        if (device_sm_count(&sms) != 0) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
        config = select_config(p.ta, p.tb, p.M, p.N, p.K, p.batch, aligned, sms);
    }
    if (kConfigs[config].needs_vec && !aligned) return FGEMM_ERR_NOT_SUPPORTED;

    GemmParams g{};
    g.A = products ? p.A : nullptr;
    g.B = products ? p.B : nullptr;
    g.C = p.C;
    g.bias = p.bias;
    g.row_bias = p.row_bias;
    g.lda = p.lda;
    g.ldb = p.ldb;
    g.ldc = p.ldc;
    g.strideA = p.batch > 1 ? p.sA : 0;
    g.strideB = p.batch > 1 ? p.sB : 0;
    g.strideC = p.batch > 1 ? p.sC : 0;
    g.M = p.M;
    g.N = p.N;
    g.K = products ? p.K : 0;
    g.alpha = p.alpha;
    g.beta = p.beta;
    g.relu = p.relu ? 1 : 0;
    g.c_vec = aligned16(p.C, p.ldc, p.sC, p.batch) ? 1 : 0;

    const LaunchFn *table = p.ta ? (p.tb ? kLaunchTT : kLaunchTN) : (p.tb ? kLaunchNT : kLaunchNN);
    if (table[config] == nullptr) return FGEMM_ERR_NOT_SUPPORTED;
    return table[config](g, p.batch, p.stream);
}

Problem make_problem(fgemm_op ta, fgemm_op tb, int M, int N, int K, float alpha, const float *A,
                     int lda, long long sA, const float *B, int ldb, long long sB, float beta,
                     float *C, int ldc, long long sC, int batch, const float *bias, int relu,
                     cudaStream_t stream)
{
    Problem p;
    p.ta = (int)ta;
    p.tb = (int)tb;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.A = A;
    p.lda = lda;
    p.sA = sA;
    p.B = B;
    p.ldb = ldb;
    p.sB = sB;
    p.C = C;
    p.ldc = ldc;
    p.sC = sC;
    p.batch = batch;
    p.bias = bias;
    p.relu = relu;
    p.stream = stream;
    return p;
}

}  // namespace
}  // namespace fgemm

using fgemm::make_problem;
using fgemm::run;

namespace fgemm {
namespace {

// Split-K: the K range is cut into slices of Ks (a multiple of 32) and slice s,
// covering k in [s*Ks, min(K, (s+1)*Ks)), is an independent GEMM whose unscaled
// product lands in workspace slice s (M x N, leading dimension N).  Slices of equal
// length run as one strided batch of the CUDA-core kernel, the shorter last slice as
// a second launch; a reduction kernel then sums the slices in order and applies the
// epilogue.  Nothing is atomic: the result is the same on every run.
long long splitk_slice(long long K, int splits)
{
    long long ks = (K + splits - 1) / splits;
    return (ks + 31) / 32 * 32;
}

fgemm_status run_splitk(const Problem &p, int splits, float *W, size_t ws_bytes)
{
    bool noop = false;
    fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK || noop) return st;
    if (p.batch != 1 || splits < 1 || splits > 64) return FGEMM_ERR_INVALID_VALUE;
    const bool products = p.K > 0 && p.alpha != 0.0f;
    if (splits == 1 || !products) return run(-1, p);
    const long long Ks = splitk_slice(p.K, splits);
    const int S = (int)((p.K + Ks - 1) / Ks);  // slices actually used
    const long long slice = (long long)p.M * p.N;
    if (W == nullptr || ws_bytes < sat_mul(sat_mul((size_t)S, (size_t)slice), sizeof(float)))
        return FGEMM_ERR_INVALID_VALUE;
    // Offsets of one K slice in A and B.
    const long long dA = p.ta ? Ks * p.lda : Ks;
    const long long dB = p.tb ? Ks : Ks * p.ldb;
    const long long Klast = p.K - (long long)(S - 1) * Ks;
    Problem q = p;
    q.alpha = 1.0f;
    q.beta = 0.0f;
    q.bias = nullptr;
    q.row_bias = nullptr;
    q.relu = 0;
    q.C = W;
    q.ldc = p.N;
    q.sC = slice;
    q.sA = dA;
    q.sB = dB;
    const int full = Klast == Ks ? S : S - 1;
    if (full > 0) {
        q.K = (int)Ks;
        q.batch = full;
        st = run(-1, q);
        if (st != FGEMM_OK) return st;
    }
    if (full < S) {
        q.K = (int)Klast;
        q.batch = 1;
        q.A = p.A + (long long)(S - 1) * dA;
        q.B = p.B + (long long)(S - 1) * dB;
        q.C = W + (long long)(S - 1) * slice;
        st = run(-1, q);
        if (st != FGEMM_OK) return st;
    }
    return launch_splitk_reduce(W, S, p.C, p.ldc, p.M, p.N, p.alpha, p.beta, p.bias, p.relu,
                                p.stream);
}

TcProblem tc_problem(const Problem &p)
{
    TcProblem q;
    q.ta = p.ta;
    q.tb = p.tb;
    q.M = p.M;
    q.N = p.N;
    q.K = p.K;
    q.alpha = p.alpha;
    q.beta = p.beta;
    q.A = p.A;
    q.lda = p.lda;
    q.sA = p.sA;
    q.B = p.B;
    q.ldb = p.ldb;
    q.sB = p.sB;
    q.C = p.C;
    q.ldc = p.ldc;
    q.sC = p.sC;
    q.batch = p.batch;
    q.bias = p.bias;
    q.relu = p.relu;
    return q;
}

// Staged calls: operands are first copied into the caller's workspace -- one stored
// with k contiguous (A for op N, B for op T) transposed k-major, one already k-major but
// not 16-byte aligned re-pitched into aligned rows -- and the GEMM then runs on the
// copies (op(A) = T and op(B) = N for a copied operand), whose tiles move them with
// 16-byte copies.  Workspace layout: the chosen copies packed, A's (K x ld4(M) floats a
// problem) first, B's (K x ld4(N)) at the next multiple of 256 bytes (stage_bytes).
long long ld4(long long x) { return (x + 3) / 4 * 4; }

fgemm_status run_staged(const Problem &p, int stage, void *workspace, size_t workspace_bytes)
{
    bool noop = false;
    fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK) return st;
    if (stage < -1 || stage > 3) return FGEMM_ERR_INVALID_VALUE;
    if (workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return FGEMM_ERR_INVALID_VALUE;
    if (noop) return FGEMM_OK;
    const bool products = p.K > 0 && p.alpha != 0.0f;
    if (!products) return run(-1, p);
    // An operand a batch shares (stride 0) is copied once.
    const long long problems_a = p.batch > 1 && p.sA != 0 ? p.batch : 1;
    const long long problems_b = p.batch > 1 && p.sB != 0 ? p.batch : 1;
    const size_t avail = workspace != nullptr ? workspace_bytes : 0;
    int mask = stage;
    if (stage < 0) {
        int sms = 0;
        if (device_sm_count(&sms) != 0) {
            (void)cudaGetLastError();
            return FGEMM_ERR_LAUNCH;
        }
        mask = staging_choice(p.ta, p.tb, p.M, p.N, p.K, p.batch, problems_a, problems_b,
                              aligned16(p.A, p.lda, p.sA, p.batch),
                              aligned16(p.B, p.ldb, p.sB, p.batch), avail, sms);
    } else if (stage_bytes(mask, p.M, p.N, p.K, problems_a, problems_b) > avail) {
        return FGEMM_ERR_INVALID_VALUE;  // the copies asked for do not fit
    }
    if (mask == 0) return run(-1, p);
    char *const ws = static_cast<char *>(workspace);
    Problem q = p;
    if (mask & 1) {
        float *const Ac = reinterpret_cast<float *>(ws);
        const long long ld = ld4(p.M), s = p.K * ld;
        const long long sx = problems_a > 1 ? p.sA : 0;
        st = p.ta == 0 ? launch_stage_transpose(p.A, p.lda, sx, p.M, p.K, (int)problems_a, Ac, ld,
                                                s, p.stream)
                       : launch_stage_repitch(p.A, p.lda, sx, p.K, p.M, (int)problems_a, Ac, ld, s,
                                              p.stream);
        if (st != FGEMM_OK) return st;
        q.ta = 1;
        q.A = Ac;
        q.lda = ld;
        q.sA = problems_a > 1 ? s : 0;
    }
    if (mask & 2) {
        const size_t off = (mask & 1) ? stage_bytes(1, p.M, p.N, p.K, problems_a, problems_b) : 0;
        float *const Bc = reinterpret_cast<float *>(ws + (off + 255) / 256 * 256);
        const long long ld = ld4(p.N), s = p.K * ld;
        const long long sx = problems_b > 1 ? p.sB : 0;
        st = p.tb == 1 ? launch_stage_transpose(p.B, p.ldb, sx, p.N, p.K, (int)problems_b, Bc, ld,
                                                s, p.stream)
                       : launch_stage_repitch(p.B, p.ldb, sx, p.K, p.N, (int)problems_b, Bc, ld, s,
                                              p.stream);
        if (st != FGEMM_OK) return st;
        q.tb = 0;
        q.B = Bc;
        q.ldb = ld;
        q.sB = problems_b > 1 ? s : 0;
    }
    return run(-1, q);
}

fgemm_status run_math(fgemm_math math, const Problem &p)
{
    if (math == FGEMM_MATH_FP32) return run(-1, p);
    if (math != FGEMM_MATH_TF32 && math != FGEMM_MATH_3XTF32) return FGEMM_ERR_INVALID_VALUE;
    bool noop = false;
    const fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK || noop) return st;
    const TcProblem q = tc_problem(p);
    if (!tc_supported(q)) return run(-1, p);
    return launch_tc(math == FGEMM_MATH_3XTF32 ? 3 : 1, q, p.stream);
}

// Tensor-core calls with operand staging.  The tcgen05 kernel reads an operand stored
// K-major (A for op N, B for op T) straight from its TMA tiles; an MN-major one goes
// through registers into tensor memory, and with both MN-major (TN) one of them is also
// transposed in shared memory, at about half the rate of the other layouts (TF32 at
// 4096^3: TN 335, TT 598, NN 643, NT 686 TFLOP/s).  The copies here are K-major: A as
// M x ld4(K) floats a problem, B as N x ld4(K), B's at the next multiple of 256 bytes.
size_t tc_stage_bytes(int mask, long long M, long long N, long long K, long long problems_a,
                      long long problems_b)
{
    const auto copy = [&](long long rows, long long problems) {
        return sat_mul(sat_mul(sat_mul((size_t)problems, (size_t)rows), (size_t)ld4(K)),
                       sizeof(float));
    };
    const size_t a = (mask & 1) ? copy(M, problems_a) : 0;
    const size_t b = (mask & 2) ? copy(N, problems_b) : 0;
    return b == 0 ? a : sat_add(sat_add(a, 255) / 256 * 256, b);
}

// The copies a tensor-core staged call makes by default, among those that fit: every
// operand whose alignment would keep the call off the tensor cores (then all of them or
// none: one copy alone does not help), else in a TN call the copy of A, which turns it
// into NN (measured at 4096^3 in TF32: 585 TFLOP/s with the copy against 335; copying
// both, to NT, 568), or B's copy (to TT) when only that fits.
int tc_staging_choice(int ta, int tb, long long M, long long N, long long K,
                      long long problems_a, long long problems_b, bool aligned_a,
                      bool aligned_b, size_t workspace_bytes)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const auto fits = [&](int mask) {
        return tc_stage_bytes(mask, M, N, K, problems_a, problems_b) <= workspace_bytes;
    };
    const int needed = (aligned_a ? 0 : 1) | (aligned_b ? 0 : 2);
    if (needed != 0) return fits(needed) ? needed : 0;
    if (ta == 1 && tb == 0) {
        if (fits(1)) return 1;
        if (fits(2)) return 2;
    }
    return 0;
}

fgemm_status run_math_staged(fgemm_math math, const Problem &p, int stage, void *workspace,
                             size_t workspace_bytes)
{
    if (math == FGEMM_MATH_FP32) return run_staged(p, stage, workspace, workspace_bytes);
    if (math != FGEMM_MATH_TF32 && math != FGEMM_MATH_3XTF32) return FGEMM_ERR_INVALID_VALUE;
    bool noop = false;
    fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK) return st;
    if (stage < -1 || stage > 3) return FGEMM_ERR_INVALID_VALUE;
    if (workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return FGEMM_ERR_INVALID_VALUE;
    if (noop) return FGEMM_OK;
    const bool products = p.K > 0 && p.alpha != 0.0f;
    if (!products) return run_math(math, p);
    // An operand a batch shares (stride 0) is copied once.
    const long long problems_a = p.batch > 1 && p.sA != 0 ? p.batch : 1;
    const long long problems_b = p.batch > 1 && p.sB != 0 ? p.batch : 1;
    const size_t avail = workspace != nullptr ? workspace_bytes : 0;
    int mask = stage;
    if (stage < 0) {
        mask = tc_staging_choice(p.ta, p.tb, p.M, p.N, p.K, problems_a, problems_b,
                                 aligned16(p.A, p.lda, p.sA, p.batch),
                                 aligned16(p.B, p.ldb, p.sB, p.batch), avail);
    } else if (tc_stage_bytes(mask, p.M, p.N, p.K, problems_a, problems_b) > avail) {
        return FGEMM_ERR_INVALID_VALUE;  // the copies asked for do not fit
    }
    if (mask == 0) return run_math(math, p);
    char *const ws = static_cast<char *>(workspace);
    const long long ld = ld4(p.K);
    Problem q = p;
    if (mask & 1) {
        // A as M x K rows: transposed when stored K x M, re-pitched when already K-major.
        float *const Ac = reinterpret_cast<float *>(ws);
        const long long s = (long long)p.M * ld;
        const long long sx = problems_a > 1 ? p.sA : 0;
        st = p.ta == 1 ? launch_stage_transpose(p.A, p.lda, sx, p.K, p.M, (int)problems_a, Ac, ld,
                                                s, p.stream)
                       : launch_stage_repitch(p.A, p.lda, sx, p.M, p.K, (int)problems_a, Ac, ld, s,
                                              p.stream);
        if (st != FGEMM_OK) return st;
        q.ta = 0;
        q.A = Ac;
        q.lda = ld;
        q.sA = problems_a > 1 ? s : 0;
    }
    if (mask & 2) {
        // B as N x K rows: transposed when stored K x N, re-pitched when already K-major.
        const size_t off = (mask & 1) ? tc_stage_bytes(1, p.M, p.N, p.K, problems_a, problems_b) : 0;
        float *const Bc = reinterpret_cast<float *>(ws + (off + 255) / 256 * 256);
        const long long s = (long long)p.N * ld;
        const long long sx = problems_b > 1 ? p.sB : 0;
        st = p.tb == 0 ? launch_stage_transpose(p.B, p.ldb, sx, p.K, p.N, (int)problems_b, Bc, ld,
                                                s, p.stream)
                       : launch_stage_repitch(p.B, p.ldb, sx, p.N, p.K, (int)problems_b, Bc, ld, s,
                                              p.stream);
        if (st != FGEMM_OK) return st;
        q.tb = 1;
        q.B = Bc;
        q.ldb = ld;
        q.sB = problems_b > 1 ? s : 0;
    }
    return run_math(math, q);
}

}  // namespace

fgemm_status splitk_plan(int ta, int tb, int M, int N, int K, float alpha, const float *A, int lda,
                         const float *B, int ldb, float beta, float *C, int ldc, int splits,
                         size_t *workspace_bytes)
{
    *workspace_bytes = 0;
    const Problem p = make_problem((fgemm_op)ta, (fgemm_op)tb, M, N, K, alpha, A, lda, 0, B, ldb,
                                   0, beta, C, ldc, 0, 1, nullptr, 0, nullptr);
    bool noop = false;
    const fgemm_status st = validate(p, &noop);
    if (st != FGEMM_OK || noop) return st;
    if (splits < 1 || splits > 64) return FGEMM_ERR_INVALID_VALUE;
    const bool products = p.K > 0 && p.alpha != 0.0f;
    if (splits == 1 || !products) return FGEMM_OK;
    const long long Ks = splitk_slice(p.K, splits);
    const long long S = (p.K + Ks - 1) / Ks;
    *workspace_bytes = sat_mul(sat_mul(sat_mul((size_t)S, (size_t)p.M), (size_t)p.N), sizeof(float));
    return FGEMM_OK;
}

namespace {

}  // namespace
}  // namespace fgemm

extern "C" {

fgemm_status fgemm_sgemm(fgemm_op transa, fgemm_op transb, int M, int N, int K, float alpha,
                         const float *A, int lda, const float *B, int ldb, float beta, float *C,
                         int ldc, cudaStream_t stream)
{
    return run(-1, make_problem(transa, transb, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc,
                                0, 1, nullptr, 0, stream));
}

fgemm_status fgemm_sgemm_bias_relu(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                   float alpha, const float *A, int lda, const float *B, int ldb,
                                   float beta, float *C, int ldc, const float *bias,
                                   int apply_relu, cudaStream_t stream)
{
    return run(-1, make_problem(transa, transb, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc,
                                0, 1, bias, apply_relu, stream));
}

fgemm_status fgemm_sgemm_row_bias_relu(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                       float alpha, const float *A, int lda, const float *B,
                                       int ldb, float beta, float *C, int ldc,
                                       const float *row_bias, int apply_relu, cudaStream_t stream)
{
    fgemm::Problem p = make_problem(transa, transb, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C,
                                    ldc, 0, 1, nullptr, apply_relu, stream);
    p.row_bias = row_bias;
    return run(-1, p);
}

fgemm_status fgemm_sgemm_strided_batched(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                         float alpha, const float *A, int lda, long long strideA,
                                         const float *B, int ldb, long long strideB, float beta,
                                         float *C, int ldc, long long strideC, int batch,
                                         cudaStream_t stream)
{
    return run(-1, make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                                beta, C, ldc, strideC, batch, nullptr, 0, stream));
}

fgemm_status fgemm_gemm_explicit(int config, fgemm_op transa, fgemm_op transb, int M, int N,
                                 int K, float alpha, const float *A, int lda, long long strideA,
                                 const float *B, int ldb, long long strideB, float beta, float *C,
                                 int ldc, long long strideC, int batch, const float *bias,
                                 int apply_relu, cudaStream_t stream)
{
    return run(config < 0 ? -1 : config,
               make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta,
                            C, ldc, strideC, batch, bias, apply_relu, stream));
}

fgemm_status fgemm_gemm_math(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N,
                             int K, float alpha, const float *A, int lda, long long strideA,
                             const float *B, int ldb, long long strideB, float beta, float *C,
                             int ldc, long long strideC, int batch, const float *bias,
                             int apply_relu, cudaStream_t stream)
{
    return fgemm::run_math(math, make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B,
                                              ldb, strideB, beta, C, ldc, strideC, batch, bias,
                                              apply_relu, stream));
}

fgemm_status fgemm_device_status(int clear) { return fgemm::tc_device_status(clear); }

int fgemm_math_supported(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N, int K,
                         float alpha, const float *A, int lda, long long strideA, const float *B,
                         int ldb, long long strideB, int batch)
{
    if (math == FGEMM_MATH_FP32) return 1;
    if (math != FGEMM_MATH_TF32 && math != FGEMM_MATH_3XTF32) return -1;
    if (!fgemm::dims_supported(M, N, K)) return 0;  // the call runs nothing
    const fgemm::Problem p = make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb,
                                          strideB, 0.0f, nullptr, 1, 0, batch, nullptr, 0, nullptr);
    return fgemm::tc_supported(fgemm::tc_problem(p)) ? 1 : 0;
}

size_t fgemm_splitk_workspace_size(int M, int N, int K, int splits)
{
    if (M < 0 || N < 0 || K < 0 || splits < 1 || splits > 64) return 0;
    if (K == 0) return 0;
    const long long Ks = fgemm::splitk_slice(K, splits);
    const long long S = (K + Ks - 1) / Ks;
    return fgemm::sat_mul(fgemm::sat_mul(fgemm::sat_mul((size_t)S, (size_t)M), (size_t)N),
                          sizeof(float));
}

fgemm_status fgemm_sgemm_splitk(fgemm_op transa, fgemm_op transb, int M, int N, int K, float alpha,
                                const float *A, int lda, const float *B, int ldb, float beta,
                                float *C, int ldc, const float *bias, int apply_relu, int splits,
                                float *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return fgemm::run_splitk(make_problem(transa, transb, M, N, K, alpha, A, lda, 0, B, ldb, 0,
                                          beta, C, ldc, 0, 1, bias, apply_relu, stream),
                             splits, workspace, workspace_bytes);
}

size_t fgemm_staged_workspace_size(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                   int batch)
{
    if ((transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M <= 0 || N <= 0 || K <= 0 ||
        batch <= 0)
        return 0;
    return fgemm::stage_bytes(3, M, N, K, batch, batch);
}

int fgemm_staged_choice(fgemm_op transa, fgemm_op transb, int M, int N, int K, int batch,
                        int shared_a, int shared_b, int aligned_a, int aligned_b,
                        size_t workspace_bytes, int num_sms)
{
    if ((transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M < 0 || N < 0 || K < 0 ||
        batch < 0 || num_sms < 1)
        return -1;
    const long long problems_a = batch > 1 && !shared_a ? batch : 1;
    const long long problems_b = batch > 1 && !shared_b ? batch : 1;
    return fgemm::staging_choice((int)transa, (int)transb, M, N, K, batch, problems_a,
                                 problems_b, aligned_a != 0, aligned_b != 0, workspace_bytes,
                                 num_sms);
}

fgemm_status fgemm_sgemm_staged(fgemm_op transa, fgemm_op transb, int M, int N, int K,
                                float alpha, const float *A, int lda, long long strideA,
                                const float *B, int ldb, long long strideB, float beta, float *C,
                                int ldc, long long strideC, int batch, const float *bias,
                                int apply_relu, int stage, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream)
{
    return fgemm::run_staged(make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B,
                                          ldb, strideB, beta, C, ldc, strideC, batch, bias,
                                          apply_relu, stream),
                             stage, workspace, workspace_bytes);
}

size_t fgemm_math_staged_workspace_size(fgemm_math math, fgemm_op transa, fgemm_op transb, int M,
                                        int N, int K, int batch)
{
    if (math == FGEMM_MATH_FP32) return fgemm_staged_workspace_size(transa, transb, M, N, K, batch);
    if ((math != FGEMM_MATH_TF32 && math != FGEMM_MATH_3XTF32) ||
        (transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M <= 0 || N <= 0 || K <= 0 ||
        batch <= 0)
        return 0;
    return fgemm::tc_stage_bytes(3, M, N, K, batch, batch);
}

int fgemm_math_staged_choice(fgemm_math math, fgemm_op transa, fgemm_op transb, int M, int N,
                             int K, int batch, int shared_a, int shared_b, int aligned_a,
                             int aligned_b, size_t workspace_bytes, int num_sms)
{
    if (math == FGEMM_MATH_FP32)
        return fgemm_staged_choice(transa, transb, M, N, K, batch, shared_a, shared_b, aligned_a,
                                   aligned_b, workspace_bytes, num_sms);
    if ((math != FGEMM_MATH_TF32 && math != FGEMM_MATH_3XTF32) ||
        (transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M < 0 || N < 0 || K < 0 ||
        batch < 0 || num_sms < 1)
        return -1;
    const long long problems_a = batch > 1 && !shared_a ? batch : 1;
    const long long problems_b = batch > 1 && !shared_b ? batch : 1;
    return fgemm::tc_staging_choice((int)transa, (int)transb, M, N, K, problems_a, problems_b,
                                    aligned_a != 0, aligned_b != 0, workspace_bytes);
}

fgemm_status fgemm_gemm_math_staged(fgemm_math math, fgemm_op transa, fgemm_op transb, int M,
                                    int N, int K, float alpha, const float *A, int lda,
                                    long long strideA, const float *B, int ldb, long long strideB,
                                    float beta, float *C, int ldc, long long strideC, int batch,
                                    const float *bias, int apply_relu, int stage, void *workspace,
                                    size_t workspace_bytes, cudaStream_t stream)
{
    return fgemm::run_math_staged(math,
                                  make_problem(transa, transb, M, N, K, alpha, A, lda, strideA, B,
                                               ldb, strideB, beta, C, ldc, strideC, batch, bias,
                                               apply_relu, stream),
                                  stage, workspace, workspace_bytes);
}

void fgemm_debug_withhold_tensor_core(int k_block, long long wait_limit_ns)
{
    fgemm::tc_debug_withhold(k_block, wait_limit_ns);
}

const char *fgemm_status_string(fgemm_status status)
{
    switch (status) {
    case FGEMM_OK: return "FGEMM_OK: success";
    case FGEMM_ERR_INVALID_VALUE: return "FGEMM_ERR_INVALID_VALUE: an argument is out of range";
    case FGEMM_ERR_LAUNCH: return "FGEMM_ERR_LAUNCH: a CUDA call or kernel launch failed";
    case FGEMM_ERR_NOT_SUPPORTED:
        return "FGEMM_ERR_NOT_SUPPORTED: the configuration cannot run this call";
    case FGEMM_ERR_TIMEOUT:
        return "FGEMM_ERR_TIMEOUT: a tensor-core kernel gave up waiting; its output is undefined";
    }
    return "unknown fgemm_status";
}

int fgemm_num_configs(void) { return fgemm::NUM_CONFIGS; }

const char *fgemm_config_name(int config)
{
    if (config < 0 || config >= fgemm::NUM_CONFIGS) return nullptr;
    return fgemm::kConfigs[config].name;
}

int fgemm_launch_count(int config, fgemm_op transa, fgemm_op transb, int M, int N, int K,
                       int batch, int aligned, int num_sms)
{
    if ((transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M < 0 || N < 0 || K < 0 || batch < 0 ||
        config >= fgemm::NUM_CONFIGS || num_sms < 1)
        return -1;
    if (M == 0 || N == 0 || batch == 0) return 0;
    // Calls the library refuses (FGEMM_ERR_NOT_SUPPORTED) launch nothing: a size above
    // FGEMM_MAX_DIM, or a tile grid larger than one launch takes.
    if (!fgemm::dims_supported(M, N, K)) return 0;
    if (config < 0)
        config = fgemm::select_config((int)transa, (int)transb, M, N, K, batch, aligned != 0,
                                      num_sms);
    const long long bm = fgemm::kConfigs[config].bm, bn = fgemm::kConfigs[config].bn;
    const long long tiles = ((long long)M + bm - 1) / bm * (((long long)N + bn - 1) / bn);
    if (config == fgemm::CFG_128x128_SPLIT || config == fgemm::CFG_128x128_KSPLIT ||
        config == fgemm::CFG_128x128_KCHAIN) {
        const long long total = tiles * batch;
        const long long r = total % num_sms;
        const long long tail_ctas = config == fgemm::CFG_128x128_KCHAIN ? 1 : 4;
        if (total - r > INT_MAX || tail_ctas * r > INT_MAX) return 0;
        const int tail = config == fgemm::CFG_128x128_KCHAIN
                             ? fgemm::kchain_slices((int)transa, (int)transb, r, K, num_sms)
                             : 1;
        return (total - r > 0 ? 1 : 0) + (r > 0 ? tail : 0);
    }
    if (tiles > INT_MAX) return 0;
    // TT whole 128 x 128 tiles run in linear-order launches of up to INT_MAX CTAs; the
    // other configurations in one launch per 65535 problems
    if ((config == fgemm::CFG_128x128 || config == fgemm::CFG_128x128_SCALAR) &&
        transa == FGEMM_OP_T && transb == FGEMM_OP_T) {
        const long long per_launch = INT_MAX / tiles;
        return (int)((batch + per_launch - 1) / per_launch);
    }
    return (batch + 65534) / 65535;
}

int fgemm_select_config(fgemm_op transa, fgemm_op transb, int M, int N, int K, int batch,
                        int aligned, int num_sms)
{
    if ((transa != FGEMM_OP_N && transa != FGEMM_OP_T) ||
        (transb != FGEMM_OP_N && transb != FGEMM_OP_T) || M < 0 || N < 0 || K < 0 || batch < 0)
        return -1;
    return fgemm::select_config((int)transa, (int)transb, M, N, K, batch, aligned != 0, num_sms);
}

}  // extern "C"
