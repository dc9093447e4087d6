// splitk_reduce.cu -- second half of the split-K GEMM: sum the per-slice partial
// products in slice order and apply the epilogue.
//
//   C[i][j] = act( alpha * sum_{s<S} W[s][i][j] + beta * C[i][j] + bias[j] )
//
// W holds S slices of M x N (leading dimension N, slice stride M*N).  The sum runs
// s = 0, 1, ..., S-1 for every element, so the result does not depend on the launch.
// Memory-bound: each thread handles 4 consecutive columns (16-byte loads and stores
// when C allows them), a grid-stride loop over the rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "fgemm_internal.h"

namespace fgemm {
namespace {

__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ W, int S,
                                                            float *C, long long ldc, int M, int N,
                                                            float alpha, float beta,
                                                            const float *__restrict__ bias,
                                                            int relu, int c_vec)
{
    const long long slice = (long long)M * N;
    const int groups = (N + 3) / 4;
    const long long total = (long long)M * groups;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(g / groups);
        const int j0 = (int)(g % groups) * 4;
        const float *w = W + (long long)i * N + j0;
        float *c = C + (long long)i * ldc + j0;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const bool full = j0 + 3 < N;
        if (full && (N % 4) == 0) {
            for (int s = 0; s < S; ++s) {
                const float4 v = *reinterpret_cast<const float4 *>(w + s * slice);
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
        } else {
            for (int s = 0; s < S; ++s)
                for (int e = 0; e < 4 && j0 + e < N; ++e) acc[e] += w[s * slice + e];
        }
        float v[4];
        for (int e = 0; e < 4; ++e) v[e] = alpha * acc[e];
        if (full && c_vec) {
            if (beta != 0.0f) {
                const float4 o = *reinterpret_cast<const float4 *>(c);
                v[0] = fmaf(beta, o.x, v[0]);
                v[1] = fmaf(beta, o.y, v[1]);
                v[2] = fmaf(beta, o.z, v[2]);
                v[3] = fmaf(beta, o.w, v[3]);
            }
            for (int e = 0; e < 4; ++e) {
                if (bias) v[e] += __ldg(bias + j0 + e);
                if (relu) v[e] = fmaxf(v[e], 0.0f);
            }
            *reinterpret_cast<float4 *>(c) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            for (int e = 0; e < 4 && j0 + e < N; ++e) {
                float o = v[e];
                if (beta != 0.0f) o = fmaf(beta, c[e], o);
                if (bias) o += __ldg(bias + j0 + e);
                if (relu) o = fmaxf(o, 0.0f);
                c[e] = o;
            }
        }
    }
}

}  // namespace

fgemm_status launch_splitk_reduce(const float *W, int S, float *C, long long ldc, int M, int N,
                                  float alpha, float beta, const float *bias, int relu,
                                  cudaStream_t stream)
{
    int sms = 0;
    if (device_sm_count(&sms) != 0) {
        (void)cudaGetLastError();
        return FGEMM_ERR_LAUNCH;
    }
    const long long groups = (long long)M * ((N + 3) / 4);
    long long blocks = (groups + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0) ? 1 : 0;
    splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(W, S, C, ldc, M, N, alpha, beta,
                                                               bias, relu, c_vec);
    return cudaGetLastError() == cudaSuccess ? FGEMM_OK : FGEMM_ERR_LAUNCH;
}

}  // namespace fgemm
