/*
 * A C99 client of the fgemm C ABI (include/fgemm.h), with no Python and no C++: it
 * shows that the header compiles as C and that a C program links and calls the
 * library.  tests/test_c_abi.py builds and runs it.
 *
 *   c_abi_client host
 *       Host-only checks: the configuration table, the size queries, and argument
 *       validation before any CUDA call (fake pointers, never dereferenced).  Prints
 *       "ok host".
 *
 *   c_abi_client run IN OUT
 *       Reads one problem from IN -- seven int32 (transa, transb, M, N, K, has_bias,
 *       apply_relu), two float32 (alpha, beta), then op(A) as stored (M x K, or K x M
 *       for transa = T), B as stored, C0 (M x N) and, with has_bias, the bias (N
 *       floats) -- copies it to the device, calls fgemm_sgemm_bias_relu with tight
 *       leading dimensions on a stream of its own, and writes C (M x N float32) to OUT.
 *       Prints "ok run".
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fgemm.h"

static int fail(const char *what)
{
    fprintf(stderr, "FAIL: %s\n", what);
    return 1;
}

static int host_checks(void)
{
    float *fake = (float *)(size_t)0x10000; /* validation never dereferences it */
    int n = fgemm_num_configs(), i;
    if (n < 1) return fail("fgemm_num_configs");
    for (i = 0; i < n; ++i)
        if (fgemm_config_name(i) == NULL) return fail("fgemm_config_name");
    if (fgemm_config_name(n) != NULL) return fail("fgemm_config_name past the table");
    if (fgemm_select_config(FGEMM_OP_N, FGEMM_OP_N, 4096, 4096, 4096, 1, 1, 152) < 0)
        return fail("fgemm_select_config");
    if (fgemm_staged_workspace_size(FGEMM_OP_N, FGEMM_OP_N, 4096, 4096, 4096, 1) !=
        (size_t)2 * 4096 * 4096 * sizeof(float))
        return fail("fgemm_staged_workspace_size");
    if (fgemm_splitk_workspace_size(64, 64, 256, 4) != (size_t)4 * 64 * 64 * sizeof(float))
        return fail("fgemm_splitk_workspace_size");
    if (fgemm_sgemm(FGEMM_OP_N, FGEMM_OP_N, 4, 4, 4, 1.0f, fake, 3, fake, 4, 0.0f, fake, 4, NULL) !=
        FGEMM_ERR_INVALID_VALUE)
        return fail("lda below K accepted");
    if (fgemm_sgemm(FGEMM_OP_N, FGEMM_OP_N, FGEMM_MAX_DIM + 1, 4, 4, 1.0f, fake, 4, fake, 4, 0.0f,
                    fake, 4, NULL) != FGEMM_ERR_NOT_SUPPORTED)
        return fail("size above FGEMM_MAX_DIM accepted");
    if (fgemm_sgemm(FGEMM_OP_N, FGEMM_OP_N, 0, 4, 4, 1.0f, NULL, 4, NULL, 4, 0.0f, NULL, 4, NULL) !=
        FGEMM_OK)
        return fail("empty problem");
    if (strncmp(fgemm_status_string(FGEMM_ERR_INVALID_VALUE), "FGEMM_", 6) != 0)
        return fail("fgemm_status_string");
    puts("ok host");
    return 0;
}

static int read_all(FILE *f, void *p, size_t bytes)
{
    return fread(p, 1, bytes, f) == bytes ? 0 : -1;
}

static int run(const char *in_path, const char *out_path)
{
    FILE *f = fopen(in_path, "rb");
    int hdr[7];
    float ab[2];
    if (f == NULL || read_all(f, hdr, sizeof(hdr)) || read_all(f, ab, sizeof(ab)))
        return fail("reading the problem header");
    {
        const fgemm_op ta = hdr[0] ? FGEMM_OP_T : FGEMM_OP_N, tb = hdr[1] ? FGEMM_OP_T : FGEMM_OP_N;
        const int M = hdr[2], N = hdr[3], K = hdr[4], has_bias = hdr[5], relu = hdr[6];
        const size_t na = (size_t)M * K, nb = (size_t)K * N, nc = (size_t)M * N;
        const int lda = ta == FGEMM_OP_T ? M : K, ldb = tb == FGEMM_OP_T ? K : N;
        float *h = (float *)malloc((na + nb + nc + (size_t)N) * sizeof(float));
        float *dA = NULL, *dB = NULL, *dC = NULL, *dbias = NULL;
        cudaStream_t stream = NULL;
        fgemm_status st;
        FILE *o;
        if (h == NULL) return fail("host memory");
        if (read_all(f, h, (na + nb + nc) * sizeof(float)) ||
            (has_bias && read_all(f, h + na + nb + nc, (size_t)N * sizeof(float))))
            return fail("reading the operands");
        fclose(f);
        if (cudaMalloc((void **)&dA, na * sizeof(float)) != cudaSuccess ||
            cudaMalloc((void **)&dB, nb * sizeof(float)) != cudaSuccess ||
            cudaMalloc((void **)&dC, nc * sizeof(float)) != cudaSuccess ||
            cudaMalloc((void **)&dbias, (size_t)N * sizeof(float)) != cudaSuccess ||
            cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess)
            return fail("device memory or stream");
        cudaMemcpy(dA, h, na * sizeof(float), cudaMemcpyHostToDevice);
        cudaMemcpy(dB, h + na, nb * sizeof(float), cudaMemcpyHostToDevice);
        cudaMemcpy(dC, h + na + nb, nc * sizeof(float), cudaMemcpyHostToDevice);
        if (has_bias)
            cudaMemcpy(dbias, h + na + nb + nc, (size_t)N * sizeof(float), cudaMemcpyHostToDevice);
        st = fgemm_sgemm_bias_relu(ta, tb, M, N, K, ab[0], dA, lda, dB, ldb, ab[1], dC, N,
                                   has_bias ? dbias : NULL, relu, stream);
        if (st != FGEMM_OK) {
            fprintf(stderr, "%s\n", fgemm_status_string(st));
            return fail("fgemm_sgemm_bias_relu");
        }
        if (cudaStreamSynchronize(stream) != cudaSuccess) return fail("the call's stream");
        if (cudaMemcpy(h, dC, nc * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
            return fail("copying C back");
        o = fopen(out_path, "wb");
        if (o == NULL || fwrite(h, sizeof(float), nc, o) != nc) return fail("writing C");
        fclose(o);
        cudaFree(dA);
        cudaFree(dB);
        cudaFree(dC);
        cudaFree(dbias);
        cudaStreamDestroy(stream);
        free(h);
    }
    puts("ok run");
    return 0;
}

int main(int argc, char **argv)
{
    if (argc == 2 && strcmp(argv[1], "host") == 0) return host_checks();
    if (argc == 4 && strcmp(argv[1], "run") == 0) return run(argv[2], argv[3]);
    fprintf(stderr, "usage: %s host | run IN OUT\n", argv[0]);
    return 2;
}
