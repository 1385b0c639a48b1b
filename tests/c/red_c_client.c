/*
 * A plain C99 client of libred.so: includes only red.h and the CUDA runtime
 * API, allocates its own device buffers, calls the library on its own
 * stream and checks the results against closed forms.  Built and run by
 * tests/test_gpu_c_client.py; exit status 0 and "ok" on success.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "red.h"

#define CHECK_CUDA(call)                                                                 \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

#define CHECK_RED(call)                                                                  \
    do {                                                                                 \
        int s_ = (call);                                                                 \
        if (s_ != RED_OK) {                                                              \
            fprintf(stderr, "%s:%d %s -> %d (%s)\n", __FILE__, __LINE__, #call, s_, red_last_error()); \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

#define EXPECT(cond)                                                                     \
    do {                                                                                 \
        if (!(cond)) {                                                                   \
            fprintf(stderr, "%s:%d expected %s\n", __FILE__, __LINE__, #cond);           \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

int main(void)
{
    cudaStream_t s;
    CHECK_CUDA(cudaStreamCreate(&s));
    red_stream_t rs = (red_stream_t)s;
    EXPECT(red_version() >= 1);

    /* full reduction of 2^24 + 3 integer-valued floats (i mod 7) - 3 */
    const int64_t n = (1 << 24) + 3;
    float *hx = (float *)malloc((size_t)n * sizeof(float));
    double want = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        hx[i] = (float)(i % 7) - 3.0f;
        want += hx[i];
    }
    float *dx, *dout;
    CHECK_CUDA(cudaMalloc((void **)&dx, (size_t)n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&dout, 3 * sizeof(float)));
    CHECK_CUDA(cudaMemcpyAsync(dx, hx, (size_t)n * sizeof(float), cudaMemcpyHostToDevice, s));
    CHECK_RED(red_full(RED_SUM, dx, n, dout + 0, rs));
    CHECK_RED(red_full(RED_MAX, dx, n, dout + 1, rs));
    CHECK_RED(red_full(RED_MIN, dx, n, dout + 2, rs));
    float got[3];
    CHECK_CUDA(cudaMemcpyAsync(got, dout, sizeof got, cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    EXPECT((double)got[0] == want); /* integer partial sums: exact */
    EXPECT(got[1] == 3.0f && got[2] == -3.0f);

    /* per-row sums of a 1000 x 777 view of the same data, with accum */
    const int64_t rows = 1000, len = 777;
    float *drow;
    CHECK_CUDA(cudaMalloc((void **)&drow, (size_t)rows * sizeof(float)));
    CHECK_CUDA(cudaMemsetAsync(drow, 0, (size_t)rows * sizeof(float), s));
    CHECK_RED(red_rows(RED_SUM, dx, rows, len, 1, drow, rs));
    CHECK_RED(red_rows(RED_SUM, dx, rows, len, 1, drow, rs));
    float *hrow = (float *)malloc((size_t)rows * sizeof(float));
    CHECK_CUDA(cudaMemcpyAsync(hrow, drow, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    for (int64_t r = 0; r < rows; ++r) {
        double w = 0.0;
        for (int64_t k = 0; k < len; ++k)
            w += hx[r * len + k];
        EXPECT((double)hrow[r] == 2.0 * w);
    }

    /* TCOLPROD, int32: a column of 31 twos wraps to INT32_MIN, of 32 to 0 */
    const int64_t R = 32, C = 40;
    int32_t hm[32 * 40];
    for (int64_t i = 0; i < R * C; ++i)
        hm[i] = 2;
    int32_t *dm, *dp, hp[40];
    CHECK_CUDA(cudaMalloc((void **)&dm, sizeof hm));
    CHECK_CUDA(cudaMalloc((void **)&dp, sizeof hp));
    CHECK_CUDA(cudaMemcpyAsync(dm, hm, sizeof hm, cudaMemcpyHostToDevice, s));
    CHECK_RED(red_colprod(RED_I32, dm, R - 1, C, dp, rs));
    CHECK_CUDA(cudaMemcpyAsync(hp, dp, sizeof hp, cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    for (int64_t j = 0; j < C; ++j)
        EXPECT(hp[j] == INT32_MIN);
    CHECK_RED(red_colprod(RED_I32, dm, R, C, dp, rs));
    CHECK_CUDA(cudaMemcpyAsync(hp, dp, sizeof hp, cudaMemcpyDeviceToHost, s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    for (int64_t j = 0; j < C; ++j)
        EXPECT(hp[j] == 0);

    /* errors are reported on the host, before any launch */
    EXPECT(red_full(7, dx, n, dout, rs) == RED_EINVAL);
    EXPECT(strlen(red_last_error()) > 0);
    EXPECT(red_rows(RED_MAX, dx, 3, 0, 0, drow, rs) == RED_EINVAL);

    cudaFree(dx);
    cudaFree(dout);
    cudaFree(drow);
    cudaFree(dm);
    cudaFree(dp);
    free(hx);
    free(hrow);
    CHECK_RED(red_release_workspace());
    CHECK_CUDA(cudaStreamDestroy(s));
    printf("ok\n");
    return 0;
}
