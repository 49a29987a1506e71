/* A plain C caller of the library (no Python, no PyTorch): cross-entropy of
 * N rows of V equal fp32 logits on the GPU through ce_fwd_bwd, checked
 * against the closed form (loss ln V per valid row, gradient 1/(n_valid V)
 * - [j = y]/n_valid under the mean).  Built and run by tests/test_c_abi_gpu.py.
 * Exit status 0 when every check passes. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "vlmce.h"

#define CHECK(c)                                                              \
    do {                                                                      \
        if (!(c)) {                                                           \
            fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__);    \
            return 1;                                                         \
        }                                                                     \
    } while (0)

int main(void) {
    const int64_t N = 4, V = 1000, stride = 1003;
    float *hx = (float *)calloc((size_t)(N * stride), sizeof(float));
    int64_t hy[4] = {7, -100, 999, 0};
    float *x = NULL, *loss = NULL, *reduced = NULL;
    int64_t *y = NULL, *amax = NULL, *counts = NULL;
    void *ws = NULL;
    const size_t wsb = vlmce_ce_workspace_bytes(N, V, VLMCE_F32);
    CHECK(hx != NULL && wsb > 0);
    CHECK(cudaMalloc((void **)&x, (size_t)(N * stride) * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void **)&y, sizeof(hy)) == cudaSuccess);
    CHECK(cudaMalloc((void **)&loss, (size_t)N * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void **)&amax, (size_t)N * sizeof(int64_t)) == cudaSuccess);
    CHECK(cudaMalloc((void **)&reduced, 2 * sizeof(float)) == cudaSuccess);
    CHECK(cudaMalloc((void **)&counts, 4 * sizeof(int64_t)) == cudaSuccess);
    CHECK(cudaMalloc(&ws, wsb) == cudaSuccess);
    CHECK(cudaMemcpy(x, hx, (size_t)(N * stride) * sizeof(float), cudaMemcpyHostToDevice) ==
          cudaSuccess);
    CHECK(cudaMemcpy(y, hy, sizeof(hy), cudaMemcpyHostToDevice) == cudaSuccess);

    /* an argument error is returned before anything is enqueued */
    CHECK(ce_fwd_bwd(x, VLMCE_F32, y, N, V, V - 1, -100, 0.f, 0.f, VLMCE_MEAN, 1.f, loss, amax,
                     reduced, counts, ws, wsb, NULL) == VLMCE_ERR_INVALID_ARG);
    CHECK(ce_fwd_bwd(x, VLMCE_F32, y, N, V, stride, -100, 0.f, 0.f, VLMCE_MEAN, 1.f, loss, amax,
                     reduced, counts, ws, wsb, NULL) == VLMCE_OK);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);

    float hl[4], hr[2];
    int64_t ha[4], hc[4];
    CHECK(cudaMemcpy(hl, loss, sizeof(hl), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(ha, amax, sizeof(ha), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hr, reduced, sizeof(hr), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hc, counts, sizeof(hc), cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hx, x, (size_t)(N * stride) * sizeof(float), cudaMemcpyDeviceToHost) ==
          cudaSuccess);

    const double lnV = log((double)V);
    const int64_t n_valid = 3;
    for (int r = 0; r < N; ++r) {
        CHECK(ha[r] == 0); /* equal logits: the smallest column */
        CHECK(fabs(hl[r] - (hy[r] == -100 ? 0.0 : lnV)) < 1e-4);
        for (int64_t j = 0; j < V; ++j) {
            const double want =
                hy[r] == -100 ? 0.0 : (1.0 / (double)V - (j == hy[r] ? 1.0 : 0.0)) / (double)n_valid;
            CHECK(fabs(hx[r * stride + j] - want) <= 1e-6 * fabs(want) + 1e-9);
        }
        for (int64_t j = V; j < stride; ++j) CHECK(hx[r * stride + j] == 0.f); /* padding */
    }
    CHECK(hc[0] == n_valid && hc[1] == 1 && hc[2] == 0 && hc[3] == 0); /* row 3: argmax 0 = label */
    CHECK(fabs(hr[0] - lnV) < 1e-4);
    CHECK(fabs(hr[1] - 1.0 / 3.0) < 1e-6);
    printf("c abi ok: loss %.6f (ln V %.6f)\n", hr[0], lnV);
    return 0;
}
