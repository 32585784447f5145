/*
 * A plain C consumer of include/mt_norm.h: the library used with no Python and no torch.
 * RMSNorm forward and backward on one constant row, checked against closed forms:
 *   x_j = 2 (j < D), gamma_j = 1 + j/D: ms = 4, rstd = 1/sqrt(4 + eps), y_j = 2 rstd gamma_j;
 *   dY = gamma: g = gamma^2, xhat = 2 rstd, c = mean(g xhat) = 2 rstd mean(gamma^2),
 *   dX_j = rstd (g_j - xhat c) = rstd (gamma_j^2 - 4 rstd^2 mean(gamma^2)),
 *   dgamma_j = dY_j xhat = 2 rstd gamma_j.
 * Exit status 0 when every value is within fp16 rounding of its closed form.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "mt_norm.h"

/* IEEE binary16 <-> float for this test's values (normal numbers only). */
static uint16_t to_half(float f) {
    union { float f; uint32_t u; } v = {f};
    uint32_t sign = (v.u >> 16) & 0x8000u;
    int32_t e = (int32_t)((v.u >> 23) & 0xff) - 127 + 15;
    uint32_t m = v.u & 0x7fffffu;
    uint32_t h = sign | ((uint32_t)e << 10) | (m >> 13);
    uint32_t rem = m & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u; /* nearest even */
    return (uint16_t)h;
}
static float from_half(uint16_t h) {
    int32_t e = (int32_t)((h >> 10) & 0x1f) - 15 + 127;
    union { uint32_t u; float f; } v;
    v.u = ((uint32_t)(h & 0x8000u) << 16) | ((uint32_t)e << 23) | ((uint32_t)(h & 0x3ffu) << 13);
    return v.f;
}

#define CHECK(x) do { if (!(x)) { fprintf(stderr, "check failed: %s (line %d)\n", #x, __LINE__); return 1; } } while (0)

int main(void) {
    const int64_t N = 3, D = 1000;
    const float eps = 1e-5f;
    uint16_t *hx = malloc(N * D * 2), *hg = malloc(D * 2), *hy = malloc(N * D * 2), *hdx = malloc(N * D * 2);
    float *hr = malloc(N * 4), *hdg = malloc(D * 4);
    for (int64_t j = 0; j < D; ++j) hg[j] = to_half(1.0f + (float)j / (float)D);
    for (int64_t i = 0; i < N * D; ++i) hx[i] = to_half(2.0f);
    void *x, *g, *y, *dy, *dx;
    float *r, *dg;
    CHECK(cudaMalloc(&x, N * D * 2) == cudaSuccess && cudaMalloc(&g, D * 2) == cudaSuccess);
    CHECK(cudaMalloc(&y, N * D * 2) == cudaSuccess && cudaMalloc(&dy, N * D * 2) == cudaSuccess);
    CHECK(cudaMalloc(&dx, N * D * 2) == cudaSuccess && cudaMalloc((void **)&r, N * 4) == cudaSuccess);
    CHECK(cudaMalloc((void **)&dg, D * 4) == cudaSuccess);
    CHECK(cudaMemcpy(x, hx, N * D * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(g, hg, D * 2, cudaMemcpyHostToDevice) == cudaSuccess);
    for (int64_t i = 0; i < N; ++i)  /* dY = gamma in every row */
        CHECK(cudaMemcpy((char *)dy + i * D * 2, hg, D * 2, cudaMemcpyHostToDevice) == cudaSuccess);

    CHECK(mt_rmsnorm_forward(x, g, y, r, N, D, eps, NULL) == MT_OK);
    CHECK(mt_rmsnorm_backward(x, g, dy, r, dx, dg, N, D, NULL) == MT_OK);
    CHECK(mt_rmsnorm_forward(x, g, x, r, N, D, eps, NULL) == MT_ERR_INVALID_ARG); /* in place */
    CHECK(mt_rmsnorm_forward(x, g, y, r, N, MT_MAX_COLS + 1, eps, NULL) == MT_ERR_UNSUPPORTED);
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    CHECK(cudaMemcpy(hy, y, N * D * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hdx, dx, N * D * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hr, r, N * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    CHECK(cudaMemcpy(hdg, dg, D * 4, cudaMemcpyDeviceToHost) == cudaSuccess);

    const double rstd = 1.0 / sqrt(4.0 + (double)eps);
    double mg2 = 0.0;
    for (int64_t j = 0; j < D; ++j) { double gj = from_half(hg[j]); mg2 += gj * gj; }
    mg2 /= (double)D;
    for (int64_t i = 0; i < N; ++i) {
        CHECK(fabs(hr[i] - rstd) <= 1e-5 * rstd);
        for (int64_t j = 0; j < D; ++j) {
            const double gj = from_half(hg[j]);
            const double yref = 2.0 * rstd * gj;
            const double dxref = rstd * (gj * gj - 4.0 * rstd * rstd * mg2);
            CHECK(fabs(from_half(hy[i * D + j]) - yref) <= 2e-3 + 2e-3 * fabs(yref));
            CHECK(fabs(from_half(hdx[i * D + j]) - dxref) <= 2e-3 + 2e-3 * fabs(dxref));
        }
    }
    for (int64_t j = 0; j < D; ++j) {
        const double dgref = (double)N * 2.0 * rstd * from_half(hg[j]);
        CHECK(fabs(hdg[j] - dgref) <= 1e-4 * fabs(dgref));
    }
    printf("c_abi_consumer: ok (mt_norm_version %d)\n", mt_norm_version());
    return 0;
}
