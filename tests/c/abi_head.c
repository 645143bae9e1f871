/*
 * The C ABI used from plain C: device buffers from cudaMalloc, the workspace
 * sized by its query, the LM-head estimator and the embedding scatter called
 * on a caller-created stream, errors read as status codes.  Inputs come from a
 * small integer hash, so the Python side can rebuild them exactly.
 *
 *   abi_head <out.bin>   writes G_W (V x d fp32) then G_E (V x d fp32)
 * Exit status 0 on success; a failed check prints its line and exits 1.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "../../include/dust.h"

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            return 1;                                                \
        }                                                            \
    } while (0)

enum { T = 300, V = 1000, D = 24 };

/* uniform in [-1, 1) from an index: the same formula as the Python side */
static float hval(uint32_t i, uint32_t salt) {
    uint32_t x = i * 2654435761u ^ salt * 2246822519u;
    x ^= x >> 15;
    x *= 2246822519u;
    x ^= x >> 13;
    return (float)(x >> 8) / 8388608.0f - 1.0f;
}

int main(int argc, char** argv) {
    if (argc != 2) return 2;
    CHECK(dust_abi_version() >= 100);
    float* z = malloc(sizeof(float) * T * V);
    float* x = malloc(sizeof(float) * T * D);
    int32_t* y = malloc(sizeof(int32_t) * T);
    float* G = malloc(sizeof(float) * V * D);
    float* GE = malloc(sizeof(float) * V * D);
    for (int i = 0; i < T * V; ++i) z[i] = 3.0f * hval((uint32_t)i, 1u);
    for (int i = 0; i < T * D; ++i) x[i] = hval((uint32_t)i, 2u);
    for (int t = 0; t < T; ++t) y[t] = (int32_t)((uint32_t)(hval((uint32_t)t, 3u) * 0.5f * V + V) % V);

    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess);
    float *dz, *dx, *dG, *dGE;
    int32_t *dy, *dperm;
    CHECK(cudaMalloc((void**)&dz, sizeof(float) * T * V) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dx, sizeof(float) * T * D) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dy, sizeof(int32_t) * T) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dG, sizeof(float) * V * D) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dGE, sizeof(float) * V * D) == cudaSuccess);
    CHECK(cudaMalloc((void**)&dperm, sizeof(int32_t) * T) == cudaSuccess);
    CHECK(cudaMemcpy(dz, z, sizeof(float) * T * V, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dx, x, sizeof(float) * T * D, cudaMemcpyHostToDevice) == cudaSuccess);
    CHECK(cudaMemcpy(dy, y, sizeof(int32_t) * T, cudaMemcpyHostToDevice) == cudaSuccess);

    dust_noise nz = {1234u, 0u, 0u, 16u, 0u, 0.05f, 0.0f};
    size_t wsb = dust_head_workspace(T, V, D, nz.num_draws);
    CHECK(wsb > 0);
    void* ws;
    CHECK(cudaMalloc(&ws, wsb) == cudaSuccess);
    /* errors come back as codes, before any launch */
    CHECK(dust_head_estimate(NULL, dy, dx, DUST_F32, T, V, D, nz, NULL, dG, ws, wsb, s) ==
          DUST_ERR_INVALID_ARG);
    CHECK(dust_head_estimate(dz, dy, dx, DUST_F32, T, V, D, nz, NULL, dG, ws, wsb - 1, s) ==
          DUST_ERR_WORKSPACE);
    CHECK(dust_status_string(DUST_ERR_WORKSPACE) != NULL);
    /* the estimator (g not returned), then its status word */
    CHECK(dust_head_estimate(dz, dy, dx, DUST_F32, T, V, D, nz, NULL, dG, ws, wsb, s) == DUST_OK);
    dust_status dev_status = DUST_ERR_CUDA;
    CHECK(dust_workspace_status(ws, s, &dev_status) == DUST_OK);
    CHECK(dev_status == DUST_OK);

    /* the embedding scatter of x's rows by target id (any T x d rows will do) */
    size_t wse = dust_embed_workspace(T, D, V);
    void* wse_p;
    CHECK(cudaMalloc(&wse_p, wse) == cudaSuccess);
    CHECK(dust_embed_scatter(dx, dy, T, D, V, dGE, dperm, wse_p, wse, s) == DUST_OK);
    CHECK(dust_workspace_status(wse_p, s, &dev_status) == DUST_OK && dev_status == DUST_OK);

    CHECK(cudaMemcpyAsync(G, dG, sizeof(float) * V * D, cudaMemcpyDeviceToHost, s) == cudaSuccess);
    CHECK(cudaMemcpyAsync(GE, dGE, sizeof(float) * V * D, cudaMemcpyDeviceToHost, s) ==
          cudaSuccess);
    CHECK(cudaStreamSynchronize(s) == cudaSuccess);
    for (int i = 0; i < V * D; ++i) CHECK(isfinite(G[i]) && isfinite(GE[i]));

    FILE* f = fopen(argv[1], "wb");
    CHECK(f != NULL);
    CHECK(fwrite(G, sizeof(float), V * D, f) == V * D);
    CHECK(fwrite(GE, sizeof(float), V * D, f) == V * D);
    fclose(f);
    cudaFree(dz); cudaFree(dx); cudaFree(dy); cudaFree(dG); cudaFree(dGE); cudaFree(dperm);
    cudaFree(ws); cudaFree(wse_p);
    cudaStreamDestroy(s);
    free(z); free(x); free(y); free(G); free(GE);
    return 0;
}
