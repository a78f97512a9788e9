/* A plain C caller of libzg.so: no torch, no Python between it and the
 * library. Used by tests/test_gpu_c_abi.py.
 *
 *   c_abi_caller N P STEPS LOSS_SCALE in.bin out.bin
 *
 * in.bin:  N float32 initial master weights, then STEPS x P x N uint16 bf16
 *          gradient buffers (step-major, then rank).
 * out.bin: N float32 w, N float32 m, N float32 v, N uint16 bf16 params, then
 *          for each step: double sumsq, double norm, float clip, int found_inf,
 *          int64 step_t, int status.
 * Before the steps it checks that ordinary host memory (aligned_alloc) passed
 * as a gradient buffer or as the master weights is refused with
 * ZG_ERR_INVALID_ARG.
 * Exit status 0 on success; on any failure a message on stderr and 1. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "zg.h"

static int cuda_ok(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return 1;
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 0;
}

static int zg_ok(int rc, const char *what)
{
    if (rc == ZG_OK) return 1;
    fprintf(stderr, "%s: %s (%s)\n", what, zg_strerror(rc), zg_last_error());
    return 0;
}

int main(int argc, char **argv)
{
    if (argc != 7) {
        fprintf(stderr, "usage: %s N P STEPS LOSS_SCALE in.bin out.bin\n", argv[0]);
        return 1;
    }
    const int64_t n = atoll(argv[1]);
    const int p = atoi(argv[2]);
    const int steps = atoi(argv[3]);
    const float loss_scale = (float)atof(argv[4]);
    if (n <= 0 || p <= 0 || p > ZG_MAX_RANKS || steps <= 0) {
        fprintf(stderr, "bad sizes\n");
        return 1;
    }
    FILE *fin = fopen(argv[5], "rb");
    if (!fin) {
        fprintf(stderr, "cannot open %s\n", argv[5]);
        return 1;
    }
    float *w0 = (float *)malloc((size_t)n * sizeof(float));
    uint16_t *grads = (uint16_t *)malloc((size_t)steps * p * n * sizeof(uint16_t));
    if (!w0 || !grads || fread(w0, sizeof(float), (size_t)n, fin) != (size_t)n ||
        fread(grads, sizeof(uint16_t), (size_t)steps * p * n, fin) != (size_t)steps * p * n) {
        fprintf(stderr, "short input\n");
        return 1;
    }
    fclose(fin);

    zg_hparams hp = {1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 1e-6, 1};
    zg_ctx *ctx = NULL;
    if (!zg_ok(zg_init(n, p, &hp, &ctx), "zg_init")) return 1;
    const int64_t s = zg_shard_len(ctx);
    const size_t len = (size_t)(p * s); /* buffers padded to P * S elements */

    float *w, *m, *v;
    uint16_t *params;
    uint16_t *g[ZG_MAX_RANKS];
    if (!cuda_ok(cudaMalloc((void **)&w, len * 4), "cudaMalloc w") ||
        !cuda_ok(cudaMalloc((void **)&m, len * 4), "cudaMalloc m") ||
        !cuda_ok(cudaMalloc((void **)&v, len * 4), "cudaMalloc v") ||
        !cuda_ok(cudaMalloc((void **)&params, len * 2), "cudaMalloc params"))
        return 1;
    for (int r = 0; r < p; ++r)
        if (!cuda_ok(cudaMalloc((void **)&g[r], len * 2), "cudaMalloc grads") ||
            !cuda_ok(cudaMemset(g[r], 0, len * 2), "cudaMemset grads"))
            return 1;
    if (!cuda_ok(cudaMemcpy(w, w0, (size_t)n * 4, cudaMemcpyHostToDevice), "copy w") ||
        !cuda_ok(cudaMemset(m, 0, len * 4), "zero m") || !cuda_ok(cudaMemset(v, 0, len * 4), "zero v") ||
        !cuda_ok(cudaMemset(params, 0, len * 2), "zero params"))
        return 1;
    if (!zg_ok(zg_bind(ctx, w, m, v, params), "zg_bind")) return 1;

    cudaStream_t stream;
    if (!cuda_ok(cudaStreamCreate(&stream), "stream")) return 1;

    /* ordinary host memory is refused before anything is launched: as a
     * gradient buffer, and as the master weights */
    {
        uint16_t *host_grad = (uint16_t *)aligned_alloc(16, len * 2);
        float *host_w = (float *)aligned_alloc(16, len * 4);
        const uint16_t *gh[ZG_MAX_RANKS];
        if (!host_grad || !host_w) {
            fprintf(stderr, "host allocation failed\n");
            return 1;
        }
        for (int r = 0; r < p; ++r) gh[r] = g[r];
        gh[p - 1] = host_grad;
        if (zg_step(ctx, gh, loss_scale, (zg_stream)stream) != ZG_ERR_INVALID_ARG) {
            fprintf(stderr, "a host gradient buffer was not refused\n");
            return 1;
        }
        if (zg_bind(ctx, host_w, m, v, params) != ZG_ERR_INVALID_ARG) {
            fprintf(stderr, "host master weights were not refused\n");
            return 1;
        }
        free(host_grad);
        free(host_w);
    }
    FILE *fout = fopen(argv[6], "wb");
    if (!fout) {
        fprintf(stderr, "cannot open %s\n", argv[6]);
        return 1;
    }
    zg_step_info *infos = (zg_step_info *)calloc((size_t)steps, sizeof(zg_step_info));
    for (int t = 0; t < steps; ++t) {
        for (int r = 0; r < p; ++r)
            if (!cuda_ok(cudaMemcpyAsync(g[r], grads + ((size_t)t * p + r) * n, (size_t)n * 2,
                                         cudaMemcpyHostToDevice, stream),
                         "copy grads"))
                return 1;
        if (!zg_ok(zg_step(ctx, (const uint16_t *const *)g, loss_scale, (zg_stream)stream), "zg_step")) return 1;
        if (!zg_ok(zg_get_info(ctx, (zg_stream)stream, &infos[t]), "zg_get_info")) return 1;
    }
    float *hw = (float *)malloc((size_t)n * 4);
    uint16_t *hp16 = (uint16_t *)malloc((size_t)n * 2);
    float *const bufs[3] = {w, m, v};
    for (int k = 0; k < 3; ++k) {
        if (!cuda_ok(cudaMemcpy(hw, bufs[k], (size_t)n * 4, cudaMemcpyDeviceToHost), "read state")) return 1;
        fwrite(hw, 4, (size_t)n, fout);
    }
    if (!cuda_ok(cudaMemcpy(hp16, params, (size_t)n * 2, cudaMemcpyDeviceToHost), "read params")) return 1;
    fwrite(hp16, 2, (size_t)n, fout);
    for (int t = 0; t < steps; ++t) {
        fwrite(&infos[t].sumsq, sizeof(double), 1, fout);
        fwrite(&infos[t].norm, sizeof(double), 1, fout);
        fwrite(&infos[t].clip_coef, sizeof(float), 1, fout);
        fwrite(&infos[t].found_inf, sizeof(int), 1, fout);
        fwrite(&infos[t].step_t, sizeof(int64_t), 1, fout);
        fwrite(&infos[t].status, sizeof(int), 1, fout);
    }
    fclose(fout);
    zg_destroy(ctx);
    cudaStreamDestroy(stream);
    for (int r = 0; r < p; ++r) cudaFree(g[r]);
    cudaFree(w);
    cudaFree(m);
    cudaFree(v);
    cudaFree(params);
    free(w0);
    free(grads);
    free(hw);
    free(hp16);
    free(infos);
    return 0;
}
