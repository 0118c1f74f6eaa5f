/* A plain C caller of the library (no Python): reads n float32 weights and
 * gradients from files, runs `steps` clipped-AdamW steps through the C ABI of
 * adamw_ckpt.h on the current CUDA device, writes the checkpoint of the final
 * state into a directory and prints its path and the last gradient norm.
 *
 *   step_ckpt <n> <w.f32> <g.f32> <steps> <lr> <wd> <clip> <dir>
 *
 * Exit status 0 on success; on a library error the status name and the
 * library's explanation go to stderr. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "adamw_ckpt.h"

static int check(int status, const char* what)
{
    if (status != ADAMW_OK)
        fprintf(stderr, "%s: %s: %s\n", what, adamw_strerror(status), adamw_last_error());
    return status == ADAMW_OK;
}

static float* read_f32(const char* path, int64_t n)
{
    FILE* f = fopen(path, "rb");
    float* h = (float*)malloc((size_t)n * sizeof(float));
    size_t got = (f && h) ? fread(h, sizeof(float), (size_t)n, f) : 0;
    if (f)
        fclose(f);
    if (got != (size_t)n) {
        free(h);
        return NULL;
    }
    return h;
}

int main(int argc, char** argv)
{
    if (argc != 9) {
        fprintf(stderr, "usage: step_ckpt n w.f32 g.f32 steps lr wd clip dir\n");
        return 2;
    }
    const int64_t n = atoll(argv[1]);
    const int steps = atoi(argv[4]);
    const double lr = atof(argv[5]), wd = atof(argv[6]), clip = atof(argv[7]);
    float* hw = read_f32(argv[2], n);
    float* hg = read_f32(argv[3], n);
    if (n < 1 || steps < 1 || !hw || !hg) {
        fprintf(stderr, "bad arguments or input files\n");
        return 2;
    }
    const size_t bytes = (size_t)n * sizeof(float);
    float *w = NULL, *g = NULL, *m = NULL, *v = NULL;
    if (cudaMalloc((void**)&w, bytes) != cudaSuccess || cudaMalloc((void**)&g, bytes) != cudaSuccess ||
        cudaMalloc((void**)&m, bytes) != cudaSuccess || cudaMalloc((void**)&v, bytes) != cudaSuccess ||
        cudaMemcpy(w, hw, bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(g, hg, bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(m, 0, bytes) != cudaSuccess || cudaMemset(v, 0, bytes) != cudaSuccess) {
        fprintf(stderr, "device setup failed\n");
        return 1;
    }
    adamw_ctx* ctx = NULL;
    int ok = check(adamw_create(n, NULL, NULL, 0, 0, &ctx), "adamw_create");
    for (int t = 1; ok && t <= steps; ++t)
        ok = check(adamw_clip_step(ctx, w, g, m, v, t, lr, wd, clip, NULL), "adamw_clip_step");
    double norm = 0.0;
    float scale = 0.0f;
    if (ok)
        ok = check(adamw_last_norm(ctx, &norm, &scale), "adamw_last_norm");
    char path[4096] = {0};
    if (ok)
        ok = check(ckpt_pack(ctx, steps, w, m, v, NULL, NULL), "ckpt_pack") &&
             check(ckpt_write(ctx, argv[8], path, sizeof path), "ckpt_write");
    if (ok)
        printf("%s %.17g %.9g\n", path, norm, (double)scale);
    adamw_destroy(ctx);
    cudaFree(w);
    cudaFree(g);
    cudaFree(m);
    cudaFree(v);
    free(hw);
    free(hg);
    return ok ? 0 : 1;
}
