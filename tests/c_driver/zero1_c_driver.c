/* A plain-C client of the zero1 C ABI (test infrastructure): it includes
 * only zero1.h and the CUDA runtime's C header, runs a few steps on device
 * buffers, and writes its inputs and results to binary files for the
 * Python test to check against the oracle.
 *
 * usage: zero1_c_driver N W STEPS OUTDIR
 * writes OUTDIR/master0.f32 (N floats), OUTDIR/grads_t<t>_r<r>.bf16 (N
 * uint16 per step and rank), OUTDIR/clip.f32 (STEPS floats: the clip
 * coefficient each step used), OUTDIR/master.f32, m.f32, v.f32 (N floats
 * after the last step), OUTDIR/rep_<r>.bf16 (replicas 0 and W-1). */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero1.h"

static uint64_t lcg_state = 0x9E3779B97F4A7C15ull;

/* A uniform double in [-1, 1) from a 64-bit linear congruential generator
 * (Knuth's MMIX constants). */
static double uniform(void)
{
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(lcg_state >> 11) / 9007199254740992.0 * 2.0 - 1.0;
}

/* Round-to-nearest-even float -> bf16 bits (finite inputs only). */
static uint16_t to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes)
{
    char path[1024];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return -1;
    size_t w = fwrite(p, 1, bytes, f);
    fclose(f);
    return w == bytes ? 0 : -1;
}

#define CHECK(call)                                                                  \
    do {                                                                             \
        int rc_ = (call);                                                            \
        if (rc_ != 0) {                                                              \
            fprintf(stderr, "%s failed: %d (%s)\n", #call, rc_, zero1_last_error()); \
            return 1;                                                                \
        }                                                                            \
    } while (0)
#define CUDA(call)                                                                          \
    do {                                                                                    \
        cudaError_t e_ = (call);                                                            \
        if (e_ != cudaSuccess) {                                                            \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));              \
            return 1;                                                                       \
        }                                                                                   \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 5) {
        fprintf(stderr, "usage: %s N W STEPS OUTDIR\n", argv[0]);
        return 2;
    }
    const uint64_t n = strtoull(argv[1], NULL, 10);
    const int world = atoi(argv[2]);
    const int steps = atoi(argv[3]);
    const char *dir = argv[4];
    if (n == 0 || world < 1 || world > ZERO1_MAX_WORLD || steps < 1) return 2;

    zero1_hparams hp = {1e-3, 0.9, 0.95, 1e-8, 0.1, 0.05};
    zero1_options opts;
    memset(&opts, 0, sizeof opts);
    opts.size = sizeof opts;
    opts.small_step = -1;                 /* the two-kernel path */
    zero1_handle h = NULL;
    CHECK(zero1_create_ex(n, world, &hp, &opts, &h));

    float *host_f = (float *)malloc(n * sizeof(float));
    uint16_t *host_b = (uint16_t *)malloc(n * sizeof(uint16_t));
    float *clips = (float *)malloc((size_t)steps * sizeof(float));
    void **grads = (void **)calloc((size_t)world, sizeof(void *));
    void **params = (void **)calloc((size_t)world, sizeof(void *));
    if (!host_f || !host_b || !clips || !grads || !params) return 3;
    for (int r = 0; r < world; ++r) {
        CUDA(cudaMalloc(&grads[r], n * 2));
        CUDA(cudaMalloc(&params[r], n * 2));
    }

    for (uint64_t i = 0; i < n; ++i) host_f[i] = (float)(0.02 * uniform());
    CHECK(write_file(dir, "master0.f32", host_f, n * 4));
    CHECK(zero1_set_state(h, host_f, NULL, NULL, 0, NULL));   /* host source, m = v = 0 */

    char name[64];
    for (int t = 1; t <= steps; ++t) {
        for (int r = 0; r < world; ++r) {
            for (uint64_t i = 0; i < n; ++i) host_b[i] = to_bf16((float)(0.01 * uniform()));
            snprintf(name, sizeof name, "grads_t%d_r%d.bf16", t, r);
            CHECK(write_file(dir, name, host_b, n * 2));
            CUDA(cudaMemcpy(grads[r], host_b, n * 2, cudaMemcpyHostToDevice));
        }
        CHECK(zero1_step(h, (const void *const *)grads, (void *const *)params, NULL));
        double norm = 0.0;
        CHECK(zero1_get_grad_norm(h, &norm, &clips[t - 1], NULL));
    }
    CHECK(write_file(dir, "clip.f32", clips, (size_t)steps * 4));

    float *m = (float *)malloc(n * 4), *v = (float *)malloc(n * 4);
    uint64_t t_done = 0;
    if (!m || !v) return 3;
    CHECK(zero1_get_state(h, host_f, m, v, &t_done, NULL));
    CUDA(cudaDeviceSynchronize());
    if (t_done != (uint64_t)steps) return 4;
    CHECK(write_file(dir, "master.f32", host_f, n * 4));
    CHECK(write_file(dir, "m.f32", m, n * 4));
    CHECK(write_file(dir, "v.f32", v, n * 4));
    const int reps[2] = {0, world - 1};
    for (int k = 0; k < 2; ++k) {
        CUDA(cudaMemcpy(host_b, params[reps[k]], n * 2, cudaMemcpyDeviceToHost));
        snprintf(name, sizeof name, "rep_%d.bf16", reps[k]);
        CHECK(write_file(dir, name, host_b, n * 2));
    }

    for (int r = 0; r < world; ++r) {
        cudaFree(grads[r]);
        cudaFree(params[r]);
    }
    CHECK(zero1_destroy(h));
    free(host_f); free(host_b); free(clips); free(grads); free(params); free(m); free(v);
    printf("c driver ok: n=%llu W=%d steps=%d\n", (unsigned long long)n, world, steps);
    return 0;
}
