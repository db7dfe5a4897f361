/*
 * abi_client.c -- a plain C client of include/z3.h (no Python, no torch).
 *
 * Usage: abi_client [mode] <in.bin> <out.bin> <n_ranks> <steps> <n_params> n_0 n_1 ...
 * mode   : --layer (default) z3_step_layer from device gradients;
 *          --host  the same steps through z3_host_step_run from page-locked
 *                  host gradients, downloading the shards every step;
 *          --model z3_model_step over one unit per parameter (unit 0 kept
 *                  resident), with prefetch depth 1 on a second stream.
 * in.bin : fp32 master [Psi], then for each step the bf16 gradients
 *          [n_ranks][grad_stride] (grad_stride = Psi rounded up to 8)
 * out.bin: --layer / --host: after partition and `steps` layer steps
 *          (t = 1..steps, Adam lr 1e-3, betas 0.9/0.999, eps 1e-8, scale
 *          1/N): shards bf16, master, m, v fp32 (each [N*S]), then the last
 *          gathered layer (bf16 [Psi]).
 *          --model: for every unit p: shards, master, m, v of its own layout
 *          (each [N*s_p]), then unit 0's resident copy (bf16 [n_0]).
 * Device memory is allocated here with cudaMalloc; the library allocates
 * nothing.  Exit status 0 on success, 1 on any error (message on stderr).
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "z3.h"

#define CUDA_OK(x)                                                             \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));           \
            return 1;                                                          \
        }                                                                      \
    } while (0)

#define Z3_OK_OR_FAIL(x)                                                       \
    do {                                                                       \
        z3_status s_ = (x);                                                    \
        if (s_ != Z3_OK) {                                                     \
            char msg_[256];                                                    \
            z3_last_error(msg_, sizeof msg_);                                  \
            fprintf(stderr, "%s: %s (%s)\n", #x, z3_status_string(s_), msg_);  \
            return 1;                                                          \
        }                                                                      \
    } while (0)

static int run_model(const char *in_path, const char *out_path, int32_t n_ranks, int steps,
                     int32_t n_params, const int64_t *numel);

int main(int argc, char **argv) {
    int mode = 0;  /* 0 layer, 1 host, 2 model */
    if (argc > 1 && argv[1][0] == '-') {
        if (strcmp(argv[1], "--host") == 0) mode = 1;
        else if (strcmp(argv[1], "--model") == 0) mode = 2;
        else if (strcmp(argv[1], "--layer") != 0) {
            fprintf(stderr, "unknown mode %s\n", argv[1]);
            return 1;
        }
        ++argv;
        --argc;
    }
    if (argc < 6) {
        fprintf(stderr, "usage: %s [mode] in out n_ranks steps n_params n...\n", argv[0]);
        return 1;
    }
    const int32_t n_ranks = atoi(argv[3]);
    const int steps = atoi(argv[4]);
    const int32_t n_params = atoi(argv[5]);
    if (n_params < 1 || argc != 6 + n_params) {
        fprintf(stderr, "bad parameter list\n");
        return 1;
    }
    int64_t *numel = malloc(sizeof(int64_t) * (size_t)n_params);
    for (int32_t p = 0; p < n_params; ++p) numel[p] = atoll(argv[6 + p]);
    if (mode == 2) return run_model(argv[1], argv[2], n_ranks, steps, n_params, numel);

    z3_layout *L = NULL;
    Z3_OK_OR_FAIL(z3_layout_create(numel, n_params, n_ranks, &L));
    int64_t S, psi, T;
    Z3_OK_OR_FAIL(z3_layout_info(L, NULL, NULL, &S, &psi, &T));
    const int64_t stride = (psi + 7) / 8 * 8;

    FILE *in = fopen(argv[1], "rb");
    if (!in) { fprintf(stderr, "cannot open %s\n", argv[1]); return 1; }
    float *h_full = malloc(sizeof(float) * (size_t)psi);
    uint16_t *h_grads = malloc(sizeof(uint16_t) * (size_t)(n_ranks * stride));
    if (fread(h_full, sizeof(float), (size_t)psi, in) != (size_t)psi) {
        fprintf(stderr, "short input\n");
        return 1;
    }

    float *full, *master, *m, *v;
    uint16_t *shards, *gathered, *grads;
    CUDA_OK(cudaMalloc((void **)&full, sizeof(float) * (size_t)psi));
    CUDA_OK(cudaMalloc((void **)&master, sizeof(float) * (size_t)T));
    CUDA_OK(cudaMalloc((void **)&m, sizeof(float) * (size_t)T));
    CUDA_OK(cudaMalloc((void **)&v, sizeof(float) * (size_t)T));
    CUDA_OK(cudaMalloc((void **)&shards, sizeof(uint16_t) * (size_t)T));
    CUDA_OK(cudaMalloc((void **)&gathered, sizeof(uint16_t) * (size_t)psi));
    CUDA_OK(cudaMalloc((void **)&grads, sizeof(uint16_t) * (size_t)(n_ranks * stride)));
    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));

    CUDA_OK(cudaMemcpyAsync(full, h_full, sizeof(float) * (size_t)psi, cudaMemcpyHostToDevice, stream));
    Z3_OK_OR_FAIL(z3_partition(L, full, shards, master, m, v, stream));
    const z3_adam_hp hp = {1e-3, 0.9, 0.999, 1e-8, 0.0};
    if (mode == 1) {
        /* every step's gradients and downloaded shards in their own
         * page-locked buffers, so no host buffer is reused while a copy of
         * an earlier step may still run */
        const size_t n = (size_t)(n_ranks * stride);
        uint16_t *staging[2], **hg = malloc(sizeof(uint16_t *) * (size_t)steps),
                 **hs = malloc(sizeof(uint16_t *) * (size_t)steps);
        CUDA_OK(cudaMalloc((void **)&staging[0], sizeof(uint16_t) * n));
        CUDA_OK(cudaMalloc((void **)&staging[1], sizeof(uint16_t) * n));
        cudaStream_t up, down;
        CUDA_OK(cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking));
        CUDA_OK(cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking));
        for (int t = 0; t < steps; ++t) {
            CUDA_OK(cudaMallocHost((void **)&hg[t], sizeof(uint16_t) * n));
            CUDA_OK(cudaMallocHost((void **)&hs[t], sizeof(uint16_t) * (size_t)T));
            if (fread(hg[t], sizeof(uint16_t), n, in) != n) {
                fprintf(stderr, "short input (step %d)\n", t + 1);
                return 1;
            }
        }
        CUDA_OK(cudaStreamSynchronize(stream));
        z3_host_step *pipe = NULL;
        Z3_OK_OR_FAIL(z3_host_step_create(L, staging[0], staging[1], stride, up, down, &pipe));
        for (int t = 1; t <= steps; ++t)
            Z3_OK_OR_FAIL(z3_host_step_run(pipe, hg[t - 1], shards, gathered,
                                           1.0f / (float)n_ranks, master, m, v, &hp, t,
                                           hs[t - 1], stream));
        CUDA_OK(cudaDeviceSynchronize());
        z3_host_step_destroy(pipe);
        uint16_t *last = malloc(sizeof(uint16_t) * (size_t)T);
        CUDA_OK(cudaMemcpy(last, shards, sizeof(uint16_t) * (size_t)T, cudaMemcpyDeviceToHost));
        if (steps > 0 && memcmp(last, hs[steps - 1], sizeof(uint16_t) * (size_t)T) != 0) {
            fprintf(stderr, "the last downloaded shards differ from the device shards\n");
            return 1;
        }
        free(last);
        for (int t = 0; t < steps; ++t) {
            cudaFreeHost(hg[t]);
            cudaFreeHost(hs[t]);
        }
        free(hg); free(hs);
        cudaFree(staging[0]); cudaFree(staging[1]);
        cudaStreamDestroy(up); cudaStreamDestroy(down);
    } else {
        for (int t = 1; t <= steps; ++t) {
            const size_t n = (size_t)(n_ranks * stride);
            if (fread(h_grads, sizeof(uint16_t), n, in) != n) {
                fprintf(stderr, "short input (step %d)\n", t);
                return 1;
            }
            CUDA_OK(cudaMemcpyAsync(grads, h_grads, sizeof(uint16_t) * n, cudaMemcpyHostToDevice, stream));
            Z3_OK_OR_FAIL(z3_step_layer(L, shards, gathered, grads, stride, 1.0f / (float)n_ranks,
                                        master, m, v, NULL, &hp, t, stream));
            CUDA_OK(cudaStreamSynchronize(stream));  /* h_grads is reused next step */
        }
    }
    fclose(in);

    FILE *out = fopen(argv[2], "wb");
    if (!out) { fprintf(stderr, "cannot open %s\n", argv[2]); return 1; }
    void *h = malloc(sizeof(float) * (size_t)(T > psi ? T : psi));
    CUDA_OK(cudaMemcpy(h, shards, sizeof(uint16_t) * (size_t)T, cudaMemcpyDeviceToHost));
    fwrite(h, sizeof(uint16_t), (size_t)T, out);
    float *bufs[3] = {master, m, v};
    for (int b = 0; b < 3; ++b) {
        CUDA_OK(cudaMemcpy(h, bufs[b], sizeof(float) * (size_t)T, cudaMemcpyDeviceToHost));
        fwrite(h, sizeof(float), (size_t)T, out);
    }
    CUDA_OK(cudaMemcpy(h, gathered, sizeof(uint16_t) * (size_t)psi, cudaMemcpyDeviceToHost));
    fwrite(h, sizeof(uint16_t), (size_t)psi, out);
    fclose(out);

    z3_layout_destroy(L);
    cudaFree(full); cudaFree(master); cudaFree(m); cudaFree(v);
    cudaFree(shards); cudaFree(gathered); cudaFree(grads);
    cudaStreamDestroy(stream);
    free(h); free(h_full); free(h_grads); free(numel);
    return 0;
}

/* --model: one unit per parameter, unit 0 resident, prefetch depth 1. */
static int run_model(const char *in_path, const char *out_path, int32_t n_ranks, int steps,
                     int32_t n_params, const int64_t *numel) {
    int64_t psi = 0;
    for (int32_t p = 0; p < n_params; ++p) psi += numel[p];
    const int64_t stride = (psi + 7) / 8 * 8;
    FILE *in = fopen(in_path, "rb");
    if (!in) { fprintf(stderr, "cannot open %s\n", in_path); return 1; }
    float *h_full = malloc(sizeof(float) * (size_t)(psi > 0 ? psi : 1));
    if (fread(h_full, sizeof(float), (size_t)psi, in) != (size_t)psi) {
        fprintf(stderr, "short input\n");
        return 1;
    }
    cudaStream_t stream, gstream;
    CUDA_OK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    CUDA_OK(cudaStreamCreateWithFlags(&gstream, cudaStreamNonBlocking));
    float *d_full;
    uint16_t *d_grads_all;
    CUDA_OK(cudaMalloc((void **)&d_full, sizeof(float) * (size_t)(psi > 0 ? psi : 1)));
    CUDA_OK(cudaMalloc((void **)&d_grads_all, sizeof(uint16_t) * (size_t)(n_ranks * stride + 8)));
    /* every copy goes on `stream`: the library's launches there (and on
     * gstream, which the library orders after `stream`) see them complete */
    CUDA_OK(cudaMemcpyAsync(d_full, h_full, sizeof(float) * (size_t)psi, cudaMemcpyHostToDevice,
                            stream));

    z3_unit *units = calloc((size_t)n_params, sizeof(z3_unit));
    z3_layout **L = calloc((size_t)n_params, sizeof(z3_layout *));
    int64_t *T = calloc((size_t)n_params, sizeof(int64_t)), *ustride = calloc((size_t)n_params, sizeof(int64_t));
    uint16_t **ugrads = calloc((size_t)n_params, sizeof(uint16_t *));
    int64_t off = 0, big = 8;
    for (int32_t p = 0; p < n_params; ++p) {
        Z3_OK_OR_FAIL(z3_layout_create(&numel[p], 1, n_ranks, &L[p]));
        Z3_OK_OR_FAIL(z3_layout_info(L[p], NULL, NULL, NULL, NULL, &T[p]));
        ustride[p] = (numel[p] + 7) / 8 * 8;
        const size_t t = (size_t)(T[p] > 0 ? T[p] : 8);
        z3_unit *u = &units[p];
        u->layout = L[p];
        CUDA_OK(cudaMalloc((void **)&u->shards, sizeof(uint16_t) * t));
        CUDA_OK(cudaMalloc((void **)&u->master, sizeof(float) * t));
        CUDA_OK(cudaMalloc((void **)&u->m, sizeof(float) * t));
        CUDA_OK(cudaMalloc((void **)&u->v, sizeof(float) * t));
        CUDA_OK(cudaMalloc((void **)&ugrads[p], sizeof(uint16_t) * (size_t)(n_ranks * ustride[p] + 8)));
        u->grads = ugrads[p];
        u->grad_stride = ustride[p];
        u->scale = 1.0f / (float)n_ranks;
        /* the library wants 16-byte-aligned buffers: copy the unit's slice of
         * the full parameter vector to the start of its own allocation */
        float *d_unit = NULL;
        CUDA_OK(cudaMalloc((void **)&d_unit, sizeof(float) * (size_t)(numel[p] > 0 ? numel[p] : 1)));
        CUDA_OK(cudaMemcpyAsync(d_unit, d_full + off, sizeof(float) * (size_t)numel[p],
                                cudaMemcpyDeviceToDevice, stream));
        Z3_OK_OR_FAIL(z3_partition(L[p], d_unit, u->shards, u->master, u->m, u->v, stream));
        CUDA_OK(cudaStreamSynchronize(stream));
        cudaFree(d_unit);
        if (p == 0 && numel[0] > 0) {
            CUDA_OK(cudaMalloc((void **)&u->resident, sizeof(uint16_t) * (size_t)numel[0]));
            Z3_OK_OR_FAIL(z3_allgather(L[p], u->shards, u->resident, stream));
        } else if (numel[p] > big) {
            big = numel[p];
        }
        off += numel[p];
    }
    uint16_t *fulls[2];
    CUDA_OK(cudaMalloc((void **)&fulls[0], sizeof(uint16_t) * (size_t)big));
    CUDA_OK(cudaMalloc((void **)&fulls[1], sizeof(uint16_t) * (size_t)big));
    uint16_t *h_grads = malloc(sizeof(uint16_t) * (size_t)(n_ranks * stride + 8));
    const z3_adam_hp hp = {1e-3, 0.9, 0.999, 1e-8, 0.0};
    for (int t = 1; t <= steps; ++t) {
        const size_t n = (size_t)(n_ranks * stride);
        if (fread(h_grads, sizeof(uint16_t), n, in) != n) {
            fprintf(stderr, "short input (step %d)\n", t);
            return 1;
        }
        CUDA_OK(cudaStreamSynchronize(stream));   /* the last step no longer reads the grads */
        CUDA_OK(cudaMemcpyAsync(d_grads_all, h_grads, sizeof(uint16_t) * n, cudaMemcpyHostToDevice,
                                stream));
        off = 0;
        for (int32_t p = 0; p < n_params; ++p) {    /* unit p's columns of every rank's row */
            if (numel[p] > 0)
                CUDA_OK(cudaMemcpy2DAsync(ugrads[p], sizeof(uint16_t) * (size_t)ustride[p],
                                          d_grads_all + off, sizeof(uint16_t) * (size_t)stride,
                                          sizeof(uint16_t) * (size_t)numel[p], (size_t)n_ranks,
                                          cudaMemcpyDeviceToDevice, stream));
            off += numel[p];
        }
        Z3_OK_OR_FAIL(z3_model_step(units, n_params, fulls, 2, &hp, t, stream, gstream));
    }
    CUDA_OK(cudaDeviceSynchronize());
    fclose(in);

    FILE *out = fopen(out_path, "wb");
    if (!out) { fprintf(stderr, "cannot open %s\n", out_path); return 1; }
    for (int32_t p = 0; p < n_params; ++p) {
        const size_t t = (size_t)T[p];
        void *h = malloc(sizeof(float) * (t > 0 ? t : 1));
        CUDA_OK(cudaMemcpy(h, units[p].shards, sizeof(uint16_t) * t, cudaMemcpyDeviceToHost));
        fwrite(h, sizeof(uint16_t), t, out);
        float *bufs[3] = {units[p].master, units[p].m, units[p].v};
        for (int b = 0; b < 3; ++b) {
            CUDA_OK(cudaMemcpy(h, bufs[b], sizeof(float) * t, cudaMemcpyDeviceToHost));
            fwrite(h, sizeof(float), t, out);
        }
        free(h);
    }
    if (numel[0] > 0) {
        uint16_t *h = malloc(sizeof(uint16_t) * (size_t)numel[0]);
        CUDA_OK(cudaMemcpy(h, units[0].resident, sizeof(uint16_t) * (size_t)numel[0],
                           cudaMemcpyDeviceToHost));
        fwrite(h, sizeof(uint16_t), (size_t)numel[0], out);
        free(h);
    }
    fclose(out);
    for (int32_t p = 0; p < n_params; ++p) {
        cudaFree(units[p].shards); cudaFree(units[p].master); cudaFree(units[p].m);
        cudaFree(units[p].v); cudaFree(ugrads[p]); cudaFree(units[p].resident);
        z3_layout_destroy(L[p]);
    }
    cudaFree(fulls[0]); cudaFree(fulls[1]); cudaFree(d_full); cudaFree(d_grads_all);
    cudaStreamDestroy(stream); cudaStreamDestroy(gstream);
    free(units); free(L); free(T); free(ustride); free(ugrads); free(h_grads); free(h_full);
    return 0;
}
