/*
 * abi_client.c -- a plain C client of include/z3.h (no Python, no torch).
 *
 * Usage: abi_client <in.bin> <out.bin> <n_ranks> <steps> <n_params> n_0 n_1 ...
 * in.bin : fp32 master [Psi], then for each step the bf16 gradients
 *          [n_ranks][grad_stride] (grad_stride = Psi rounded up to 8)
 * out.bin: after partition and `steps` layer steps (t = 1..steps, Adam
 *          lr 1e-3, betas 0.9/0.999, eps 1e-8, scale 1/N): shards bf16,
 *          master, m, v fp32 (each [N*S]), then the last gathered layer
 *          (bf16 [Psi]).
 * Device memory is allocated here with cudaMalloc; the library allocates
 * nothing.  Exit status 0 on success, 1 on any error (message on stderr).
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

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

int main(int argc, char **argv) {
    if (argc < 6) {
        fprintf(stderr, "usage: %s in out n_ranks steps n_params n...\n", argv[0]);
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
    for (int t = 1; t <= steps; ++t) {
        const size_t n = (size_t)(n_ranks * stride);
        if (fread(h_grads, sizeof(uint16_t), n, in) != n) {
            fprintf(stderr, "short input (step %d)\n", t);
            return 1;
        }
        CUDA_OK(cudaMemcpyAsync(grads, h_grads, sizeof(uint16_t) * n, cudaMemcpyHostToDevice, stream));
        Z3_OK_OR_FAIL(z3_step_layer(L, shards, gathered, grads, stride, 1.0f / (float)n_ranks,
                                    master, m, v, &hp, t, stream));
        CUDA_OK(cudaStreamSynchronize(stream));  /* h_grads is reused next step */
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
