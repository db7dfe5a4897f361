// z3_launch.h -- the kernels' argument blocks and their launchers, shared by
// the kernel translation unit (z3_kernels.cu) and the C-ABI entry points
// (z3_api.cpp).  Not part of the public ABI.
//
// A launcher enqueues the kernels of one operation on a stream and returns
// the launch error (cudaGetLastError); it validates nothing.  Every caller
// validates its arguments first (z3_api.cpp).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "z3_internal.h"

namespace z3 {

// Binary32 constants of one Adam step (each rounded once on the host).
struct AdamK {
    float b1, c1, b2, c2, rb1, rb2, lr, eps, lwd;
};

// What the reduce kernels do with the rank fold of each owned position.
enum Mode : int {
    kRS = 0,         // grad_shards = fold * scale
    kRSAcc = 1,      // grad_shards = grad_shards + fold * scale
    kRSAdam = 2,     // Adam(fold * scale)
    kRSAccAdam = 3,  // Adam(grad_acc + fold * scale)
    kRSAdamOut = 4,  // Adam(fold * scale), and fold * scale stored to grad_shards
};

struct ReduceArgs {
    const uint16_t *__restrict__ grads;  // [N][stride] bf16
    int64_t stride;
    float scale;
    float *out;             // grad_shards (kRS, kRSAcc, kRSAdamOut)
    const float *acc_in;    // grad_acc (kRSAccAdam)
    float *master;
    float *m;
    float *v;
    uint16_t *shards;
    AdamK k;
};

struct PartitionArgs {
    const float *__restrict__ full;
    uint16_t *__restrict__ shards;
    float *__restrict__ master;
    float *__restrict__ m;
    float *__restrict__ v;
};

struct AdamArgs {
    float *master;
    float *m;
    float *v;
    const float *grad;
    uint16_t *shards;
    int64_t total;
    AdamK k;
};

struct AllreduceArgs {
    const uint16_t *__restrict__ grads;
    int64_t stride;
    float *__restrict__ out;
    int64_t psi;
    float scale;
    int n_ranks;
};

struct ScatterArgs {
    const float *__restrict__ full;
    float *__restrict__ shards;
};

// CTA sizes of the flat (table-free) kernels; each thread owns one vector.
constexpr int kAdamThreads = 256;
constexpr int kFlatThreads = 256;

// CTAs of a flat kernel over `total` elements.
inline int64_t flat_blocks(int64_t total, int threads) {
    return (total + (int64_t)threads * kVec - 1) / ((int64_t)threads * kVec);
}

cudaError_t launch_partition(const z3_layout *L, const PartitionArgs &a, cudaStream_t stream);
// early: the kernel of this stream just before this launch was enqueued by
// the library in the same call and writes nothing this launch reads (for
// the gather: not the shards; for a fused reduce: not the gradients, running
// sums, master, m or v).  The launch may then read before it waits for that
// kernel (its stores still wait).  Ignored by the unfused reduce modes and
// by kRSAdamOut.
cudaError_t launch_allgather(const z3_layout *L, const uint16_t *shards, uint16_t *full,
                             cudaStream_t stream, bool early);
cudaError_t launch_reduce(const z3_layout *L, const ReduceArgs &a, Mode mode,
                          cudaStream_t stream, bool early);
cudaError_t launch_adam(const AdamArgs &a, cudaStream_t stream);
cudaError_t launch_allreduce(const AllreduceArgs &a, cudaStream_t stream);
cudaError_t launch_scatter(const z3_layout *L, const ScatterArgs &a, cudaStream_t stream);
// elem_bytes 2 or 4; both layouts describe the same parameters
cudaError_t launch_reshard(const z3_layout *Ls, const z3_layout *Ld, int elem_bytes,
                           const void *src, void *dst, cudaStream_t stream);

}  // namespace z3
