// z3_noalloc.cu -- z3_step_layer_noalloc: the layer step for callers that
// cannot allocate device memory themselves.
//
// z3_step_layer needs one piece of memory beyond the caller's state and
// gradients: the transient buffer its two all-gathers write the layer's full
// bf16 parameters into (nothing in the step reads it back; in a training
// framework the model's forward and backward would).  Some callers cannot
// provide it: code that runs where it may not call cudaMalloc (an allocator
// callback, a plugin handed pre-allocated buffers by its host framework, a
// process whose device memory is fully reserved up front).  For them this
// file holds that buffer as a statically sized array in the library's own
// device memory, and the entry point below passes it to the ordinary layer
// step.  Nothing here allocates.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "z3_internal.h"

// The gather scratch: up to 16 Mi bf16 elements (32 MiB), enough for one
// transformer layer of d_model = 1024 (12.6 M elements).  As a static device
// array it occupies 32 MiB on every GPU where this library's device code is
// loaded, until the process exits.
static constexpr int64_t kScratchElems = int64_t(1) << 24;
static __device__ __align__(256) uint16_t g_gather_scratch[kScratchElems];

namespace z3 {
namespace {

// In host code `g_gather_scratch` names a host-side stand-in, not device
// memory: its device address is looked up once per device (with that
// device current) and kept here.
constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

z3_status scratch_address(const char *fn, void **out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return fail(Z3_ERR_CUDA, std::string(fn) + ": cudaGetDevice: " + cudaGetErrorString(err));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(Z3_ERR_CUDA, std::string(fn) + ": device ordinal beyond the supported range");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_gather_scratch);
        if (err != cudaSuccess)
            return fail(Z3_ERR_CUDA, std::string(fn) + ": cudaGetSymbolAddress: " +
                                         cudaGetErrorString(err));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return Z3_OK;
}

}  // namespace
}  // namespace z3

using namespace z3;

extern "C" z3_status z3_step_layer_noalloc(const z3_layout *L, uint16_t *shards,
                                           const uint16_t *grads, int64_t grad_stride,
                                           float scale, float *master, float *m, float *v,
                                           const z3_adam_hp *hp, int64_t step,
                                           z3_stream stream) {
    const char *fn = "z3_step_layer_noalloc";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_step_layer_noalloc: layout is NULL");
    if (L->psi > kScratchElems)
        return fail(Z3_ERR_INVALID_ARG,
                    "z3_step_layer_noalloc: the layer has " + std::to_string(L->psi) +
                        " elements, more than the " + std::to_string(kScratchElems) +
                        " the library's gather scratch holds; use z3_step_layer with a "
                        "buffer of your own");
    void *scratch = nullptr;
    if (L->psi > 0) {
        const z3_status st = scratch_address(fn, &scratch);
        if (st != Z3_OK) return st;
    }
    return z3_step_layer(L, shards, static_cast<uint16_t *>(scratch), grads, grad_stride, scale,
                         master, m, v, nullptr, hp, step, stream);
}
