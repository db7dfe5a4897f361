// z3_api.cpp -- the C-ABI entry points of include/z3.h: argument validation
// on the host, NVTX ranges, and the calls into the kernel launchers
// (z3_launch.h, z3_kernels.cu).  No device code here; the whole-model step
// (z3_model_step) orders its launches on two streams with CUDA events.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <cstdint>
#include <string>
#include <vector>

#include "z3_launch.h"

namespace z3 {
namespace {

// --------------------------------------------------------------------------
// argument validation and launch-error reporting
// --------------------------------------------------------------------------

struct Buf {
    const void *ptr;
    int64_t bytes;
    const char *name;
};

z3_status check_bufs(const char *fn, const Buf *bufs, int n) {
    for (int i = 0; i < n; ++i) {
        if (bufs[i].bytes == 0) continue;
        if (bufs[i].ptr == nullptr)
            return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": " + bufs[i].name + " is NULL");
        if (reinterpret_cast<uintptr_t>(bufs[i].ptr) % 16 != 0)
            return fail(Z3_ERR_ALIGNMENT,
                        std::string(fn) + ": " + bufs[i].name + " is not 16-byte aligned");
    }
    for (int i = 0; i < n; ++i) {
        for (int j = i + 1; j < n; ++j) {
            if (bufs[i].bytes == 0 || bufs[j].bytes == 0) continue;
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(bufs[i].ptr);
            const uintptr_t b0 = reinterpret_cast<uintptr_t>(bufs[j].ptr);
            if (a0 < b0 + (uintptr_t)bufs[j].bytes && b0 < a0 + (uintptr_t)bufs[i].bytes)
                return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": " + bufs[i].name +
                                                    " overlaps " + bufs[j].name);
        }
    }
    return Z3_OK;
}

z3_status check_grads(const char *fn, const z3_layout *L, int64_t grad_stride, int64_t *bytes) {
    if (grad_stride < L->psi)
        return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": grad_stride < psi");
    if (grad_stride % kVec != 0)
        return fail(Z3_ERR_ALIGNMENT,
                    std::string(fn) + ": grad_stride is not a multiple of 8 elements");
    int64_t elems;
    if (__builtin_mul_overflow(grad_stride, (int64_t)L->n_ranks, &elems) ||
        __builtin_mul_overflow(elems, (int64_t)2, bytes))
        return fail(Z3_ERR_OVERFLOW, std::string(fn) + ": N * grad_stride overflows");
    return Z3_OK;
}

// The binary32 constants of one Adam step.  Rejected: non-finite values,
// beta1 or beta2 outside [0, 1) (at 1 a bias correction divides by zero),
// eps <= 0 (a pad position, g = m = v = 0, would compute 0/0), negative lr or
// weight decay, and any constant that is not finite in binary32 or an eps
// that rounds to 0 there.
z3_status adam_constants(const char *fn, const z3_adam_hp *hp, int64_t step, AdamK *k) {
    if (hp == nullptr) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": hp is NULL");
    if (step < 1) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": step < 1");
    const double vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : vals)
        if (!std::isfinite(x))
            return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": non-finite hyperparameter");
    if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0) || !(hp->beta2 >= 0.0 && hp->beta2 < 1.0))
        return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": beta1 and beta2 must lie in [0, 1)");
    if (!(hp->eps > 0.0)) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": eps must be > 0");
    if (hp->lr < 0.0 || hp->weight_decay < 0.0)
        return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": lr and weight_decay must be >= 0");
    k->b1 = (float)hp->beta1;
    k->c1 = (float)(1.0 - hp->beta1);
    k->b2 = (float)hp->beta2;
    k->c2 = (float)(1.0 - hp->beta2);
    k->rb1 = (float)(1.0 / (1.0 - std::pow(hp->beta1, (double)step)));
    k->rb2 = (float)(1.0 / (1.0 - std::pow(hp->beta2, (double)step)));
    k->lr = (float)hp->lr;
    k->eps = (float)hp->eps;
    k->lwd = (float)(hp->lr * hp->weight_decay);
    const float consts[9] = {k->b1, k->c1, k->b2, k->c2, k->rb1, k->rb2, k->lr, k->eps, k->lwd};
    for (float x : consts)
        if (!std::isfinite(x))
            return fail(Z3_ERR_INVALID_ARG,
                        std::string(fn) + ": an Adam constant is not finite in binary32");
    if (!(k->eps > 0.0f))
        return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": eps rounds to 0 in binary32");
    return Z3_OK;
}

z3_status launched(const char *fn, cudaError_t err) {
    if (err != cudaSuccess)
        return fail(Z3_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(err));
    return Z3_OK;
}

// Host-side NVTX range around the launches of one call, named after the
// collective it enqueues, so a trace shows the AllGather / ReduceScatter /
// update pattern of "The ZeRO-3 Diagram Most People Remember Is Wrong", s.6.
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

// early: see launch_allgather / launch_reduce.  Only the calls that enqueue
// several dependent launches pass true, for a launch whose stream
// predecessor they enqueued themselves.
z3_status run_allgather(const z3_layout *L, const uint16_t *shards, uint16_t *full,
                        cudaStream_t stream, bool early = false) {
    return launched("z3_allgather", launch_allgather(L, shards, full, stream, early));
}

z3_status run_reduce(const z3_layout *L, const ReduceArgs &a, Mode mode, cudaStream_t stream,
                     const char *fn, bool early = false) {
    return launched(fn, launch_reduce(L, a, mode, stream, early));
}

}  // namespace
}  // namespace z3

using namespace z3;

extern "C" z3_status z3_partition(const z3_layout *L, const float *full, uint16_t *shards,
                                  float *master, float *m, float *v, z3_stream stream) {
    const char *fn = "z3_partition";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_partition: layout is NULL");
    const int64_t T = L->psi_padded;
    const Buf bufs[5] = {{full, 4 * L->psi, "full"}, {shards, 2 * T, "shards"},
                         {master, 4 * T, "master"}, {m, 4 * T, "m"}, {v, 4 * T, "v"}};
    z3_status st = check_bufs(fn, bufs, 5);
    if (st != Z3_OK) return st;
    if (T == 0) return Z3_OK;
    const PartitionArgs a{full, shards, master, m, v};
    return launched(fn, launch_partition(L, a, (cudaStream_t)stream));
}

extern "C" z3_status z3_allgather(const z3_layout *L, const uint16_t *shards, uint16_t *full,
                                  z3_stream stream) {
    const char *fn = "z3_allgather";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_allgather: layout is NULL");
    const Buf bufs[2] = {{shards, 2 * L->psi_padded, "shards"}, {full, 2 * L->psi, "full"}};
    z3_status st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    if (L->psi == 0) return Z3_OK;
    Range range("z3/AllGather");
    return run_allgather(L, shards, full, (cudaStream_t)stream);
}

extern "C" z3_status z3_reduce_scatter(const z3_layout *L, const uint16_t *grads,
                                       int64_t grad_stride, float *grad_shards, float scale,
                                       int32_t accumulate, z3_stream stream) {
    const char *fn = "z3_reduce_scatter";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_reduce_scatter: layout is NULL");
    if (!std::isfinite(scale)) return fail(Z3_ERR_INVALID_ARG, "z3_reduce_scatter: scale");
    int64_t gbytes;
    z3_status st = check_grads(fn, L, grad_stride, &gbytes);
    if (st != Z3_OK) return st;
    const Buf bufs[2] = {{grads, L->psi ? gbytes : 0, "grads"},
                         {grad_shards, 4 * L->psi_padded, "grad_shards"}};
    st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    if (L->psi_padded == 0) return Z3_OK;
    ReduceArgs a{};
    a.grads = grads;
    a.stride = grad_stride;
    a.scale = scale;
    a.out = grad_shards;
    Range range(accumulate ? "z3/ReduceScatter+acc" : "z3/ReduceScatter");
    return run_reduce(L, a, accumulate ? kRSAcc : kRS, (cudaStream_t)stream, fn);
}

extern "C" z3_status z3_adam_shard_step(const z3_layout *L, float *master, float *m, float *v,
                                        const float *grad_shards, uint16_t *shards,
                                        const z3_adam_hp *hp, int64_t step, z3_stream stream) {
    const char *fn = "z3_adam_shard_step";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_adam_shard_step: layout is NULL");
    AdamArgs a{};
    z3_status st = adam_constants(fn, hp, step, &a.k);
    if (st != Z3_OK) return st;
    const int64_t T = L->psi_padded;
    const Buf bufs[5] = {{master, 4 * T, "master"}, {m, 4 * T, "m"}, {v, 4 * T, "v"},
                         {grad_shards, 4 * T, "grad_shards"}, {shards, 2 * T, "shards"}};
    st = check_bufs(fn, bufs, 5);
    if (st != Z3_OK) return st;
    if (T == 0) return Z3_OK;
    a.master = master;
    a.m = m;
    a.v = v;
    a.grad = grad_shards;
    a.shards = shards;
    a.total = T;
    if (flat_blocks(T, kAdamThreads) > 0x7fffffff)
        return fail(Z3_ERR_OVERFLOW, "z3_adam_shard_step: grid too large");
    Range range("z3/Adam(shard)");
    return launched(fn, launch_adam(a, (cudaStream_t)stream));
}

namespace {
z3_status prepare_rs_adam(const char *fn, const z3_layout *L, const uint16_t *grads,
                          int64_t grad_stride, float scale, const float *grad_acc, float *master,
                          float *m, float *v, uint16_t *shards, const uint16_t *extra_full,
                          const z3_adam_hp *hp, int64_t step, ReduceArgs *a,
                          const char *extra_name = "full", float *grad_out = nullptr) {
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": layout is NULL");
    if (!std::isfinite(scale)) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": scale");
    z3_status st = adam_constants(fn, hp, step, &a->k);
    if (st != Z3_OK) return st;
    int64_t gbytes;
    st = check_grads(fn, L, grad_stride, &gbytes);
    if (st != Z3_OK) return st;
    const int64_t T = L->psi_padded;
    const Buf bufs[8] = {{grads, L->psi ? gbytes : 0, "grads"},
                         {master, 4 * T, "master"},
                         {m, 4 * T, "m"},
                         {v, 4 * T, "v"},
                         {shards, 2 * T, "shards"},
                         {grad_acc, grad_acc ? 4 * T : 0, "grad_acc"},
                         {extra_full, extra_full ? 2 * L->psi : 0, extra_name},
                         {grad_out, grad_out ? 4 * T : 0, "grad_shards"}};
    st = check_bufs(fn, bufs, 8);
    if (st != Z3_OK) return st;
    a->out = grad_out;
    a->grads = grads;
    a->stride = grad_stride;
    a->scale = scale;
    a->acc_in = grad_acc;
    a->master = master;
    a->m = m;
    a->v = v;
    a->shards = shards;
    return Z3_OK;
}
// forward AllGather, backward AllGather, then ReduceScatter + Adam.  The
// backward gather's predecessor (the forward gather) writes only `full`, so
// it reads the shards early; the update's predecessor (the backward gather)
// writes only `full`, so it reads gradients and state early.  With a.out set
// the update also stores the reduced gradient and runs plain.
z3_status enqueue_step_layer(const char *fn, const z3_layout *L, const ReduceArgs &a,
                             uint16_t *shards, uint16_t *full, cudaStream_t s) {
    z3_status st;
    {
        Range r1("z3/AllGather(forward)");
        st = run_allgather(L, shards, full, s);
    }
    if (st != Z3_OK) return st;
    {
        Range r2("z3/AllGather(backward)");
        st = run_allgather(L, shards, full, s, true);
    }
    if (st != Z3_OK) return st;
    Range r3("z3/ReduceScatter+Adam");
    return a.out ? run_reduce(L, a, kRSAdamOut, s, fn) : run_reduce(L, a, kRSAdam, s, fn, true);
}
}  // namespace

extern "C" z3_status z3_reduce_scatter_adam(const z3_layout *L, const uint16_t *grads,
                                            int64_t grad_stride, float scale,
                                            const float *grad_acc, float *master, float *m,
                                            float *v, uint16_t *shards, const z3_adam_hp *hp,
                                            int64_t step, z3_stream stream) {
    const char *fn = "z3_reduce_scatter_adam";
    ReduceArgs a{};
    z3_status st = prepare_rs_adam(fn, L, grads, grad_stride, scale, grad_acc, master, m, v,
                                   shards, nullptr, hp, step, &a);
    if (st != Z3_OK) return st;
    if (L->psi_padded == 0) return Z3_OK;
    Range range("z3/ReduceScatter+Adam");
    return run_reduce(L, a, grad_acc ? kRSAccAdam : kRSAdam, (cudaStream_t)stream, fn);
}

extern "C" z3_status z3_step_layer(const z3_layout *L, uint16_t *shards, uint16_t *full,
                                   const uint16_t *grads, int64_t grad_stride, float scale,
                                   float *master, float *m, float *v, float *grad_shards,
                                   const z3_adam_hp *hp, int64_t step, z3_stream stream) {
    const char *fn = "z3_step_layer";
    ReduceArgs a{};
    z3_status st = prepare_rs_adam(fn, L, grads, grad_stride, scale, nullptr, master, m, v,
                                   shards, full, hp, step, &a, "full", grad_shards);
    if (st != Z3_OK) return st;
    if (L->psi_padded == 0) return Z3_OK;
    Range range("z3/step_layer");
    return enqueue_step_layer(fn, L, a, shards, full, (cudaStream_t)stream);
}

extern "C" z3_status z3_allreduce(const z3_layout *L, const uint16_t *grads, int64_t grad_stride,
                                  float *out, float scale, z3_stream stream) {
    const char *fn = "z3_allreduce";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_allreduce: layout is NULL");
    if (!std::isfinite(scale)) return fail(Z3_ERR_INVALID_ARG, "z3_allreduce: scale");
    int64_t gbytes;
    z3_status st = check_grads(fn, L, grad_stride, &gbytes);
    if (st != Z3_OK) return st;
    const Buf bufs[2] = {{grads, L->psi ? gbytes : 0, "grads"}, {out, 4 * L->psi, "out"}};
    st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    if (L->psi == 0) return Z3_OK;
    if (flat_blocks(L->psi, kFlatThreads) > 0x7fffffff)
        return fail(Z3_ERR_OVERFLOW, "z3_allreduce: grid too large");
    const AllreduceArgs a{grads, grad_stride, out, L->psi, scale, L->n_ranks};
    Range range("z3/AllReduce");
    return launched(fn, launch_allreduce(a, (cudaStream_t)stream));
}

extern "C" z3_status z3_scatter(const z3_layout *L, const float *full, float *shards,
                                z3_stream stream) {
    const char *fn = "z3_scatter";
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_scatter: layout is NULL");
    const Buf bufs[2] = {{full, 4 * L->psi, "full"}, {shards, 4 * L->psi_padded, "shards"}};
    z3_status st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    if (L->psi_padded == 0) return Z3_OK;
    const ScatterArgs a{full, shards};
    return launched(fn, launch_scatter(L, a, (cudaStream_t)stream));
}

extern "C" z3_status z3_reshard(const z3_layout *Ls, const z3_layout *Ld, int32_t elem_bytes,
                                const void *src, void *dst, z3_stream stream) {
    const char *fn = "z3_reshard";
    if (Ls == nullptr || Ld == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_reshard: layout is NULL");
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(Z3_ERR_INVALID_ARG, "z3_reshard: elem_bytes must be 2 or 4");
    if (Ls->n_params != Ld->n_params || Ls->numel != Ld->numel)
        return fail(Z3_ERR_INVALID_ARG, "z3_reshard: the layouts describe different parameters");
    const Buf bufs[2] = {{src, elem_bytes * Ls->psi_padded, "src"},
                         {dst, elem_bytes * Ld->psi_padded, "dst"}};
    z3_status st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    if (Ld->psi_padded == 0) return Z3_OK;
    Range range("z3/Reshard");
    return launched(fn, launch_reshard(Ls, Ld, elem_bytes, src, dst, (cudaStream_t)stream));
}

namespace {
// Events used by one prefetching model step; destroyed when the step has
// been enqueued (the runtime releases them once their work completes).
struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
    cudaError_t make(int n) {
        for (int i = 0; i < n; ++i) {
            cudaEvent_t e;
            const cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (err != cudaSuccess) return err;
            ev.push_back(e);
        }
        return cudaSuccess;
    }
};
}  // namespace

namespace {
// The body of z3_model_step.  Every host allocation happens before the
// first launch, so a std::bad_alloc (thrown out of here) leaves nothing
// enqueued.
z3_status model_step(const z3_unit *units, int32_t n_units, uint16_t *const *full,
                     int32_t n_full, const z3_adam_hp *hp, int64_t step, z3_stream stream,
                     z3_stream gather_stream) {
    const char *fn = "z3_model_step";
    if (units == nullptr || n_units < 1)
        return fail(Z3_ERR_INVALID_ARG, "z3_model_step: no units");
    if (full == nullptr || n_full < 1 || n_full > 8)
        return fail(Z3_ERR_INVALID_ARG, "z3_model_step: n_full must be 1..8");
    if (n_full >= 2 && (gather_stream == nullptr || gather_stream == stream))
        return fail(Z3_ERR_INVALID_ARG,
                    "z3_model_step: prefetch needs a gather stream distinct from stream");
    // the transient buffers hold the largest unit that is gathered through them
    int64_t full_bytes = 0;
    for (int32_t i = 0; i < n_units; ++i) {
        if (units[i].layout == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_model_step: layout is NULL");
        if (units[i].resident == nullptr) full_bytes = std::max(full_bytes, 2 * units[i].layout->psi);
    }
    std::vector<ReduceArgs> args((size_t)n_units);
    std::vector<int64_t> grad_bytes((size_t)n_units, 0);
    for (int32_t i = 0; i < n_units; ++i) {
        const z3_unit &u = units[i];
        z3_status st = prepare_rs_adam(fn, u.layout, u.grads, u.grad_stride, u.scale, nullptr,
                                       u.master, u.m, u.v, u.shards, u.resident,
                                       u.hp != nullptr ? u.hp : hp, step, &args[i], "resident");
        if (st != Z3_OK) return st;
        const int64_t T = u.layout->psi_padded;
        int64_t gbytes = 0;
        st = check_grads(fn, u.layout, u.grad_stride, &gbytes);
        if (st != Z3_OK) return st;
        grad_bytes[(size_t)i] = u.layout->psi ? gbytes : 0;
        for (int32_t k = 0; k < n_full; ++k) {
            const Buf bufs[7] = {{full[k], full_bytes, "full[k]"},
                                 {u.resident, u.resident ? 2 * u.layout->psi : 0, "resident"},
                                 {u.shards, 2 * T, "shards"},
                                 {u.master, 4 * T, "master"},
                                 {u.m, 4 * T, "m"},
                                 {u.v, 4 * T, "v"},
                                 {u.grads, u.layout->psi ? gbytes : 0, "grads"}};
            st = check_bufs(fn, bufs, 7);
            if (st != Z3_OK) return st;
            for (int32_t j = 0; j < k; ++j) {
                const Buf pair[2] = {{full[k], full_bytes, "full[k]"},
                                     {full[j], full_bytes, "full[j]"}};
                st = check_bufs(fn, pair, 2);
                if (st != Z3_OK) return st;
            }
        }
    }
    // The units' written buffers must be disjoint from every buffer of every
    // other unit: a launch then never reads what its stream predecessor (a
    // launch of another unit, or of this unit's gather) writes, which lets
    // the gathers read shards and the updates read gradients and state
    // before they wait for that predecessor.  Units may share read-only
    // gradients.  A sweep over the buffers sorted by address finds every
    // overlap in O(B log B) for B buffers (plus the overlaps themselves).
    {
        struct Span {
            uintptr_t lo, hi;
            int32_t unit;
            bool written;
            const char *name;
        };
        std::vector<Span> spans;
        spans.reserve((size_t)n_units * 6);
        auto add = [&](const void *p, int64_t bytes, int32_t unit, bool written,
                       const char *name) {
            if (bytes <= 0) return;
            const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
            spans.push_back({lo, lo + (uintptr_t)bytes, unit, written, name});
        };
        for (int32_t i = 0; i < n_units; ++i) {
            const z3_unit &u = units[i];
            const int64_t T = u.layout->psi_padded;
            add(u.shards, 2 * T, i, true, "shards");
            add(u.master, 4 * T, i, true, "master");
            add(u.m, 4 * T, i, true, "m");
            add(u.v, 4 * T, i, true, "v");
            add(u.resident, u.resident ? 2 * u.layout->psi : 0, i, true, "resident copy");
            add(u.grads, grad_bytes[(size_t)i], i, false, "grads");
        }
        std::sort(spans.begin(), spans.end(),
                  [](const Span &a, const Span &b) { return a.lo < b.lo; });
        std::vector<const Span *> open;   // spans that may still overlap the next one
        for (const Span &x : spans) {
            size_t keep = 0;
            for (const Span *y : open) {
                if (y->hi <= x.lo) continue;  // ended before x starts
                open[keep++] = y;
                if (y->unit != x.unit && (y->written || x.written))
                    return fail(Z3_ERR_INVALID_ARG,
                                std::string(fn) + ": unit " + std::to_string(y->unit) + "'s " +
                                    y->name + " overlaps another unit's (" +
                                    std::to_string(x.unit) + ") " + x.name);
            }
            open.resize(keep);
            open.push_back(&x);
        }
    }
    const cudaStream_t s = (cudaStream_t)stream;
    const int nb = n_full;
    std::vector<bool> buffer_used((size_t)nb, false);
    Events E;
    E.ev.reserve((size_t)(2 + 2 * nb));
    Range range("z3/model_step");
    z3_status st = Z3_OK;
    // whether this call has enqueued a kernel on s (on g) yet: a launch may
    // read early only after one of its own
    bool ours_s = false, ours_g = false;
    // the update of unit i; a resident unit is gathered into its own copy
    // right after it, on the same stream (that gather reads the shards the
    // update just wrote, so it never reads early)
    auto update = [&](int32_t i) -> z3_status {
        const z3_layout *L = units[i].layout;
        if (L->psi_padded == 0) return Z3_OK;
        z3_status us;
        {
            Range r("z3/ReduceScatter+Adam");
            us = run_reduce(L, args[i], kRSAdam, s, fn, ours_s);
            ours_s = true;
        }
        if (us != Z3_OK || units[i].resident == nullptr || L->psi == 0) return us;
        Range r("z3/AllGather(resident)");
        return run_allgather(L, units[i].shards, units[i].resident, s, false);
    };
    if (n_full == 1) {
        for (int32_t i = 0; i < n_units && st == Z3_OK; ++i) {
            Range r("z3/AllGather(forward)");
            if (units[i].layout->psi && !units[i].resident) {
                st = run_allgather(units[i].layout, units[i].shards, full[0], s, ours_s);
                ours_s = true;
            }
        }
        for (int32_t i = n_units - 1; i >= 0 && st == Z3_OK; --i) {
            const z3_layout *L = units[i].layout;
            if (L->psi && !units[i].resident) {
                Range r("z3/AllGather(backward)");
                st = run_allgather(L, units[i].shards, full[0], s, ours_s);
                ours_s = true;
            }
            if (st == Z3_OK) st = update(i);
        }
        return st;
    }
    // Prefetch depth D = n_full - 1: the gathers run on gather_stream up to
    // D units ahead of the updates, unit i in buffer i mod n_full.  A gather
    // into a buffer waits until the update of the unit that used it last
    // (n_full units later in backward order) has run; an update waits for its
    // unit's gather.  Gathers are enqueued before the update they run beside,
    // so their small grids reach the GPU first.
    // Events: 0 = entry, 1 = gathers done, 2.. = gathered[b], then freed[b].
    const cudaStream_t g = (cudaStream_t)gather_stream;
    cudaError_t err = E.make(2 + 2 * nb);
    auto cuda_fail = [&](cudaError_t e) {
        return fail(Z3_ERR_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
    };
    auto gathered = [&](int b) { return E.ev[2 + b]; };
    auto freed = [&](int b) { return E.ev[2 + nb + b]; };
    if (err != cudaSuccess) return cuda_fail(err);
    if ((err = cudaEventRecord(E.ev[0], s)) != cudaSuccess) return cuda_fail(err);
    if ((err = cudaStreamWaitEvent(g, E.ev[0], 0)) != cudaSuccess) return cuda_fail(err);
    for (int32_t i = 0; i < n_units && st == Z3_OK; ++i) {
        Range r("z3/AllGather(forward)");
        if (units[i].layout->psi && !units[i].resident) {
            st = run_allgather(units[i].layout, units[i].shards, full[i % nb], g, ours_g);
            ours_g = true;
        }
    }
    auto gather = [&](int32_t i) -> z3_status {
        const int b = i % nb;
        if (buffer_used[b]) {   // the unit that last used this buffer has been updated
            cudaError_t e = cudaStreamWaitEvent(g, freed(b), 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        Range r("z3/AllGather(backward)");
        z3_status gs = Z3_OK;
        if (units[i].layout->psi && !units[i].resident) {
            gs = run_allgather(units[i].layout, units[i].shards, full[b], g, ours_g);
            ours_g = true;
        }
        if (gs != Z3_OK) return gs;
        cudaError_t e = cudaEventRecord(gathered(b), g);
        return e == cudaSuccess ? Z3_OK : cuda_fail(e);
    };
    const int depth = nb - 1;
    int32_t next = n_units - 1;   // next unit to gather (backward order)
    for (int32_t i = n_units - 1; i >= 0 && st == Z3_OK; --i) {
        while (st == Z3_OK && next >= 0 && next >= i - depth) st = gather(next--);
        if (st != Z3_OK) break;
        if ((err = cudaStreamWaitEvent(s, gathered(i % nb), 0)) != cudaSuccess) return cuda_fail(err);
        st = update(i);
        if (st != Z3_OK) break;
        if ((err = cudaEventRecord(freed(i % nb), s)) != cudaSuccess) return cuda_fail(err);
        buffer_used[i % nb] = true;
    }
    if (st != Z3_OK) return st;
    if ((err = cudaEventRecord(E.ev[1], g)) != cudaSuccess) return cuda_fail(err);
    if ((err = cudaStreamWaitEvent(s, E.ev[1], 0)) != cudaSuccess) return cuda_fail(err);
    return Z3_OK;
}
}  // namespace

extern "C" z3_status z3_model_step(const z3_unit *units, int32_t n_units, uint16_t *const *full,
                                   int32_t n_full, const z3_adam_hp *hp, int64_t step,
                                   z3_stream stream, z3_stream gather_stream) {
    try {
        return model_step(units, n_units, full, n_full, hp, step, stream, gather_stream);
    } catch (const std::bad_alloc &) {
        return fail_host_memory("z3_model_step");
    }
}

// --------------------------------------------------------------------------
// the layer step fed from host memory
// --------------------------------------------------------------------------

struct z3_host_step {
    const z3_layout *L = nullptr;
    uint16_t *staging[2] = {nullptr, nullptr};
    int64_t stride = 0;
    int64_t grad_bytes = 0;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t done[2] = {nullptr, nullptr};  // the step that last read staging[b] has run
    cudaEvent_t uploaded = nullptr;            // this call's upload has landed
    cudaEvent_t read = nullptr;                // the last download has finished
    bool done_valid[2] = {false, false};
    bool read_valid = false;
    int64_t calls = 0;

    ~z3_host_step() {
        for (cudaEvent_t e : {done[0], done[1], uploaded, read})
            if (e != nullptr) cudaEventDestroy(e);
    }
};

extern "C" z3_status z3_host_step_create(const z3_layout *L, uint16_t *staging0,
                                         uint16_t *staging1, int64_t grad_stride,
                                         z3_stream upload_stream, z3_stream download_stream,
                                         z3_host_step **out) {
    const char *fn = "z3_host_step_create";
    if (out == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_host_step_create: out is NULL");
    *out = nullptr;
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_host_step_create: layout is NULL");
    if (upload_stream == nullptr || download_stream == nullptr || upload_stream == download_stream)
        return fail(Z3_ERR_INVALID_ARG,
                    "z3_host_step_create: upload and download streams must be two distinct "
                    "non-NULL streams");
    int64_t gbytes;
    z3_status st = check_grads(fn, L, grad_stride, &gbytes);
    if (st != Z3_OK) return st;
    // a zero-element layer still needs two distinct staging pointers
    const int64_t b = gbytes > 0 ? gbytes : 16;
    const Buf bufs[2] = {{staging0, b, "staging0"}, {staging1, b, "staging1"}};
    st = check_bufs(fn, bufs, 2);
    if (st != Z3_OK) return st;
    auto *p = new (std::nothrow) z3_host_step();
    if (p == nullptr) return fail_host_memory(fn);
    p->L = L;
    p->staging[0] = staging0;
    p->staging[1] = staging1;
    p->stride = grad_stride;
    p->grad_bytes = gbytes;
    p->up = (cudaStream_t)upload_stream;
    p->down = (cudaStream_t)download_stream;
    for (cudaEvent_t *e : {&p->done[0], &p->done[1], &p->uploaded, &p->read}) {
        const cudaError_t err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        if (err != cudaSuccess) {
            delete p;
            return launched(fn, err);
        }
    }
    *out = p;
    return Z3_OK;
}

extern "C" z3_status z3_host_step_run(z3_host_step *p, const uint16_t *grads_host,
                                      uint16_t *shards, uint16_t *full, float scale,
                                      float *master, float *m, float *v, const z3_adam_hp *hp,
                                      int64_t step, uint16_t *shards_host, z3_stream stream) {
    const char *fn = "z3_host_step_run";
    if (p == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_host_step_run: pipeline is NULL");
    const cudaStream_t s = (cudaStream_t)stream;
    if (s == p->up || s == p->down)
        return fail(Z3_ERR_INVALID_ARG,
                    "z3_host_step_run: stream must differ from the pipeline's streams");
    const z3_layout *L = p->L;
    const int b = (int)(p->calls & 1);
    ReduceArgs a{};
    z3_status st = prepare_rs_adam(fn, L, p->staging[b], p->stride, scale, nullptr, master, m,
                                   v, shards, full, hp, step, &a);
    if (st != Z3_OK) return st;
    const int64_t T = L->psi_padded;
    const Buf dev[6] = {{p->staging[1 - b], p->grad_bytes, "the other staging buffer"},
                        {shards, 2 * T, "shards"},
                        {master, 4 * T, "master"},
                        {m, 4 * T, "m"},
                        {v, 4 * T, "v"},
                        {full, 2 * L->psi, "full"}};
    st = check_bufs(fn, dev, 6);
    if (st != Z3_OK) return st;
    if (p->grad_bytes > 0 && grads_host == nullptr)
        return fail(Z3_ERR_INVALID_ARG, "z3_host_step_run: grads_host is NULL");
    Range range("z3/host_step");
    cudaError_t err = cudaSuccess;
    auto ok = [&](cudaError_t e) { err = e; return e == cudaSuccess; };
    // upload into staging[b] once the step that last read it has run
    if (p->done_valid[b] && !ok(cudaStreamWaitEvent(p->up, p->done[b], 0))) return launched(fn, err);
    if (p->grad_bytes > 0) {
        Range r("z3/upload gradients");
        if (!ok(cudaMemcpyAsync(p->staging[b], grads_host, (size_t)p->grad_bytes,
                                cudaMemcpyHostToDevice, p->up)))
            return launched(fn, err);
    }
    if (!ok(cudaEventRecord(p->uploaded, p->up))) return launched(fn, err);
    // the step: after its upload, and after the previous download of the shards it rewrites
    if (!ok(cudaStreamWaitEvent(s, p->uploaded, 0))) return launched(fn, err);
    if (p->read_valid && !ok(cudaStreamWaitEvent(s, p->read, 0))) return launched(fn, err);
    if (T > 0) {
        st = enqueue_step_layer(fn, L, a, shards, full, s);
        if (st != Z3_OK) return st;
    }
    if (!ok(cudaEventRecord(p->done[b], s))) return launched(fn, err);
    p->done_valid[b] = true;
    p->calls += 1;
    if (shards_host != nullptr && T > 0) {
        Range r("z3/download parameters");
        if (!ok(cudaStreamWaitEvent(p->down, p->done[b], 0))) return launched(fn, err);
        if (!ok(cudaMemcpyAsync(shards_host, shards, (size_t)(2 * T), cudaMemcpyDeviceToHost,
                                p->down)))
            return launched(fn, err);
        if (!ok(cudaEventRecord(p->read, p->down))) return launched(fn, err);
        p->read_valid = true;
    }
    return Z3_OK;
}

extern "C" void z3_host_step_destroy(z3_host_step *p) { delete p; }
