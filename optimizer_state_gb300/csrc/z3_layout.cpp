// z3_layout.cpp -- host side of the C ABI: layout construction (flatten, pad,
// contiguous slice per rank), byte accounting, launch tables and errors.
//
// Layout ("The ZeRO-3 Diagram Most People Remember Is Wrong", s.2 "The
// Actual Parameter Partition"; "ZeRO Stages: Sharding Optimizer State,
// Gradients, and Parameters", "What stage 1 partitions"): parameter p of
// n_p elements is padded to N*s_p with s_p = ceil(n_p/N); rank r owns
// padded positions [r*s_p, (r+1)*s_p); a rank's shard concatenates its
// slices in parameter order with no gaps.
#include <algorithm>
#include <cstring>
#include <limits>
#include <memory>
#include <new>

#include "z3_internal.h"

namespace z3 {

namespace {
thread_local std::string g_last_error;

bool add_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_add_overflow(a, b, out); }
bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }

int64_t ceil_div(int64_t a, int64_t b) { return a / b + (a % b != 0); }

int64_t floor8(int64_t x) { return x >= 0 ? x / kVec : -((-x + kVec - 1) / kVec); }

// Aligned vectors that intersect [begin, begin + len), len > 0.
int64_t vectors_spanned(int64_t begin, int64_t len) {
    return floor8(begin + len - 1) - floor8(begin) + 1;
}

// Builds the launch tables of one kernel family.  `gather` selects the
// driving index space: the unpadded full buffer (chunk (p, r) is
// [F_p + r*s_p, + valid length)) or the shard buffers (chunk (p, r) is
// [r*S + o_p, + s_p), pad included).
z3_status build_tabs(z3_layout *L, bool gather, int64_t vec_per_tile, std::vector<Tab> *out) {
    out->clear();
    Tab cur{};
    bool cur_misaligned = false;
    auto reset = [&]() {
        std::memset(&cur, 0, sizeof cur);
        cur_misaligned = false;
        cur.n_ranks = L->n_ranks;
        cur.S = L->S;
        cur.total = L->psi_padded;
    };
    reset();
    const int64_t N = L->n_ranks;
    for (int32_t p = 0; p < L->n_params; ++p) {
        const int64_t n = L->numel[p], s = L->shard_numel[p];
        const int64_t o = L->shard_off[p], F = L->full_off[p];
        if (n == 0) continue;
        int64_t nvmax = 0;
        bool misaligned_p = false;
        for (int64_t r = 0; r < N; ++r) {
            // element offset between the two index spaces of chunk (p, r)
            const int64_t delta = F + r * s - (r * L->S + o);
            if (delta % kVec != 0) misaligned_p = true;
            int64_t nv = 0;
            if (gather) {
                int64_t len = std::min(s, std::max<int64_t>(0, n - r * s));
                if (len > 0) nv = vectors_spanned(F + r * s, len);
            } else {
                nv = vectors_spanned(r * L->S + o, s);
            }
            nvmax = std::max(nvmax, nv);
        }
        const int64_t tpc = ceil_div(nvmax, vec_per_tile);
        int64_t tiles_p;
        if (!mul_ok(tpc, N, &tiles_p))
            return fail(Z3_ERR_OVERFLOW, "tile count overflows int64");
        if (cur.count == kTabMax ||
            cur.tiles + tiles_p > (int64_t)std::numeric_limits<int32_t>::max()) {
            if (cur.count == 0)
                return fail(Z3_ERR_OVERFLOW, "one parameter needs more than 2^31-1 CTAs");
            out->push_back(cur);
            reset();
        }
        cur_misaligned = cur_misaligned || misaligned_p;
        cur.phase0 = cur_misaligned ? 0 : 1;
        TabEntry &e = cur.e[cur.count++];
        e.n = n;
        e.s = s;
        e.o = o;
        e.F = F;
        e.tile0 = cur.tiles;
        e.tpc = tpc;
        cur.tiles += tiles_p;
    }
    if (cur.count > 0) out->push_back(cur);
    return Z3_OK;
}
}  // namespace

z3_status fail(z3_status st, const std::string &msg) {
    try {
        g_last_error = msg;
    } catch (const std::bad_alloc &) {
        g_last_error.clear();
    }
    return st;
}

z3_status fail_host_memory(const char *fn) noexcept {
    try {
        g_last_error = std::string(fn) + ": out of host memory";
    } catch (...) {
        g_last_error.clear();
    }
    return Z3_ERR_HOST_MEMORY;
}

void clear_error() { g_last_error.clear(); }

}  // namespace z3

using namespace z3;

namespace {
// The body of z3_layout_create (arguments checked).  A failed allocation
// throws std::bad_alloc out of here; the partial layout is released first.
z3_status layout_create(const int64_t *numel, int32_t n_params, int32_t n_ranks,
                        z3_layout **out) {
    std::unique_ptr<z3_layout> owner(new z3_layout());
    z3_layout *L = owner.get();
    L->n_params = n_params;
    L->n_ranks = n_ranks;
    L->numel.resize(n_params);
    L->shard_numel.resize(n_params);
    L->shard_off.resize(n_params);
    L->full_off.resize(n_params);
    int64_t S = 0, psi = 0;
    for (int32_t p = 0; p < n_params; ++p) {
        const int64_t n = numel[p];
        if (n < 0)
            return fail(Z3_ERR_INVALID_ARG, "z3_layout_create: numel[" + std::to_string(p) + "] < 0");
        const int64_t s = ceil_div(n, n_ranks);
        L->numel[p] = n;
        L->shard_numel[p] = s;
        L->shard_off[p] = S;
        L->full_off[p] = psi;
        if (!add_ok(S, s, &S) || !add_ok(psi, n, &psi))
            return fail(Z3_ERR_OVERFLOW, "z3_layout_create: element count overflows int64");
    }
    int64_t total, bytes;
    // every [N][S] buffer must be addressable in bytes at fp32 width
    if (!mul_ok(S, n_ranks, &total) || !mul_ok(total, 4, &bytes) || !mul_ok(psi, 4, &bytes))
        return fail(Z3_ERR_OVERFLOW, "z3_layout_create: N*S overflows int64");
    L->S = S;
    L->psi = psi;
    L->psi_padded = total;
    z3_status st = build_tabs(L, true, (int64_t)kGatherThreads * kGatherVecPerThread,
                              &L->gather_tabs);
    if (st == Z3_OK)
        st = build_tabs(L, false, (int64_t)kReduceThreads * kReduceVecPerThread, &L->reduce_tabs);
    if (st != Z3_OK) return st;
    *out = owner.release();
    clear_error();
    return Z3_OK;
}
}  // namespace

extern "C" z3_status z3_layout_create(const int64_t *numel, int32_t n_params, int32_t n_ranks,
                                      z3_layout **out) {
    if (out == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_layout_create: out is NULL");
    *out = nullptr;
    if (numel == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_layout_create: numel is NULL");
    if (n_params < 1) return fail(Z3_ERR_INVALID_ARG, "z3_layout_create: n_params < 1");
    if (n_ranks < 1) return fail(Z3_ERR_INVALID_ARG, "z3_layout_create: n_ranks < 1");
    try {
        return layout_create(numel, n_params, n_ranks, out);
    } catch (const std::bad_alloc &) {
        return fail_host_memory("z3_layout_create");
    }
}

extern "C" void z3_layout_destroy(z3_layout *layout) { delete layout; }

extern "C" z3_status z3_layout_info(const z3_layout *L, int32_t *n_params, int32_t *n_ranks,
                                    int64_t *S, int64_t *psi, int64_t *psi_padded) {
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_layout_info: layout is NULL");
    if (n_params) *n_params = L->n_params;
    if (n_ranks) *n_ranks = L->n_ranks;
    if (S) *S = L->S;
    if (psi) *psi = L->psi;
    if (psi_padded) *psi_padded = L->psi_padded;
    return Z3_OK;
}

extern "C" z3_status z3_layout_params(const z3_layout *L, int64_t *numel, int64_t *shard_numel,
                                      int64_t *shard_off, int64_t *full_off) {
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_layout_params: layout is NULL");
    const size_t bytes = sizeof(int64_t) * (size_t)L->n_params;
    if (numel) std::memcpy(numel, L->numel.data(), bytes);
    if (shard_numel) std::memcpy(shard_numel, L->shard_numel.data(), bytes);
    if (shard_off) std::memcpy(shard_off, L->shard_off.data(), bytes);
    if (full_off) std::memcpy(full_off, L->full_off.data(), bytes);
    return Z3_OK;
}

extern "C" z3_status z3_stats(const z3_layout *L, z3_traffic *out) {
    if (L == nullptr || out == nullptr) return fail(Z3_ERR_INVALID_ARG, "z3_stats: NULL argument");
    const int64_t psi = L->psi, N = L->n_ranks;
    z3_traffic t{};
    t.psi = psi;
    // "ZeRO Stage 3: Parameter Partitioning", communication list: a gather
    // or a reduction moves one 2-byte copy of the layer.
    t.ag_payload_bytes = 2 * psi;
    t.rs_payload_bytes = 2 * psi;
    t.step_volume_bytes = t.ag_payload_bytes * 2 + t.rs_payload_bytes;
    t.dp_allreduce_bytes = 2 * psi;
    // HBM bytes each kernel must move per unpadded element.
    t.hbm_allgather = 4 * psi;
    t.hbm_reduce_scatter = (2 * N + 4) * psi;
    t.hbm_reduce_scatter_accumulate = (2 * N + 8) * psi;
    t.hbm_adam = 30 * psi;
    t.hbm_reduce_scatter_adam = (2 * N + 26) * psi;
    t.hbm_step_layer = 2 * t.hbm_allgather + t.hbm_reduce_scatter_adam;
    // eq. M_Stage3: 2 (param) + 2 (grad) + 4 + 4 + 4 bytes per owned element.
    t.state_bytes_per_rank = 16 * L->S;
    t.state_bytes_per_rank_fp32_grad = 18 * L->S;
    *out = t;
    return Z3_OK;
}

extern "C" const char *z3_status_string(z3_status st) {
    switch (st) {
        case Z3_OK: return "Z3_OK";
        case Z3_ERR_INVALID_ARG: return "Z3_ERR_INVALID_ARG";
        case Z3_ERR_ALIGNMENT: return "Z3_ERR_ALIGNMENT";
        case Z3_ERR_OVERFLOW: return "Z3_ERR_OVERFLOW";
        case Z3_ERR_CUDA: return "Z3_ERR_CUDA";
        case Z3_ERR_HOST_MEMORY: return "Z3_ERR_HOST_MEMORY";
    }
    return "Z3_ERR_UNKNOWN";
}

extern "C" size_t z3_last_error(char *buf, size_t len) {
    const std::string &msg = g_last_error;
    if (buf != nullptr && len > 0) {
        size_t n = std::min(len - 1, msg.size());
        std::memcpy(buf, msg.data(), n);
        buf[n] = '\0';
    }
    return msg.size();
}
