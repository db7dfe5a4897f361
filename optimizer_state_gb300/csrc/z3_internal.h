// z3_internal.h -- host-side layout object and the per-launch parameter
// tables shared by the host code (z3_layout.cpp) and the kernels
// (z3_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/z3.h"

namespace z3 {

// Elements per 16-byte vector of bf16; every kernel walks 8-element aligned
// groups ("vectors") of its driving index space.
constexpr int kVec = 8;

// One parameter's slice of a launch table.  A tile is the work of one CTA:
// `vec_per_tile` consecutive aligned vectors of one (parameter, rank) chunk.
struct TabEntry {
    int64_t n;      // n_p
    int64_t s;      // s_p
    int64_t o;      // o_p
    int64_t F;      // F_p
    int64_t tile0;  // first tile of this parameter within the launch
    int64_t tpc;    // tiles per (parameter, rank) chunk
};

constexpr int kTabMax = 40;  // parameters per launch (kernel-parameter space)

struct Tab {
    int32_t count;    // entries used
    int32_t n_ranks;  // N
    int32_t phase0;   // 1 when every chunk's two index spaces agree mod 8
    int32_t pad_;
    int64_t S;        // rank stride
    int64_t total;    // N * S, elements of every [N][S] buffer
    int64_t tiles;    // tiles (CTAs) of this launch
    TabEntry e[kTabMax];
};

// Tile geometry of each kernel family (threads x vectors per thread).
constexpr int kGatherThreads = 256;
constexpr int kGatherVecPerThread = 2;
constexpr int kReduceThreads = 128;
constexpr int kReduceVecPerThread = 1;

}  // namespace z3

struct z3_layout {
    int32_t n_params = 0;
    int32_t n_ranks = 0;
    std::vector<int64_t> numel, shard_numel, shard_off, full_off;
    int64_t S = 0, psi = 0, psi_padded = 0;
    // Launch tables: gather tiles walk the full (unpadded) index space,
    // reduce tiles walk the shard index space.
    std::vector<z3::Tab> gather_tabs;
    std::vector<z3::Tab> reduce_tabs;
};

namespace z3 {

// Thread-local last-error message.
z3_status fail(z3_status st, const std::string &msg);
void clear_error();
// Z3_ERR_HOST_MEMORY with the message "<fn>: out of host memory" (or no
// message, if even that cannot be stored).  Allocates nothing that can throw.
z3_status fail_host_memory(const char *fn) noexcept;

}  // namespace z3
