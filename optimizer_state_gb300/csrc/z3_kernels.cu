// z3_kernels.cu -- sm_103a kernels of the ZeRO-3 sharded layer step and the
// device entry points of the C ABI (include/z3.h).
//
// The N logical ranks are shard regions of this GPU's HBM, so the
// collectives of "The ZeRO-3 Diagram Most People Remember Is Wrong", s.3
// ("AllGather parameter -> compute", "ReduceScatter gradients", "optimizer
// updates local shard") are data-movement kernels.  All of them are bound by
// HBM bandwidth: no tensor cores, no contraction.
//
// Work decomposition.  Every kernel walks one index space in aligned groups
// of 8 elements ("vectors": 16 bytes of bf16, 32 bytes of fp32):
//   gather:  the unpadded full buffer; chunk (p, r) = [F_p + r*s_p, + len_r)
//   reduce:  the [N][S] shard space;   chunk (p, r) = [r*S + o_p, + s_p)
// where len_r = clamp(n_p - r*s_p, 0, s_p) is the valid (non-pad) length.
// Inside chunk (p, r) the two spaces differ by a constant element offset
//   delta = F_p + r*s_p - (r*S + o_p)      (full index = shard index + delta)
// A CTA owns one tile: a run of consecutive vectors of one chunk; a host-built
// table (kernel parameter) maps blockIdx.x to (p, r, tile).  A vector that
// lies wholly in the chunk's valid range takes the vector path: 16-byte
// loads and stores, with the other space's data funnel-shifted into place when
// delta is not a multiple of 8 (the phase).  Vectors at a chunk edge or in the
// pad take an element-wise path that touches only the chunk's own elements,
// so neighbouring chunks never write the same byte.
//
// Numerics match the definitions in include/z3.h: bf16 -> fp32 is exact;
// the rank fold adds in ascending rank order; every float operation is an
// explicit round-to-nearest intrinsic (no contraction into fused multiply-
// add; the file is also built with -fmad=false); division and square root
// are CUDA's IEEE-rounded __fdiv_rn / __fsqrt_rn; fp32 -> bf16 is CUDA's
// round-to-nearest-even conversion.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdint>
#include <string>
#include <vector>

#include "z3_internal.h"

namespace z3 {
namespace {

// --------------------------------------------------------------------------
// small device helpers
// --------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void unpack8(const uint4 &w, float f[8]) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
    f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

__device__ __forceinline__ uint4 ld_nc(const uint16_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Elements [PHI, PHI+8) of the 16-element window (lo, hi) of bf16 values.
template <int PHI>
__device__ __forceinline__ uint4 window8(const uint4 &lo, const uint4 &hi) {
    if constexpr (PHI == 0) {
        return lo;
    } else {
        const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        constexpr int q = PHI >> 1;
        uint4 r;
        if constexpr ((PHI & 1) != 0) {
            r.x = __funnelshift_r(w[q], w[q + 1], 16);
            r.y = __funnelshift_r(w[q + 1], w[q + 2], 16);
            r.z = __funnelshift_r(w[q + 2], w[q + 3], 16);
            r.w = __funnelshift_r(w[q + 3], w[q + 4], 16);
        } else {
            r.x = w[q];
            r.y = w[q + 1];
            r.z = w[q + 2];
            r.w = w[q + 3];
        }
        return r;
    }
}

// Binary32 constants of one Adam step (each rounded once on the host).
struct AdamK {
    float b1, c1, b2, c2, rb1, rb2, lr, eps, lwd;
};

// Kingma & Ba, Algorithm 1, in the order fixed by include/z3.h.
__device__ __forceinline__ void adam1(float g, float &p, float &m, float &v, const AdamK &k) {
    const float m1 = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.c1, g));
    const float v1 = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.c2, __fmul_rn(g, g)));
    const float mh = __fmul_rn(m1, k.rb1);
    const float vh = __fmul_rn(v1, k.rb2);
    const float u = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), k.eps));
    const float pd = __fsub_rn(p, __fmul_rn(k.lwd, p));
    p = __fsub_rn(pd, __fmul_rn(k.lr, u));
    m = m1;
    v = v1;
}

// Maps blockIdx.x to (table entry, rank, tile within the chunk).
struct TileRef {
    int p;
    int64_t r;
    int64_t t;
};

__device__ __forceinline__ TileRef locate(const Tab &tab, int64_t g) {
    int lo = 0, hi = tab.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab.e[mid].tile0 <= g) lo = mid; else hi = mid - 1;
    }
    const int64_t local = g - tab.e[lo].tile0;
    const int64_t tpc = tab.e[lo].tpc;
    const int64_t r = local / tpc;
    return TileRef{lo, r, local - r * tpc};
}

// Programmatic dependent launch.  Every kernel lets the next kernel of the
// stream launch at once (its CTAs then wait), and waits for the previous
// kernel to complete -- memory included -- before its first global memory
// access.  Ordering between the calls is therefore exactly stream order; only
// the launch latency of a kernel overlaps the tail of the one before it.
// Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------------------
// AllGather: full[F_p + i] = shards[i / s_p][o_p + i mod s_p]
// --------------------------------------------------------------------------

struct GatherArgs {
    const uint16_t *__restrict__ shards;
    uint16_t *__restrict__ full;
};

template <int PHI>
__device__ __forceinline__ void gather_tile(const Tab &tab, const GatherArgs &a, int64_t d0,
                                            int64_t len, int64_t delta, int64_t qbeg,
                                            int64_t qend) {
    constexpr int VPT = kGatherVecPerThread;
    uint4 val[VPT];
    bool fast[VPT];
    int64_t x0[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t q = qbeg + (int64_t)i * kGatherThreads + threadIdx.x;
        x0[i] = q * kVec;
        fast[i] = false;
        if (q < qend && x0[i] >= d0 && x0[i] + kVec <= d0 + len) {
            const int64_t src = x0[i] - delta - PHI;  // aligned: x0 - delta == PHI (mod 8)
            if (PHI == 0 || src + 2 * kVec <= tab.total) {
                const uint4 lo = ld_nc(a.shards + src);
                const uint4 hi = PHI ? ld_nc(a.shards + src + kVec) : lo;
                val[i] = window8<PHI>(lo, hi);
                fast[i] = true;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t q = qbeg + (int64_t)i * kGatherThreads + threadIdx.x;
        if (q >= qend) continue;
        if (fast[i]) {
            *reinterpret_cast<uint4 *>(a.full + x0[i]) = val[i];
        } else {
            for (int l = 0; l < kVec; ++l) {
                const int64_t x = x0[i] + l;
                if (x >= d0 && x < d0 + len) a.full[x] = a.shards[x - delta];
            }
        }
    }
}

template <bool ALIGNED>
__global__ void __launch_bounds__(kGatherThreads)
k_allgather(const __grid_constant__ Tab tab, const GatherArgs a) {
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t d0 = e.F + tr.r * e.s;
    const int64_t len = min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    if (len <= 0) return;
    const int64_t q_first = d0 / kVec;
    const int64_t q_last = (d0 + len - 1) / kVec;
    const int64_t qbeg = q_first + tr.t * (int64_t)(kGatherThreads * kGatherVecPerThread);
    if (qbeg > q_last) return;
    const int64_t qend = min(q_last + 1, qbeg + (int64_t)(kGatherThreads * kGatherVecPerThread));
    const int64_t delta = d0 - (tr.r * tab.S + e.o);
    if constexpr (ALIGNED) {
        gather_tile<0>(tab, a, d0, len, delta, qbeg, qend);
    } else {
        const int phi = (int)((((-delta) % kVec) + kVec) % kVec);
        switch (phi) {
            case 0: gather_tile<0>(tab, a, d0, len, delta, qbeg, qend); break;
            case 1: gather_tile<1>(tab, a, d0, len, delta, qbeg, qend); break;
            case 2: gather_tile<2>(tab, a, d0, len, delta, qbeg, qend); break;
            case 3: gather_tile<3>(tab, a, d0, len, delta, qbeg, qend); break;
            case 4: gather_tile<4>(tab, a, d0, len, delta, qbeg, qend); break;
            case 5: gather_tile<5>(tab, a, d0, len, delta, qbeg, qend); break;
            case 6: gather_tile<6>(tab, a, d0, len, delta, qbeg, qend); break;
            default: gather_tile<7>(tab, a, d0, len, delta, qbeg, qend); break;
        }
    }
}

// --------------------------------------------------------------------------
// ReduceScatter (+ accumulate) and the fused ReduceScatter + Adam
// --------------------------------------------------------------------------

enum Mode : int {
    kRS = 0,         // grad_shards = fold * scale
    kRSAcc = 1,      // grad_shards = grad_shards + fold * scale
    kRSAdam = 2,     // Adam(fold * scale)
    kRSAccAdam = 3,  // Adam(grad_acc + fold * scale)
};

struct ReduceArgs {
    const uint16_t *__restrict__ grads;  // [N][stride] bf16
    int64_t stride;
    float scale;
    float *out;             // grad_shards (kRS, kRSAcc)
    const float *acc_in;    // grad_acc (kRSAccAdam)
    float *master;
    float *m;
    float *v;
    uint16_t *shards;
    AdamK k;
};

// Ranks whose 16-byte loads are issued together before they are folded.
constexpr int kRankBatch = 8;

__device__ __forceinline__ void ld8f(const float *p, float f[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void st8f(float *p, const float f[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// Element-wise epilogue of one shard position (edge and pad elements).
template <int MODE>
__device__ __forceinline__ void finish1(const ReduceArgs &a, int64_t x, float g, bool pad) {
    if constexpr (MODE == kRS) {
        a.out[x] = g;
    } else if constexpr (MODE == kRSAcc) {
        a.out[x] = pad ? 0.0f : __fadd_rn(a.out[x], g);
    } else {
        if constexpr (MODE == kRSAccAdam) {
            if (!pad) g = __fadd_rn(a.acc_in[x], g);
        }
        float p = a.master[x], m = a.m[x], v = a.v[x];
        adam1(g, p, m, v, a.k);
        a.master[x] = p;
        a.m[x] = m;
        a.v[x] = v;
        a.shards[x] = f32_to_bf16(p);
    }
}

template <int PHI, int MODE>
__device__ __forceinline__ void reduce_vector(const ReduceArgs &a, int n_ranks, int64_t x0,
                                              int64_t delta) {
    // Rank fold first (8 ranks' 16-byte loads in flight per batch), then the
    // epilogue state: keeping the state out of the fold keeps the kernel
    // within 64 registers, and the other resident warps cover its latency.
    const uint16_t *gp = a.grads + (x0 + delta - PHI);
    // a shifted window needs two 16-byte loads per rank: half the batch
    constexpr int RB = PHI == 0 ? kRankBatch : kRankBatch / 2;
    float acc[8];
    for (int k0 = 0; k0 < n_ranks; k0 += RB) {
        uint4 lo[RB], hi[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if (k0 + u < n_ranks) {
                const uint16_t *rp = gp + (int64_t)(k0 + u) * a.stride;
                lo[u] = ld_nc(rp);
                hi[u] = PHI ? ld_nc(rp + kVec) : lo[u];
            }
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if (k0 + u < n_ranks) {
                float f[8];
                unpack8(window8<PHI>(lo[u], hi[u]), f);
                if (k0 + u == 0) {
#pragma unroll
                    for (int l = 0; l < 8; ++l) acc[l] = f[l];
                } else {
#pragma unroll
                    for (int l = 0; l < 8; ++l) acc[l] = __fadd_rn(acc[l], f[l]);
                }
            }
        }
    }
    float g[8];
#pragma unroll
    for (int l = 0; l < 8; ++l) g[l] = __fmul_rn(acc[l], a.scale);
    if constexpr (MODE == kRS) {
        st8f(a.out + x0, g);
    } else if constexpr (MODE == kRSAcc) {
        float o[8];
        ld8f(a.out + x0, o);
#pragma unroll
        for (int l = 0; l < 8; ++l) g[l] = __fadd_rn(o[l], g[l]);
        st8f(a.out + x0, g);
    } else {
        float p[8], m[8], v[8];
        ld8f(a.master + x0, p);
        ld8f(a.m + x0, m);
        ld8f(a.v + x0, v);
        if constexpr (MODE == kRSAccAdam) {
            float c[8];
            ld8f(a.acc_in + x0, c);
#pragma unroll
            for (int l = 0; l < 8; ++l) g[l] = __fadd_rn(c[l], g[l]);
        }
#pragma unroll
        for (int l = 0; l < 8; ++l) adam1(g[l], p[l], m[l], v[l], a.k);
        st8f(a.master + x0, p);
        st8f(a.m + x0, m);
        st8f(a.v + x0, v);
        uint4 b;
        b.x = pack_bf16x2(p[0], p[1]);
        b.y = pack_bf16x2(p[2], p[3]);
        b.z = pack_bf16x2(p[4], p[5]);
        b.w = pack_bf16x2(p[6], p[7]);
        *reinterpret_cast<uint4 *>(a.shards + x0) = b;
    }
}

// --------------------------------------------------------------------------
// Reduce for tables whose chunks all have phase 0 (every transformer layout
// whose parameter sizes divide by 8N).  One vector per thread; the kernel is
// kept at <= 64 registers so that four 256-thread CTAs (32 warps) share an
// SM: with eight 16-byte gradient loads and six 16-byte state loads in
// flight per thread, that is enough memory-level parallelism to hide HBM
// latency while the Adam arithmetic of other warps runs.
// --------------------------------------------------------------------------

// Element-wise handling of a vector at a chunk edge or in the pad (rare: at
// most two vectors per chunk), kept out of line so that it does not raise
// the register count of the vector path.
template <int MODE>
__device__ __noinline__ void reduce_edges(const ReduceArgs a, int n_ranks, int64_t x0,
                                          int64_t delta, int64_t c0, int64_t c_end,
                                          int64_t valid_end) {
    for (int l = 0; l < kVec; ++l) {
        const int64_t x = x0 + l;
        if (x < c0 || x >= c_end) continue;  // another chunk's element
        const bool pad = x >= valid_end;
        float g = 0.0f;
        if (!pad) {
            const uint16_t *gp = a.grads + (x + delta);
            float s = bf16_to_f32(gp[0]);
            for (int k = 1; k < n_ranks; ++k)
                s = __fadd_rn(s, bf16_to_f32(gp[(int64_t)k * a.stride]));
            g = __fmul_rn(s, a.scale);
        }
        finish1<MODE>(a, x, g, pad);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kReduceThreads, 1024 / kReduceThreads)
k_reduce_aligned(const __grid_constant__ Tab tab, const ReduceArgs a) {
    static_assert(kReduceVecPerThread == 1, "one vector per thread");
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;  // past the chunk's last vector
    if (x0 >= c0 && x0 + kVec <= valid_end)
        reduce_vector<0, MODE>(a, tab.n_ranks, x0, delta);
    else
        reduce_edges<MODE>(a, tab.n_ranks, x0, delta, c0, c_end, valid_end);
}

// The same for tables whose chunks have other phases: each chunk's phase
// (uniform per CTA) selects a window-shifting instantiation.
template <int MODE>
__global__ void __launch_bounds__(kReduceThreads, 1024 / kReduceThreads)
k_reduce_shifted(const __grid_constant__ Tab tab, const ReduceArgs a) {
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;
    if (!(x0 >= c0 && x0 + kVec <= valid_end)) {
        reduce_edges<MODE>(a, tab.n_ranks, x0, delta, c0, c_end, valid_end);
        return;
    }
    const int n = tab.n_ranks;
    switch ((int)(((delta % kVec) + kVec) % kVec)) {
        case 0: reduce_vector<0, MODE>(a, n, x0, delta); break;
        case 1: reduce_vector<1, MODE>(a, n, x0, delta); break;
        case 2: reduce_vector<2, MODE>(a, n, x0, delta); break;
        case 3: reduce_vector<3, MODE>(a, n, x0, delta); break;
        case 4: reduce_vector<4, MODE>(a, n, x0, delta); break;
        case 5: reduce_vector<5, MODE>(a, n, x0, delta); break;
        case 6: reduce_vector<6, MODE>(a, n, x0, delta); break;
        default: reduce_vector<7, MODE>(a, n, x0, delta); break;
    }
}

// --------------------------------------------------------------------------
// Partition (initialisation): shard space <- full fp32, pad 0, m = v = 0
// --------------------------------------------------------------------------

struct PartitionArgs {
    const float *__restrict__ full;
    uint16_t *__restrict__ shards;
    float *__restrict__ master;
    float *__restrict__ m;
    float *__restrict__ v;
};

__global__ void __launch_bounds__(kReduceThreads)
k_partition(const __grid_constant__ Tab tab, const PartitionArgs a) {
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x_beg = (c0 / kVec + tr.t * (int64_t)(kReduceThreads * kReduceVecPerThread)) * kVec;
    const int64_t x_end = min(c_end, x_beg + (int64_t)(kReduceThreads * kReduceVecPerThread) * kVec);
    for (int64_t x = max(x_beg, c0) + threadIdx.x; x < x_end; x += kReduceThreads) {
        const float val = x < valid_end ? a.full[x + delta] : 0.0f;
        a.master[x] = val;
        a.m[x] = 0.0f;
        a.v[x] = 0.0f;
        a.shards[x] = f32_to_bf16(val);
    }
}

// --------------------------------------------------------------------------
// Adam over the flat [N][S] shard buffers
// --------------------------------------------------------------------------

struct AdamArgs {
    float *master;
    float *m;
    float *v;
    const float *grad;
    uint16_t *shards;
    int64_t total;
    AdamK k;
};

constexpr int kAdamThreads = 256;

__global__ void __launch_bounds__(kAdamThreads) k_adam(const AdamArgs a) {
    pdl_enter();
    const int64_t x0 = ((int64_t)blockIdx.x * kAdamThreads + threadIdx.x) * kVec;
    if (x0 >= a.total) return;
    if (x0 + kVec <= a.total) {
        float g[8], p[8], m[8], v[8];
        ld8f(a.grad + x0, g);
        ld8f(a.master + x0, p);
        ld8f(a.m + x0, m);
        ld8f(a.v + x0, v);
#pragma unroll
        for (int l = 0; l < 8; ++l) adam1(g[l], p[l], m[l], v[l], a.k);
        st8f(a.master + x0, p);
        st8f(a.m + x0, m);
        st8f(a.v + x0, v);
        uint4 b;
        b.x = pack_bf16x2(p[0], p[1]);
        b.y = pack_bf16x2(p[2], p[3]);
        b.z = pack_bf16x2(p[4], p[5]);
        b.w = pack_bf16x2(p[6], p[7]);
        *reinterpret_cast<uint4 *>(a.shards + x0) = b;
    } else {
        for (int64_t x = x0; x < a.total; ++x) {
            float p = a.master[x], m = a.m[x], v = a.v[x];
            adam1(a.grad[x], p, m, v, a.k);
            a.master[x] = p;
            a.m[x] = m;
            a.v[x] = v;
            a.shards[x] = f32_to_bf16(p);
        }
    }
}

// --------------------------------------------------------------------------
// Plain data-parallel all-reduce into one fp32 replica, and the scatter of a
// replicated fp32 tensor into the [N][S] shard layout (stage-1 variant)
// --------------------------------------------------------------------------

struct AllreduceArgs {
    const uint16_t *__restrict__ grads;
    int64_t stride;
    float *__restrict__ out;
    int64_t psi;
    float scale;
    int n_ranks;
};

constexpr int kFlatThreads = 256;

// One vector of 8 full-space elements per thread: grads rows start on
// 16-byte boundaries (stride is a multiple of 8), so every vector is aligned.
__global__ void __launch_bounds__(kFlatThreads, 4) k_allreduce(const AllreduceArgs a) {
    pdl_enter();
    const int64_t x0 = ((int64_t)blockIdx.x * kFlatThreads + threadIdx.x) * kVec;
    if (x0 >= a.psi) return;
    if (x0 + kVec <= a.psi) {
        const uint16_t *gp = a.grads + x0;
        float acc[8];
        for (int k0 = 0; k0 < a.n_ranks; k0 += kRankBatch) {
            uint4 w[kRankBatch];
#pragma unroll
            for (int u = 0; u < kRankBatch; ++u)
                if (k0 + u < a.n_ranks) w[u] = ld_nc(gp + (int64_t)(k0 + u) * a.stride);
#pragma unroll
            for (int u = 0; u < kRankBatch; ++u) {
                if (k0 + u < a.n_ranks) {
                    float f[8];
                    unpack8(w[u], f);
                    if (k0 + u == 0) {
#pragma unroll
                        for (int l = 0; l < 8; ++l) acc[l] = f[l];
                    } else {
#pragma unroll
                        for (int l = 0; l < 8; ++l) acc[l] = __fadd_rn(acc[l], f[l]);
                    }
                }
            }
        }
#pragma unroll
        for (int l = 0; l < 8; ++l) acc[l] = __fmul_rn(acc[l], a.scale);
        st8f(a.out + x0, acc);
    } else {
        for (int64_t e = x0; e < a.psi; ++e) {
            float s = bf16_to_f32(a.grads[e]);
            for (int k = 1; k < a.n_ranks; ++k)
                s = __fadd_rn(s, bf16_to_f32(a.grads[(int64_t)k * a.stride + e]));
            a.out[e] = __fmul_rn(s, a.scale);
        }
    }
}

struct ScatterArgs {
    const float *__restrict__ full;
    float *__restrict__ shards;
};

// One vector (8 elements) per thread of each reduce tile: when the whole
// vector is valid, 32-byte stores (and 32-byte loads when the table's chunks
// have phase 0, so the source is aligned too); element by element at chunk
// edges and in the pad.
__global__ void __launch_bounds__(kReduceThreads) k_scatter(const __grid_constant__ Tab tab,
                                                            const ScatterArgs a) {
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;
    if (x0 >= c0 && x0 + kVec <= valid_end) {
        float f[8];
        if (tab.phase0) {
            ld8f(a.full + x0 + delta, f);
        } else {  // source 4-byte aligned only: word loads, the warp's lines come through L1
#pragma unroll
            for (int l = 0; l < 8; ++l) f[l] = a.full[x0 + delta + l];
        }
        st8f(a.shards + x0, f);
        return;
    }
    for (int l = 0; l < kVec; ++l) {
        const int64_t x = x0 + l;
        if (x < c0 || x >= c_end) continue;
        a.shards[x] = x < valid_end ? a.full[x + delta] : 0.0f;
    }
}

// --------------------------------------------------------------------------
// Reshard: one [N][S] buffer to another rank count (checkpoint loading)
// --------------------------------------------------------------------------

// Source-layout facts of the parameters of one destination launch table,
// entry for entry.
struct SrcTab {
    int64_t S;
    int64_t s[kTabMax];
    int64_t o[kTabMax];
};

// One destination vector per thread: a run of 8 consecutive padded indices
// of one parameter, read from one or more source ranks' slices with a
// single division per vector, stored with 16-byte stores.
template <typename T>
__global__ void __launch_bounds__(kReduceThreads)
k_reshard(const __grid_constant__ Tab tab, const __grid_constant__ SrcTab src_tab,
          const T *__restrict__ src, T *__restrict__ dst) {
    static_assert(sizeof(T) == 2 || sizeof(T) == 4, "bf16 or fp32 words");
    pdl_enter();
    const TileRef tr = locate(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t s_src = src_tab.s[tr.p];
    const int64_t o_src = src_tab.o[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;
    if (x0 >= c0 && x0 + kVec <= valid_end) {
        const int64_t i0 = tr.r * e.s + (x0 - c0);   // padded index of the first element
        int64_t r = i0 / s_src;
        int64_t j = i0 - r * s_src;
        T v[8];
#pragma unroll
        for (int l = 0; l < 8; ++l) {
            v[l] = src[r * src_tab.S + o_src + j];
            if (++j == s_src) {
                j = 0;
                ++r;
            }
        }
        if constexpr (sizeof(T) == 2) {
            uint4 w;
            w.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
            w.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
            w.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
            w.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
            *reinterpret_cast<uint4 *>(dst + x0) = w;
        } else {
            *reinterpret_cast<uint4 *>(dst + x0) = make_uint4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<uint4 *>(dst + x0 + 4) = make_uint4(v[4], v[5], v[6], v[7]);
        }
        return;
    }
    for (int l = 0; l < kVec; ++l) {
        const int64_t x = x0 + l;
        if (x < c0 || x >= c_end) continue;
        T val = T(0);
        if (x < valid_end) {
            const int64_t i = tr.r * e.s + (x - c0);
            const int64_t r = i / s_src;
            val = src[r * src_tab.S + o_src + (i - r * s_src)];
        }
        dst[x] = val;
    }
}

// --------------------------------------------------------------------------
// host-side validation helpers
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

z3_status adam_constants(const char *fn, const z3_adam_hp *hp, int64_t step, AdamK *k) {
    if (hp == nullptr) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": hp is NULL");
    if (step < 1) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": step < 1");
    const double vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : vals)
        if (!std::isfinite(x))
            return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": non-finite hyperparameter");
    k->b1 = (float)hp->beta1;
    k->c1 = (float)(1.0 - hp->beta1);
    k->b2 = (float)hp->beta2;
    k->c2 = (float)(1.0 - hp->beta2);
    k->rb1 = (float)(1.0 / (1.0 - std::pow(hp->beta1, (double)step)));
    k->rb2 = (float)(1.0 / (1.0 - std::pow(hp->beta2, (double)step)));
    k->lr = (float)hp->lr;
    k->eps = (float)hp->eps;
    k->lwd = (float)(hp->lr * hp->weight_decay);
    return Z3_OK;
}

z3_status launched(const char *fn) {
    const cudaError_t err = cudaGetLastError();
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

// Launches a kernel with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
void launch(void (*kernel)(KArgs...), int64_t grid, int block, cudaStream_t stream,
            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, kernel, args...);  // errors: cudaGetLastError in launched()
}

// Enqueue helpers (no validation).
z3_status run_allgather(const z3_layout *L, const uint16_t *shards, uint16_t *full,
                        cudaStream_t stream) {
    const GatherArgs a{shards, full};
    for (const Tab &t : L->gather_tabs) {
        if (t.phase0)
            launch(k_allgather<true>, t.tiles, kGatherThreads, stream, t, a);
        else
            launch(k_allgather<false>, t.tiles, kGatherThreads, stream, t, a);
    }
    return launched("z3_allgather");
}

template <int MODE>
z3_status launch_reduce(const Tab &t, const ReduceArgs &a, cudaStream_t stream) {
    if (t.phase0)
        launch(k_reduce_aligned<MODE>, t.tiles, kReduceThreads, stream, t, a);
    else
        launch(k_reduce_shifted<MODE>, t.tiles, kReduceThreads, stream, t, a);
    return Z3_OK;
}

z3_status run_reduce(const z3_layout *L, const ReduceArgs &a, int mode, cudaStream_t stream,
                     const char *fn) {
    for (const Tab &t : L->reduce_tabs) {
        z3_status st;
        switch (mode) {
            case kRS: st = launch_reduce<kRS>(t, a, stream); break;
            case kRSAcc: st = launch_reduce<kRSAcc>(t, a, stream); break;
            case kRSAdam: st = launch_reduce<kRSAdam>(t, a, stream); break;
            default: st = launch_reduce<kRSAccAdam>(t, a, stream); break;
        }
        if (st != Z3_OK) return st;
    }
    return launched(fn);
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
    for (const Tab &t : L->reduce_tabs)
        launch(k_partition, t.tiles, kReduceThreads, (cudaStream_t)stream, t, a);
    return launched(fn);
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
    const int64_t blocks = (T + (int64_t)kAdamThreads * kVec - 1) / ((int64_t)kAdamThreads * kVec);
    if (blocks > 0x7fffffff) return fail(Z3_ERR_OVERFLOW, "z3_adam_shard_step: grid too large");
    Range range("z3/Adam(shard)");
    launch(k_adam, blocks, kAdamThreads, (cudaStream_t)stream, a);
    return launched(fn);
}

namespace {
z3_status prepare_rs_adam(const char *fn, const z3_layout *L, const uint16_t *grads,
                          int64_t grad_stride, float scale, const float *grad_acc, float *master,
                          float *m, float *v, uint16_t *shards, const uint16_t *extra_full,
                          const z3_adam_hp *hp, int64_t step, ReduceArgs *a) {
    if (L == nullptr) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": layout is NULL");
    if (!std::isfinite(scale)) return fail(Z3_ERR_INVALID_ARG, std::string(fn) + ": scale");
    z3_status st = adam_constants(fn, hp, step, &a->k);
    if (st != Z3_OK) return st;
    int64_t gbytes;
    st = check_grads(fn, L, grad_stride, &gbytes);
    if (st != Z3_OK) return st;
    const int64_t T = L->psi_padded;
    const Buf bufs[7] = {{grads, L->psi ? gbytes : 0, "grads"},
                         {master, 4 * T, "master"},
                         {m, 4 * T, "m"},
                         {v, 4 * T, "v"},
                         {shards, 2 * T, "shards"},
                         {grad_acc, grad_acc ? 4 * T : 0, "grad_acc"},
                         {extra_full, extra_full ? 2 * L->psi : 0, "full"}};
    st = check_bufs(fn, bufs, 7);
    if (st != Z3_OK) return st;
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
                                   float *master, float *m, float *v, const z3_adam_hp *hp,
                                   int64_t step, z3_stream stream) {
    const char *fn = "z3_step_layer";
    ReduceArgs a{};
    z3_status st = prepare_rs_adam(fn, L, grads, grad_stride, scale, nullptr, master, m, v,
                                   shards, full, hp, step, &a);
    if (st != Z3_OK) return st;
    if (L->psi_padded == 0) return Z3_OK;
    const cudaStream_t s = (cudaStream_t)stream;
    Range range("z3/step_layer");
    // forward AllGather, backward AllGather, then ReduceScatter + Adam
    {
        Range r1("z3/AllGather(forward)");
        st = run_allgather(L, shards, full, s);
    }
    if (st != Z3_OK) return st;
    {
        Range r2("z3/AllGather(backward)");
        st = run_allgather(L, shards, full, s);
    }
    if (st != Z3_OK) return st;
    Range r3("z3/ReduceScatter+Adam");
    return run_reduce(L, a, kRSAdam, s, fn);
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
    const int64_t blocks = (L->psi + (int64_t)kFlatThreads * kVec - 1) / ((int64_t)kFlatThreads * kVec);
    if (blocks > 0x7fffffff) return fail(Z3_ERR_OVERFLOW, "z3_allreduce: grid too large");
    const AllreduceArgs a{grads, grad_stride, out, L->psi, scale, L->n_ranks};
    Range range("z3/AllReduce");
    launch(k_allreduce, blocks, kFlatThreads, (cudaStream_t)stream, a);
    return launched(fn);
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
    for (const Tab &t : L->reduce_tabs) launch(k_scatter, t.tiles, kReduceThreads, (cudaStream_t)stream, t, a);
    return launched(fn);
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
    // parameters with elements, in the order the destination tables hold them
    std::vector<int32_t> live;
    for (int32_t p = 0; p < Ld->n_params; ++p)
        if (Ld->numel[p] > 0) live.push_back(p);
    size_t next = 0;
    for (const Tab &t : Ld->reduce_tabs) {
        SrcTab stab{};
        stab.S = Ls->S;
        for (int k = 0; k < t.count; ++k, ++next) {
            stab.s[k] = Ls->shard_numel[live[next]];
            stab.o[k] = Ls->shard_off[live[next]];
        }
        if (elem_bytes == 2)
            launch(k_reshard<uint16_t>, t.tiles, kReduceThreads, (cudaStream_t)stream, t, stab,
                   static_cast<const uint16_t *>(src), static_cast<uint16_t *>(dst));
        else
            launch(k_reshard<uint32_t>, t.tiles, kReduceThreads, (cudaStream_t)stream, t, stab,
                   static_cast<const uint32_t *>(src), static_cast<uint32_t *>(dst));
    }
    return launched(fn);
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

extern "C" z3_status z3_model_step(const z3_unit *units, int32_t n_units, uint16_t *const *full,
                                   int32_t n_full, const z3_adam_hp *hp, int64_t step,
                                   z3_stream stream, z3_stream gather_stream) {
    const char *fn = "z3_model_step";
    if (units == nullptr || n_units < 1)
        return fail(Z3_ERR_INVALID_ARG, "z3_model_step: no units");
    if (full == nullptr || n_full < 1 || n_full > 8)
        return fail(Z3_ERR_INVALID_ARG, "z3_model_step: n_full must be 1..8");
    if (n_full >= 2 && (gather_stream == nullptr || gather_stream == stream))
        return fail(Z3_ERR_INVALID_ARG,
                    "z3_model_step: prefetch needs a gather stream distinct from stream");
    std::vector<ReduceArgs> args((size_t)n_units);
    for (int32_t i = 0; i < n_units; ++i) {
        const z3_unit &u = units[i];
        z3_status st = prepare_rs_adam(fn, u.layout, u.grads, u.grad_stride, u.scale, nullptr,
                                       u.master, u.m, u.v, u.shards, full[0], hp, step, &args[i]);
        if (st != Z3_OK) return st;
        const int64_t T = u.layout->psi_padded;
        int64_t gbytes = 0;
        st = check_grads(fn, u.layout, u.grad_stride, &gbytes);
        if (st != Z3_OK) return st;
        for (int32_t k = 1; k < n_full; ++k) {
            const Buf bufs[7] = {{full[k], 2 * u.layout->psi, "full[k]"},
                                 {full[0], 2 * u.layout->psi, "full[0]"},
                                 {u.shards, 2 * T, "shards"},
                                 {u.master, 4 * T, "master"},
                                 {u.m, 4 * T, "m"},
                                 {u.v, 4 * T, "v"},
                                 {u.grads, u.layout->psi ? gbytes : 0, "grads"}};
            st = check_bufs(fn, bufs, 7);
            if (st != Z3_OK) return st;
            for (int32_t j = 1; j < k; ++j) {
                const Buf pair[2] = {{full[k], 2 * u.layout->psi, "full[k]"},
                                     {full[j], 2 * u.layout->psi, "full[j]"}};
                st = check_bufs(fn, pair, 2);
                if (st != Z3_OK) return st;
            }
        }
    }
    const cudaStream_t s = (cudaStream_t)stream;
    Range range("z3/model_step");
    z3_status st = Z3_OK;
    if (n_full == 1) {
        for (int32_t i = 0; i < n_units && st == Z3_OK; ++i) {
            Range r("z3/AllGather(forward)");
            if (units[i].layout->psi) st = run_allgather(units[i].layout, units[i].shards, full[0], s);
        }
        for (int32_t i = n_units - 1; i >= 0 && st == Z3_OK; --i) {
            const z3_layout *L = units[i].layout;
            if (L->psi_padded == 0) continue;
            {
                Range r("z3/AllGather(backward)");
                st = run_allgather(L, units[i].shards, full[0], s);
            }
            if (st != Z3_OK) break;
            Range r("z3/ReduceScatter+Adam");
            st = run_reduce(L, args[i], kRSAdam, s, fn);
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
    const int nb = n_full;
    Events E;
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
        if (units[i].layout->psi) st = run_allgather(units[i].layout, units[i].shards, full[i % nb], g);
    }
    std::vector<bool> buffer_used((size_t)nb, false);
    auto gather = [&](int32_t i) -> z3_status {
        const int b = i % nb;
        if (buffer_used[b]) {   // the unit that last used this buffer has been updated
            cudaError_t e = cudaStreamWaitEvent(g, freed(b), 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        Range r("z3/AllGather(backward)");
        z3_status gs = units[i].layout->psi ? run_allgather(units[i].layout, units[i].shards, full[b], g)
                                            : Z3_OK;
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
        const z3_layout *L = units[i].layout;
        if (L->psi_padded > 0) {
            Range r("z3/ReduceScatter+Adam");
            st = run_reduce(L, args[i], kRSAdam, s, fn);
            if (st != Z3_OK) break;
        }
        if ((err = cudaEventRecord(freed(i % nb), s)) != cudaSuccess) return cuda_fail(err);
        buffer_used[i % nb] = true;
    }
    if (st != Z3_OK) return st;
    if ((err = cudaEventRecord(E.ev[1], g)) != cudaSuccess) return cuda_fail(err);
    if ((err = cudaStreamWaitEvent(s, E.ev[1], 0)) != cudaSuccess) return cuda_fail(err);
    return Z3_OK;
}
