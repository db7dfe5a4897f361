// z3_kernels.cu -- sm_103a kernels of the ZeRO-3 sharded layer step and their
// launchers (z3_launch.h); the C-ABI entry points that validate arguments and
// call the launchers are in z3_api.cpp.
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

#include <cstdint>

#include "z3_launch.h"

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

// The tiles of one launch number at most 2^31 - 1 (the layout starts a new
// launch table before that), and every entry has at least one tile per
// chunk, so the tile arithmetic fits unsigned 32 bits.  DIV32 divides by the
// tiles per chunk in 32 bits instead of an emulated 64-bit division: the
// copy kernels take it (their few instructions per element make the
// division a large share); the reduce kernels keep the 64-bit form, with
// which their fused modes fit 64 registers without spilling.
template <bool DIV32>
__device__ __forceinline__ TileRef locate(const Tab &tab, uint32_t g) {
    int lo = 0, hi = tab.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((uint32_t)tab.e[mid].tile0 <= g) lo = mid; else hi = mid - 1;
    }
    if constexpr (DIV32) {
        const uint32_t local = g - (uint32_t)tab.e[lo].tile0;
        const uint32_t tpc = (uint32_t)tab.e[lo].tpc;
        const uint32_t r = local / tpc;
        return TileRef{lo, (int64_t)r, (int64_t)(local - r * tpc)};
    } else {
        const int64_t local = (int64_t)g - tab.e[lo].tile0;
        const int64_t tpc = tab.e[lo].tpc;
        const int64_t r = local / tpc;
        return TileRef{lo, r, local - r * tpc};
    }
}

// Programmatic dependent launch.  Every kernel is launched so that it may
// start while the previous kernel of the stream (its primary) still runs.
// A thread first waits for the primary to complete -- memory included -- and
// only then lets the next kernel launch.  Because every kernel waits before
// it releases its dependent, a kernel that has started knows that everything
// enqueued before its primary has completed: only the primary may still be
// running.  So:
//   - a plain kernel waits before its first global memory access, and the
//     ordering between calls is exactly stream order;
//   - an EARLY variant (used only where the library itself enqueued the
//     primary, inside one call) may, before it waits, read buffers that the
//     primary does not write; it waits before its first store.  Its first
//     loads overlap the primary's tail.
// Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------------
// AllGather: full[F_p + i] = shards[i / s_p][o_p + i mod s_p]
// --------------------------------------------------------------------------

struct GatherArgs {
    const uint16_t *__restrict__ shards;
    uint16_t *__restrict__ full;
};

template <int PHI, bool EARLY>
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
    if constexpr (EARLY) pdl_enter();  // the shard loads above may precede it; stores may not
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

// EARLY: the primary writes neither the shards nor anything else read here
// (it may write `full`: the stores wait).
template <bool ALIGNED, bool EARLY>
__global__ void __launch_bounds__(kGatherThreads)
k_allgather(const __grid_constant__ Tab tab, const GatherArgs a) {
    if constexpr (!EARLY) pdl_enter();
    const TileRef tr = locate<true>(tab, blockIdx.x);
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
        gather_tile<0, EARLY>(tab, a, d0, len, delta, qbeg, qend);
    } else {
        const int phi = (int)((((-delta) % kVec) + kVec) % kVec);
        switch (phi) {
            case 0: gather_tile<0, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 1: gather_tile<1, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 2: gather_tile<2, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 3: gather_tile<3, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 4: gather_tile<4, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 5: gather_tile<5, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            case 6: gather_tile<6, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
            default: gather_tile<7, EARLY>(tab, a, d0, len, delta, qbeg, qend); break;
        }
    }
}

// --------------------------------------------------------------------------
// ReduceScatter (+ accumulate) and the fused ReduceScatter + Adam
// --------------------------------------------------------------------------

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
        if constexpr (MODE == kRSAdamOut) a.out[x] = g;
        float p = a.master[x], m = a.m[x], v = a.v[x];
        adam1(g, p, m, v, a.k);
        a.master[x] = p;
        a.m[x] = m;
        a.v[x] = v;
        a.shards[x] = f32_to_bf16(p);
    }
}

template <int PHI, int MODE, bool EARLY>
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
        if constexpr (MODE == kRSAdamOut) st8f(a.out + x0, g);  // never EARLY: waited at entry
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
        if constexpr (EARLY) pdl_enter();  // every load above may precede it; stores may not
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
// kept at <= 64 registers so that eight 128-thread CTAs (32 warps) share an
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

// EARLY (fused modes only): the primary writes none of the buffers read here
// (gradients, running sums, master, m, v); it may read or write others, and
// every store waits for it.
template <int MODE, bool EARLY>
__global__ void __launch_bounds__(kReduceThreads, 1024 / kReduceThreads)
k_reduce_aligned(const __grid_constant__ Tab tab, const ReduceArgs a) {
    static_assert(kReduceVecPerThread == 1, "one vector per thread");
    static_assert(!EARLY || MODE == kRSAdam || MODE == kRSAccAdam, "EARLY: fused modes only");
    if constexpr (!EARLY) pdl_enter();
    const TileRef tr = locate<false>(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;  // past the chunk's last vector
    if (x0 >= c0 && x0 + kVec <= valid_end) {
        reduce_vector<0, MODE, EARLY>(a, tab.n_ranks, x0, delta);
    } else {
        if constexpr (EARLY) pdl_enter();
        reduce_edges<MODE>(a, tab.n_ranks, x0, delta, c0, c_end, valid_end);
    }
}

// The same for tables whose chunks have other phases: each chunk's phase
// (uniform per CTA) selects a window-shifting instantiation.
template <int MODE, bool EARLY>
__global__ void __launch_bounds__(kReduceThreads, 1024 / kReduceThreads)
k_reduce_shifted(const __grid_constant__ Tab tab, const ReduceArgs a) {
    static_assert(!EARLY || MODE == kRSAdam || MODE == kRSAccAdam, "EARLY: fused modes only");
    if constexpr (!EARLY) pdl_enter();
    const TileRef tr = locate<false>(tab, blockIdx.x);
    const TabEntry &e = tab.e[tr.p];
    const int64_t c0 = tr.r * tab.S + e.o;
    const int64_t c_end = c0 + e.s;
    const int64_t valid_end = c0 + min(e.s, max((int64_t)0, e.n - tr.r * e.s));
    const int64_t delta = e.F + tr.r * e.s - c0;
    const int64_t x0 = (c0 / kVec + tr.t * (int64_t)kReduceThreads + threadIdx.x) * kVec;
    if (x0 >= c_end) return;
    if (!(x0 >= c0 && x0 + kVec <= valid_end)) {
        if constexpr (EARLY) pdl_enter();
        reduce_edges<MODE>(a, tab.n_ranks, x0, delta, c0, c_end, valid_end);
        return;
    }
    const int n = tab.n_ranks;
    switch ((int)(((delta % kVec) + kVec) % kVec)) {
        case 0: reduce_vector<0, MODE, EARLY>(a, n, x0, delta); break;
        case 1: reduce_vector<1, MODE, EARLY>(a, n, x0, delta); break;
        case 2: reduce_vector<2, MODE, EARLY>(a, n, x0, delta); break;
        case 3: reduce_vector<3, MODE, EARLY>(a, n, x0, delta); break;
        case 4: reduce_vector<4, MODE, EARLY>(a, n, x0, delta); break;
        case 5: reduce_vector<5, MODE, EARLY>(a, n, x0, delta); break;
        case 6: reduce_vector<6, MODE, EARLY>(a, n, x0, delta); break;
        default: reduce_vector<7, MODE, EARLY>(a, n, x0, delta); break;
    }
}

// --------------------------------------------------------------------------
// Partition (initialisation): shard space <- full fp32, pad 0, m = v = 0
// --------------------------------------------------------------------------

// One vector (8 elements) per thread of each reduce tile, like k_scatter:
// when the whole vector is valid, 16-byte stores of master, m, v and the
// bf16 shard (and 16-byte loads of the full tensor when the table's chunks
// have phase 0); element by element at chunk edges and in the pad.
__global__ void __launch_bounds__(kReduceThreads)
k_partition(const __grid_constant__ Tab tab, const PartitionArgs a) {
    pdl_enter();
    const TileRef tr = locate<true>(tab, blockIdx.x);
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
        } else {  // source 4-byte aligned only
#pragma unroll
            for (int l = 0; l < 8; ++l) f[l] = a.full[x0 + delta + l];
        }
        const float zero[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st8f(a.master + x0, f);
        st8f(a.m + x0, zero);
        st8f(a.v + x0, zero);
        uint4 b;
        b.x = pack_bf16x2(f[0], f[1]);
        b.y = pack_bf16x2(f[2], f[3]);
        b.z = pack_bf16x2(f[4], f[5]);
        b.w = pack_bf16x2(f[6], f[7]);
        *reinterpret_cast<uint4 *>(a.shards + x0) = b;
        return;
    }
    for (int l = 0; l < kVec; ++l) {
        const int64_t x = x0 + l;
        if (x < c0 || x >= c_end) continue;  // another chunk's element
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

// One vector (8 elements) per thread of each reduce tile: when the whole
// vector is valid, 32-byte stores (and 32-byte loads when the table's chunks
// have phase 0, so the source is aligned too); element by element at chunk
// edges and in the pad.
__global__ void __launch_bounds__(kReduceThreads) k_scatter(const __grid_constant__ Tab tab,
                                                            const ScatterArgs a) {
    pdl_enter();
    const TileRef tr = locate<true>(tab, blockIdx.x);
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
    const TileRef tr = locate<true>(tab, blockIdx.x);
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
        int64_t r, j;
        if (i0 <= 0xffffffffll && s_src <= 0xffffffffll) {  // 32-bit division when it fits
            const uint32_t q = (uint32_t)i0 / (uint32_t)s_src;
            r = q;
            j = i0 - (int64_t)q * s_src;
        } else {
            r = i0 / s_src;
            j = i0 - r * s_src;
        }
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
    (void)cudaLaunchKernelEx(&cfg, kernel, args...);  // errors: cudaGetLastError below
}

template <int MODE, bool EARLY>
void launch_reduce_tab(const Tab &t, const ReduceArgs &a, cudaStream_t stream) {
    if (t.phase0)
        launch(k_reduce_aligned<MODE, EARLY>, t.tiles, kReduceThreads, stream, t, a);
    else
        launch(k_reduce_shifted<MODE, EARLY>, t.tiles, kReduceThreads, stream, t, a);
}

}  // namespace

// --------------------------------------------------------------------------
// launchers: enqueue only (arguments were validated by the caller)
// --------------------------------------------------------------------------

cudaError_t launch_partition(const z3_layout *L, const PartitionArgs &a, cudaStream_t stream) {
    for (const Tab &t : L->reduce_tabs) launch(k_partition, t.tiles, kReduceThreads, stream, t, a);
    return cudaGetLastError();
}

cudaError_t launch_allgather(const z3_layout *L, const uint16_t *shards, uint16_t *full,
                             cudaStream_t stream, bool early) {
    const GatherArgs a{shards, full};
    bool first = true;
    for (const Tab &t : L->gather_tabs) {
        // a later table's primary is this call's own previous launch, which
        // writes only `full`
        const bool e = early || !first;
        first = false;
        if (t.phase0) {
            if (e) launch(k_allgather<true, true>, t.tiles, kGatherThreads, stream, t, a);
            else launch(k_allgather<true, false>, t.tiles, kGatherThreads, stream, t, a);
        } else {
            if (e) launch(k_allgather<false, true>, t.tiles, kGatherThreads, stream, t, a);
            else launch(k_allgather<false, false>, t.tiles, kGatherThreads, stream, t, a);
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_reduce(const z3_layout *L, const ReduceArgs &a, Mode mode,
                          cudaStream_t stream, bool early) {
    // Later tables of one call update disjoint shard ranges, so their
    // primary (this call's previous table) writes nothing they read; an
    // unfused mode reads its own output buffer, so it never runs early, and
    // the fused mode that also stores the reduced gradient stays plain (its
    // gradient store comes before the Adam arithmetic, ahead of any wait).
    bool first = true;
    for (const Tab &t : L->reduce_tabs) {
        const bool e = early || !first;
        first = false;
        switch (mode) {
            case kRS: launch_reduce_tab<kRS, false>(t, a, stream); break;
            case kRSAcc: launch_reduce_tab<kRSAcc, false>(t, a, stream); break;
            case kRSAdam:
                if (e) launch_reduce_tab<kRSAdam, true>(t, a, stream);
                else launch_reduce_tab<kRSAdam, false>(t, a, stream);
                break;
            case kRSAccAdam:
                if (e) launch_reduce_tab<kRSAccAdam, true>(t, a, stream);
                else launch_reduce_tab<kRSAccAdam, false>(t, a, stream);
                break;
            default: launch_reduce_tab<kRSAdamOut, false>(t, a, stream); break;
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_adam(const AdamArgs &a, cudaStream_t stream) {
    launch(k_adam, flat_blocks(a.total, kAdamThreads), kAdamThreads, stream, a);
    return cudaGetLastError();
}

cudaError_t launch_allreduce(const AllreduceArgs &a, cudaStream_t stream) {
    launch(k_allreduce, flat_blocks(a.psi, kFlatThreads), kFlatThreads, stream, a);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const z3_layout *L, const ScatterArgs &a, cudaStream_t stream) {
    for (const Tab &t : L->reduce_tabs) launch(k_scatter, t.tiles, kReduceThreads, stream, t, a);
    return cudaGetLastError();
}

cudaError_t launch_reshard(const z3_layout *Ls, const z3_layout *Ld, int elem_bytes,
                           const void *src, void *dst, cudaStream_t stream) {
    // the tables hold the parameters with elements, in parameter order
    int32_t p = 0;
    for (const Tab &t : Ld->reduce_tabs) {
        SrcTab stab{};
        stab.S = Ls->S;
        for (int k = 0; k < t.count; ++k, ++p) {
            while (Ld->numel[p] == 0) ++p;
            stab.s[k] = Ls->shard_numel[p];
            stab.o[k] = Ls->shard_off[p];
        }
        if (elem_bytes == 2)
            launch(k_reshard<uint16_t>, t.tiles, kReduceThreads, stream, t, stab,
                   static_cast<const uint16_t *>(src), static_cast<uint16_t *>(dst));
        else
            launch(k_reshard<uint32_t>, t.tiles, kReduceThreads, stream, t, stab,
                   static_cast<const uint32_t *>(src), static_cast<uint32_t *>(dst));
    }
    return cudaGetLastError();
}

}  // namespace z3
