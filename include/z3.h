/*
 * z3.h -- C ABI of the ZeRO-3 sharded model-state hot path on one GPU.
 *
 * The N logical data-parallel ranks of ZeRO stage 3 are held as shard
 * regions of one GPU's memory, so the collectives are on-device data
 * movement.  The operations follow the pages that define the method:
 *
 *   [ZD] "The ZeRO-3 Diagram Most People Remember Is Wrong" (duoan.github.io):
 *        s.2 "The Actual Parameter Partition" (flatten, pad, contiguous slice
 *        per rank) and s.3 "The Collectives You Should Expect" (AllGather
 *        before forward and again before backward, ReduceScatter of the
 *        gradients, the optimizer updates the local shard).
 *   [S3] "ZeRO Stage 3: Parameter Partitioning" (mbrenndoerfer.com):
 *        eq. M_Stage3 (16 bytes of model state per owned element) and the
 *        communication list (2*Psi + 2*Psi + 2*Psi = 6*Psi bytes per step).
 *   [ZS] "ZeRO Stages: Sharding Optimizer State, Gradients, and Parameters"
 *        (mercemay.com): "Stage 2 also partitions gradients" (the reduce-
 *        scatter sums across ranks and leaves each rank its slice; reduce per
 *        micro-batch and accumulate the reduced slices).
 *
 * Notation: a layer is an ordered list of parameters; parameter p has n_p
 * elements; N = n_ranks; s_p = ceil(n_p / N); rank r owns padded positions
 * [r*s_p, (r+1)*s_p) of p (positions >= n_p are pad); o_p = sum_{q<p} s_q;
 * F_p = sum_{q<p} n_q; S = sum_p s_p; Psi = sum_p n_p.
 *
 * Buffers (all device memory, all owned by the caller; the library never
 * allocates or frees device memory -- its only device memory of its own is
 * the static array described at z3_step_layer_noalloc):
 *   shards   bf16 [N][S]   rank r's shard at r*S; p's slice at r*S + o_p
 *   master, m, v, grad_shards   fp32 [N][S], same indexing
 *   full     bf16 [Psi]    one gathered copy of the layer, parameters
 *                          concatenated unpadded: p at F_p
 *   grads    bf16 [N][grad_stride]   rank k's full gradient at k*grad_stride
 * bf16 values travel as uint16_t bit patterns.  Pad positions of every
 * [N][S] buffer are zero after z3_partition and stay zero under every other
 * call.
 *
 * Conventions:
 *   - Every call returns a z3_status; no call aborts, prints or traps, and
 *     no device code asserts.  z3_last_error() gives the message of the
 *     last failure on the calling thread.  A failed host allocation inside
 *     the library (layouts, launch tables, the model step's bookkeeping,
 *     pipelines) returns Z3_ERR_HOST_MEMORY.
 *   - Device calls validate every argument on the host, then enqueue on the
 *     caller's stream and return; a launch failure returns Z3_ERR_CUDA.
 *     Errors during execution surface at the caller's next synchronisation.
 *   - Device buffers must start on a 16-byte boundary (Z3_ERR_ALIGNMENT);
 *     grad_stride must be a multiple of 8 elements (Z3_ERR_ALIGNMENT) and
 *     >= Psi (Z3_ERR_INVALID_ARG).  Interior offsets (o_p, F_p, S) may be
 *     anything.
 *   - Output buffers must not overlap any other buffer of the same call
 *     (Z3_ERR_INVALID_ARG), except the in-place state of the Adam calls.
 *   - Calls other than z3_step_layer_noalloc (see there) make no synchronous
 *     CUDA calls and allocate no device memory, so a caller may capture them
 *     in a CUDA graph.  The only CUDA objects the library creates are events:
 *     per call in z3_model_step with prefetch (destroyed before it returns),
 *     and once per pipeline in z3_host_step_create.
 *   - A layout handle is immutable after creation and may be shared between
 *     threads.
 */
#ifndef Z3_H
#define Z3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum z3_status {
    Z3_OK = 0,
    Z3_ERR_INVALID_ARG = 1, /* null/negative/inconsistent argument */
    Z3_ERR_ALIGNMENT = 2,   /* buffer not 16-byte aligned, bad grad_stride */
    Z3_ERR_OVERFLOW = 3,    /* a size does not fit int64 / the launch grid */
    Z3_ERR_CUDA = 4,        /* the CUDA runtime reported an error */
    Z3_ERR_HOST_MEMORY = 5  /* a host allocation of the library failed */
} z3_status;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *z3_stream;

/* Opaque, library-owned host object describing one layer's layout. */
typedef struct z3_layout z3_layout;

/* Adam hyperparameters as real numbers.  Every constant of the update is
 * rounded once to binary32 on the host: beta1, 1-beta1, beta2, 1-beta2,
 * 1/(1-beta1^t), 1/(1-beta2^t), lr, eps and lr*weight_decay.  Accepted:
 * finite values with 0 <= beta1, beta2 < 1, eps > 0, lr >= 0 and
 * weight_decay >= 0, whose constants are finite in binary32 and whose eps
 * stays above 0 there (eps = 0 would turn a pad position's 0/0 into NaN);
 * anything else is Z3_ERR_INVALID_ARG. */
typedef struct z3_adam_hp {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay; /* decoupled: p <- p - (lr*wd)*p before the step */
} z3_adam_hp;

/* Byte counts of one layer ([S3] communication list; per-kernel HBM bytes
 * are the algorithmic bytes per unpadded element times Psi). */
typedef struct z3_traffic {
    int64_t psi;                 /* unpadded elements of the layer           */
    int64_t ag_payload_bytes;    /* 2*Psi: one gathered bf16 copy            */
    int64_t rs_payload_bytes;    /* 2*Psi: one bf16 gradient reduced         */
    int64_t step_volume_bytes;   /* 6*Psi: AG fwd + AG bwd + RS ([S3])       */
    int64_t dp_allreduce_bytes;  /* 2*Psi: plain data-parallel all-reduce    */
    int64_t hbm_allgather;       /* 4*Psi       (read 2, write 2)            */
    int64_t hbm_reduce_scatter;  /* (2N+4)*Psi  (read 2N, write 4)           */
    int64_t hbm_reduce_scatter_accumulate; /* (2N+8)*Psi                     */
    int64_t hbm_adam;            /* 30*Psi (read g,p,m,v 16; write p,m,v,b 14)*/
    int64_t hbm_reduce_scatter_adam;       /* (2N+26)*Psi                    */
    int64_t hbm_step_layer;      /* (2N+34)*Psi: AG + AG + fused RS/Adam     */
    int64_t state_bytes_per_rank;/* 16*S ([S3] eq. M_Stage3, 2-byte grads)   */
    int64_t state_bytes_per_rank_fp32_grad; /* 18*S ([ZS], 4-byte grads)     */
} z3_traffic;

/* ---- layout ([ZD] s.2; [ZS] "What stage 1 partitions") ---------------- */

/* Builds the layout of a layer of n_params parameters with the given
 * element counts over n_ranks logical ranks.  numel[p] >= 0 (0 is allowed:
 * s_p = 0).  Errors: n_params < 1, n_ranks < 1, numel NULL or negative,
 * out NULL (INVALID_ARG); N*S or Psi beyond int64 (OVERFLOW).  On success
 * *out owns host memory released by z3_layout_destroy. */
z3_status z3_layout_create(const int64_t *numel, int32_t n_params,
                           int32_t n_ranks, z3_layout **out);

/* Releases a layout (NULL is a no-op). */
void z3_layout_destroy(z3_layout *layout);

/* Scalar facts of a layout; any output pointer may be NULL. */
z3_status z3_layout_info(const z3_layout *layout, int32_t *n_params,
                         int32_t *n_ranks, int64_t *S, int64_t *psi,
                         int64_t *psi_padded);

/* Per-parameter arrays [n_params] (caller-owned host memory); any may be
 * NULL. */
z3_status z3_layout_params(const z3_layout *layout, int64_t *numel,
                           int64_t *shard_numel, int64_t *shard_off,
                           int64_t *full_off);

/* Byte accounting of the layout ([S3] eq. M_Stage3 and communication list). */
z3_status z3_stats(const z3_layout *layout, z3_traffic *out);

/* ---- device operations ------------------------------------------------ */

/* Initial partition ([ZD] s.2 steps 1-4; a broadcast-like step that runs
 * once at initialisation, [ZD] s.3).  full: fp32 [Psi] (read).  Writes
 * master[r][o_p+j] = full[F_p + r*s_p + j] (0 in the pad), m = v = 0 and
 * shards = bf16 round-to-nearest-even of master.  All five buffers must be
 * distinct and non-overlapping. */
z3_status z3_partition(const z3_layout *layout, const float *full,
                       uint16_t *shards, float *master, float *m, float *v,
                       z3_stream stream);

/* AllGather ([ZD] s.3; [S3] step 2): full[F_p + i] =
 * shards[i / s_p][o_p + i mod s_p] for 0 <= i < n_p.  Bit copy; the pad is
 * dropped.  shards is read; full [Psi] is written. */
z3_status z3_allgather(const z3_layout *layout, const uint16_t *shards,
                       uint16_t *full, z3_stream stream);

/* ReduceScatter ([ZD] s.3; [ZS] "Stage 2 also partitions gradients"):
 * for every owned position with padded index i = r*s_p + j < n_p,
 *   g = fp32(grads[0][F_p+i]); g = g + fp32(grads[k][F_p+i]) for k = 1..N-1
 *   (binary32, ascending rank order); g = g * scale;
 *   grad_shards[r][o_p+j] = accumulate ? grad_shards[r][o_p+j] + g : g.
 * Pad positions are written 0.  scale = 1/N gives the data-parallel mean.
 * grads is read; grad_shards is written (and read when accumulate != 0). */
z3_status z3_reduce_scatter(const z3_layout *layout, const uint16_t *grads,
                            int64_t grad_stride, float *grad_shards,
                            float scale, int32_t accumulate, z3_stream stream);

/* Local-shard Adam ([ZD] s.3 "optimizer updates local shard"; Kingma & Ba,
 * Algorithm 1) on every position of the [N][S] buffers, t = step >= 1:
 *   m' = b1*m + c1*g;  v' = b2*v + c2*(g*g);  mh = m'*rb1;  vh = v'*rb2;
 *   u = mh / (sqrt(vh) + eps);  p' = (p - lwd*p) - lr*u;  shards = bf16(p')
 * (rb1 = 1/(1-beta1^t), rb2 = 1/(1-beta2^t): the bias corrections) in
 * binary32 with IEEE-rounded division and square root, no fused
 * multiply-add.  master, m, v are updated in place; grad_shards is read;
 * shards is written.  Errors: hp NULL or non-finite, step < 1. */
z3_status z3_adam_shard_step(const z3_layout *layout, float *master, float *m,
                             float *v, const float *grad_shards,
                             uint16_t *shards, const z3_adam_hp *hp,
                             int64_t step, z3_stream stream);

/* ReduceScatter fused with Adam: the reduced gradient of each owned
 * position (as z3_reduce_scatter, accumulate into grad_acc when grad_acc is
 * not NULL; pad positions get gradient 0) feeds the Adam update of that
 * position in registers, so no fp32 gradient is written.  grad_acc (may be
 * NULL) is read only.  Equivalent to z3_reduce_scatter into a copy of
 * grad_acc followed by z3_adam_shard_step. */
z3_status z3_reduce_scatter_adam(const z3_layout *layout,
                                 const uint16_t *grads, int64_t grad_stride,
                                 float scale, const float *grad_acc,
                                 float *master, float *m, float *v,
                                 uint16_t *shards, const z3_adam_hp *hp,
                                 int64_t step, z3_stream stream);

/* One layer step in the order of [ZD] s.3: forward AllGather into full,
 * backward AllGather into full again, then the fused ReduceScatter + Adam
 * that rewrites the shards.  Three kernel launches on the stream.
 * grad_shards_or_NULL: NULL keeps the reduced gradient in registers (no
 * fp32 gradient reaches memory).  Non-NULL (fp32 [N][S], written) also
 * stores each rank's reduced gradient slice there, exactly as
 * z3_reduce_scatter would write it (pad 0): the one-slice gradient buffer
 * of [ZS] "Stage 2 also partitions gradients", for a caller that needs the
 * gradient itself.  Same fused pass, 4 more bytes written per element. */
z3_status z3_step_layer(const z3_layout *layout, uint16_t *shards,
                        uint16_t *full, const uint16_t *grads,
                        int64_t grad_stride, float scale, float *master,
                        float *m, float *v, float *grad_shards_or_NULL,
                        const z3_adam_hp *hp, int64_t step, z3_stream stream);

/* ---- a whole model step --------------------------------------------- */

/* One unit of a model (a layer, a bucket of layers, an embedding): its
 * layout, its [N][S] state and its gradients (as for z3_step_layer).
 *
 * resident: NULL for a unit whose gathered parameters are released after
 * each use ([ZD] s.6: parameters released after use; [S3] "ZeRO Stage 3":
 * the gathered parameters are discarded once the layer has run), so every
 * use gathers them again into a transient buffer.  Non-NULL (bf16 [Psi] of
 * this unit, caller-owned) for a persistent unit, the small parameters that
 * a persistence threshold ([ZD] s.8) keeps gathered between uses: the step
 * does not gather it forward or backward, and gathers it into `resident`
 * once, right after its update, so the copy always holds the current
 * parameters.  The caller fills `resident` once after z3_partition (one
 * z3_allgather).
 *
 * hp: NULL to use the step's hyperparameters, or this unit's own (a
 * parameter group, e.g. no weight decay on norm gains). */
typedef struct z3_unit {
    const z3_layout *layout;
    uint16_t *shards;
    float *master;
    float *m;
    float *v;
    const uint16_t *grads;
    int64_t grad_stride;
    float scale;
    uint16_t *resident;
    const z3_adam_hp *hp;
} z3_unit;

/* One training step of a model of n_units units, in the schedule of [ZD]
 * s.3 and [S3] (backward in reverse layer order): the forward AllGather of
 * every unit in order, then for each unit in reverse order its backward
 * AllGather followed by its fused ReduceScatter + Adam.  Every gather lands
 * in a transient buffer that must hold the largest non-resident unit (bf16
 * [max Psi]).  A resident unit instead skips both gathers and is gathered
 * into its own buffer after its update (see z3_unit).
 *   n_full = 1: everything runs on `stream`, through full[0].
 *   n_full = D + 1 (2..8) with gather_stream != NULL: the gathers run on
 *     gather_stream up to D units ahead of the updates ([S3]: the gather of
 *     the next layer proceeds while the current one computes; [ZS]: the
 *     prefetch depth trades memory -- one more buffer per unit of depth --
 *     against latency).  Unit i uses full[i mod n_full]; events order every
 *     buffer reuse.  The call returns with `stream` ordered after all work.
 * Results do not depend on n_full.  Every buffer a unit writes (shards,
 * master, m, v, resident) must be disjoint from every buffer of every other
 * unit and from the transient buffers; units may share read-only gradients.
 * Errors: as z3_step_layer for each unit, n_units < 1, n_full not in 1..8,
 * gather_stream NULL or equal to stream when n_full >= 2, overlapping
 * buffers (INVALID_ARG, naming the units). */
z3_status z3_model_step(const z3_unit *units, int32_t n_units, uint16_t *const *full,
                        int32_t n_full, const z3_adam_hp *hp, int64_t step,
                        z3_stream stream, z3_stream gather_stream);

/* ---- the layer step fed from host memory ------------------------------- */

/* A pipeline that runs z3_step_layer on gradients held in host memory and
 * returns the updated bf16 parameters to host memory: each call uploads the
 * N ranks' gradients into one of two device staging buffers, runs the layer
 * step ([ZD] s.3: AllGather, AllGather, ReduceScatter + the shard update)
 * from that buffer, and downloads the updated shards.  Consecutive calls
 * alternate the staging buffers, so the upload of call i+1 (on
 * upload_stream) overlaps the compute of call i (on the call's stream) and
 * the download of call i (on download_stream).  CUDA events order every
 * reuse: an upload into a staging buffer waits for the step that last read
 * it; a step waits for its upload and for the previous call's download (the
 * step rewrites the shards that download reads); a download waits for its
 * step.
 *
 * Ownership: the caller owns the two staging buffers (device, bf16
 * [N][grad_stride] each, 16-byte aligned, not overlapping) and both streams;
 * the pipeline owns only its CUDA events (created here, destroyed by
 * z3_host_step_destroy).  A pipeline belongs to one layout and one calling
 * thread at a time.  Its calls order work through events that persist from
 * one call to the next, so they are meant for eager use, not for capture in
 * a CUDA graph.  Errors: NULL layout, staging buffer or stream, equal
 * streams, misaligned or overlapping staging buffers, grad_stride as for
 * z3_reduce_scatter (INVALID_ARG / ALIGNMENT); event creation failing
 * (CUDA). */
typedef struct z3_host_step z3_host_step;

z3_status z3_host_step_create(const z3_layout *layout, uint16_t *staging0,
                              uint16_t *staging1, int64_t grad_stride,
                              z3_stream upload_stream, z3_stream download_stream,
                              z3_host_step **out);

/* One layer step from host memory.  grads_host: bf16 [N][grad_stride] in
 * host memory, read by the upload (page-locked memory lets the copy run
 * asynchronously; the caller keeps it unchanged until the call's stream has
 * passed this step).  shards_host: bf16 [N][S] host memory written by the
 * download, or NULL for no download.  The device state arguments and the
 * errors are those of z3_step_layer; stream must differ from both pipeline
 * streams. */
z3_status z3_host_step_run(z3_host_step *pipe, const uint16_t *grads_host,
                           uint16_t *shards, uint16_t *full, float scale,
                           float *master, float *m, float *v,
                           const z3_adam_hp *hp, int64_t step,
                           uint16_t *shards_host, z3_stream stream);

void z3_host_step_destroy(z3_host_step *pipe);

/* ---- stage 1 / stage 2 / plain data-parallel variants ------------------ */

/* Plain data-parallel all-reduce ([S3] communication list: the baseline's
 * one all-reduce; [ZS] "Stage 2 also partitions gradients": an all-reduce is
 * a reduce-scatter followed by an all-gather).  Writes the one replica of the
 * reduced gradient that every rank would hold:
 *   out[e] = scale * fold_k fp32(grads[k][e]), 0 <= e < Psi,
 * with the rank fold of z3_reduce_scatter (ascending rank order, binary32).
 * grads is read; out (fp32 [Psi]) is written. */
z3_status z3_allreduce(const z3_layout *layout, const uint16_t *grads,
                       int64_t grad_stride, float *out, float scale,
                       z3_stream stream);

/* The slice of a replicated fp32 tensor that each rank keeps ([ZS] "What
 * stage 1 partitions": each rank applies the optimiser only to its own slice
 * of the gradient it received):
 *   shards[r][o_p + j] = full[F_p + r*s_p + j] for r*s_p + j < n_p, 0 in the
 * pad.  full (fp32 [Psi]) is read; shards (fp32 [N][S]) is written. */
z3_status z3_scatter(const z3_layout *layout, const float *full, float *shards,
                     z3_stream stream);

/* ---- checkpoint resharding --------------------------------------------- */

/* Re-lays one [N][S] state buffer of a layer from src_layout's rank count to
 * dst_layout's ([ZS] "Where the shards live and what happens on failure":
 * loading a per-rank shard set at a different P needs a reshuffle, not a
 * file copy).  Both layouts must describe the same parameters (same n_p, in
 * order).  For every destination position with padded index i = r'*s'_p + j'
 * < n_p: dst[r'][o'_p + j'] = src[i / s_p][o_p + i mod s_p]; pad positions
 * get 0.  elem_bytes is 2 (bf16 shards) or 4 (fp32 master, m, v, gradient
 * shards).  src is read, dst written; they must not overlap.  Errors:
 * different parameter lists (INVALID_ARG), elem_bytes not 2 or 4
 * (INVALID_ARG), and the usual buffer checks. */
z3_status z3_reshard(const z3_layout *src_layout, const z3_layout *dst_layout,
                     int32_t elem_bytes, const void *src, void *dst,
                     z3_stream stream);

/* ---- the layer step without a caller-supplied gather buffer ------------ */

/* z3_step_layer for callers that cannot allocate device memory.  The pages
 * that define the method have no counterpart of this call; it exists because
 * some callers cannot call cudaMalloc (code running inside an allocator
 * callback, a plugin that only receives buffers from its host framework, a
 * process whose device memory is all reserved up front) and so cannot
 * provide z3_step_layer's transient gather buffer `full`.
 *
 * The step is z3_step_layer's with grad_shards_or_NULL = NULL: the same
 * kernels, the same results, and the caller still passes (and owns) shards,
 * grads, master, m and v.  The two all-gathers write into a static array in
 * the library's own device memory instead of `full`; nothing reads it back.
 * Limits and sharing:
 *   - The array holds 16,777,216 bf16 elements (32 MiB).  A layer with more
 *     elements (Psi) is rejected with Z3_ERR_INVALID_ARG and a message that
 *     names both sizes; nothing is enqueued.
 *   - The array occupies 32 MiB on every GPU where the library's device code
 *     is loaded, until the process exits.
 *   - All calls on a device share it, and it keeps what the last call wrote.
 *     Nothing in it needs to start at zero (each gather writes every element
 *     the step uses), but calls that overlap on the GPU (on different streams,
 *     without ordering between them) race on it.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and keeps it for the
 *     rest of the process.  Make that first call before any stream capture,
 *     and do not call this entry point on a device after cudaDeviceReset
 *     there (the reset ends the context that the kept address belongs to).
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  Errors: those of z3_step_layer, the size limit above, and
 * Z3_ERR_CUDA if the address lookup fails. */
z3_status z3_step_layer_noalloc(const z3_layout *layout, uint16_t *shards,
                                const uint16_t *grads, int64_t grad_stride,
                                float scale, float *master, float *m, float *v,
                                const z3_adam_hp *hp, int64_t step,
                                z3_stream stream);

/* ---- errors ------------------------------------------------------------ */

/* Static name of a status code. */
const char *z3_status_string(z3_status status);

/* Copies the message of the calling thread's last failure (NUL-terminated,
 * truncated to len) into buf; returns the full message length. */
size_t z3_last_error(char *buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* Z3_H */
