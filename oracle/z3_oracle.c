/*
 * z3_oracle.c -- plain, slow, obviously-correct CPU oracle for the ZeRO-3
 * sharded model-state path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry point and the CPU-baseline leg of the benchmark may load this
 * code.  The CUDA library never links, includes or calls it, and it shares no
 * header, helper, table or constant with the CUDA library.
 *
 * Every function is a per-element loop over the definition it cites.  No
 * blocking, fusion or reordering beyond what the definition states.  Build
 * with -O2 -ffp-contract=off (no fused multiply-add), so each float
 * expression is evaluated as separate IEEE-754 binary32 operations in the
 * order written.
 *
 * Sources (page titles; sections as printed on the pages):
 *   [ZD] "The ZeRO-3 Diagram Most People Remember Is Wrong"
 *        (duoan.github.io), s.2 "The Actual Parameter Partition",
 *        s.3 "The Collectives You Should Expect", s.4 "Why This Is Still
 *        ZeRO, Not Tensor Parallelism".
 *   [S3] "ZeRO Stage 3: Parameter Partitioning" (mbrenndoerfer.com),
 *        eq. M_Stage3, the 7B worked example and the communication-volume
 *        list.
 *   [ZS] "ZeRO Stages: Sharding Optimizer State, Gradients, and Parameters"
 *        (mercemay.com), "What stage 1 partitions", "Stage 2 also partitions
 *        gradients", "Stage 3 partitions parameters", "Communication volume
 *        compared" (table).
 *   Adam itself is not written out on any page; it is the textbook update of
 *   Kingma & Ba, "Adam: A Method for Stochastic Optimization",
 *   arXiv:1412.6980, Algorithm 1 (bias-corrected moments, eps added outside
 *   the square root), with decoupled weight decay.
 *
 * Notation (per parameter p of a layer, N = number of logical ranks):
 *   n_p  element count;  s_p = ceil(n_p / N) elements per rank;
 *   o_p  offset of p inside each rank's shard (sum of s_q, q < p);
 *   F_p  offset of p in the unpadded full buffer (sum of n_q, q < p);
 *   S    rank stride of the shard buffers (sum of s_p);
 *   rank r owns padded positions [r*s_p, (r+1)*s_p) of parameter p.
 * Shard buffers are [N][S] rank-major; rank r's shard starts at r*S.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Layout.  [ZD] s.2: each parameter is flattened to 1-D, padded when its    */
/* element count does not divide by N, and each rank gets one contiguous     */
/* slice.  [ZS] "What stage 1 partitions": rank i owns [i*N/P, (i+1)*N/P).   */
/* Readings: padding is per parameter and minimal (s_p = ceil(n_p/N)); the   */
/* pad sits at the end of the flattened parameter; a rank's shard is the     */
/* concatenation of its slices in parameter order with no gaps.              */
/* ------------------------------------------------------------------------ */
int or_layout(const int64_t *numel, int32_t n_params, int32_t n_ranks,
              int64_t *shard_numel, int64_t *shard_off, int64_t *full_off,
              int64_t *out_S, int64_t *out_psi, int64_t *out_psi_padded)
{
    if (n_params < 1 || n_ranks < 1)
        return -1;
    int64_t S = 0;
    int64_t psi = 0;
    for (int32_t p = 0; p < n_params; ++p) {
        int64_t n = numel[p];
        if (n < 0)
            return -1;
        /* smallest s with s * N >= n */
        int64_t s = n / n_ranks;
        if (s * n_ranks < n)
            s += 1;
        shard_numel[p] = s;
        shard_off[p] = S;
        full_off[p] = psi;
        S += s;
        psi += n;
    }
    *out_S = S;
    *out_psi = psi;
    *out_psi_padded = S * (int64_t)n_ranks;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32.  The 2-byte parameter copy is bfloat16: the top 16 bits of */
/* an IEEE-754 binary32.  fp32 -> bf16 rounds to nearest, ties to even,     */
/* written from the bit layout; NaN stays a (quiet) NaN.                     */
/* ------------------------------------------------------------------------ */
uint16_t or_bf16_from_f32(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint32_t exponent = (u >> 23) & 0xffu;
    uint32_t mantissa = u & 0x7fffffu;
    if (exponent == 0xffu && mantissa != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN: keep sign, set quiet bit */
    uint32_t kept = u >> 16;        /* sign, exponent, top 7 mantissa bits */
    uint32_t dropped = u & 0xffffu; /* the 16 bits that are rounded away  */
    int round_up;
    if (dropped > 0x8000u)
        round_up = 1;
    else if (dropped < 0x8000u)
        round_up = 0;
    else
        round_up = (int)(kept & 1u); /* exact tie: round to the even neighbour */
    /* A carry out of the mantissa moves to the next binade (or to infinity),
     * which is the correctly rounded result. */
    return (uint16_t)(kept + (uint32_t)round_up);
}

float or_f32_from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

void or_bf16_from_f32_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_bf16_from_f32(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Partition (initialisation).  [ZD] s.2 steps 1-4 and s.3 (a broadcast may  */
/* appear at initialisation; the steady state is gather/scatter).           */
/* shard[r][o_p + j] = x_p[r*s_p + j] if that index is < n_p, else 0 (pad). */
/* The fp32 master takes the value, m = v = 0, the bf16 shard is RNE(x).    */
/* ------------------------------------------------------------------------ */
void or_partition(const int64_t *numel, const int64_t *shard_numel,
                  const int64_t *shard_off, const int64_t *full_off,
                  int32_t n_params, int32_t n_ranks, int64_t S,
                  const float *full, uint16_t *shards_bf16, float *master,
                  float *m, float *v)
{
    for (int32_t r = 0; r < n_ranks; ++r) {
        for (int32_t p = 0; p < n_params; ++p) {
            for (int64_t j = 0; j < shard_numel[p]; ++j) {
                int64_t i = (int64_t)r * shard_numel[p] + j; /* padded index */
                float x = 0.0f;
                if (i < numel[p])
                    x = full[full_off[p] + i];
                int64_t at = (int64_t)r * S + shard_off[p] + j;
                master[at] = x;
                m[at] = 0.0f;
                v[at] = 0.0f;
                shards_bf16[at] = or_bf16_from_f32(x);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* AllGather.  [ZD] s.3: before forward or backward compute, ranks gather   */
/* the full parameter; [S3] the gathered layer is the transient buffer.     */
/* Output is one copy of the full layer, parameters concatenated unpadded: */
/* full[F_p + i] = shard[i / s_p][o_p + i mod s_p], 0 <= i < n_p.           */
/* Element-size generic (2 bytes for the bf16 parameters, 4 for fp32).      */
/* ------------------------------------------------------------------------ */
static void gather_bytes(const int64_t *numel, const int64_t *shard_numel,
                         const int64_t *shard_off, const int64_t *full_off,
                         int32_t n_params, int64_t S, const void *shards,
                         void *full, size_t elem)
{
    const unsigned char *src = (const unsigned char *)shards;
    unsigned char *dst = (unsigned char *)full;
    for (int32_t p = 0; p < n_params; ++p) {
        for (int64_t i = 0; i < numel[p]; ++i) {
            int64_t r = i / shard_numel[p];
            int64_t j = i % shard_numel[p];
            memcpy(dst + (size_t)(full_off[p] + i) * elem,
                   src + (size_t)(r * S + shard_off[p] + j) * elem, elem);
        }
    }
}

void or_allgather(const int64_t *numel, const int64_t *shard_numel,
                  const int64_t *shard_off, const int64_t *full_off,
                  int32_t n_params, int64_t S, const uint16_t *shards_bf16,
                  uint16_t *full_bf16)
{
    gather_bytes(numel, shard_numel, shard_off, full_off, n_params, S,
                 shards_bf16, full_bf16, sizeof(uint16_t));
}

void or_allgather_f32(const int64_t *numel, const int64_t *shard_numel,
                      const int64_t *shard_off, const int64_t *full_off,
                      int32_t n_params, int64_t S, const float *shards,
                      float *full)
{
    gather_bytes(numel, shard_numel, shard_off, full_off, n_params, S, shards,
                 full, sizeof(float));
}

/* ------------------------------------------------------------------------ */
/* Rank fold of one gradient element.  [ZS] "Stage 2 also partitions        */
/* gradients": the reduce-scatter sums across ranks.  Reading: fp32 left    */
/* fold in ascending rank order starting from rank 0's value (bf16 -> fp32  */
/* is exact), then one multiply by scale (1/N gives the data-parallel mean).*/
/* ------------------------------------------------------------------------ */
static float fold_ranks(const uint16_t *grads, int64_t grad_stride,
                        int32_t n_ranks, int64_t e, float scale)
{
    float acc = or_f32_from_bf16(grads[e]);
    for (int32_t k = 1; k < n_ranks; ++k)
        acc = acc + or_f32_from_bf16(grads[(int64_t)k * grad_stride + e]);
    return acc * scale;
}

/* ------------------------------------------------------------------------ */
/* ReduceScatter.  [ZD] s.3 (gradients go back to the owning shards), [ZS]  */
/* "Stage 2 also partitions gradients" (each rank receives the summed slice */
/* it owns; the output buffer holds one slice per rank) and its second      */
/* subtlety (reduce per micro-batch, accumulate the reduced slices).        */
/* grads: rank k's full gradient starts at k*grad_stride (bf16).            */
/* out[r][o_p + j] = fold(...) for r*s_p + j < n_p, 0 in the pad.           */
/* accumulate != 0: out = out_old + fold(...) (pad still written 0).        */
/* ------------------------------------------------------------------------ */
void or_reduce_scatter(const int64_t *numel, const int64_t *shard_numel,
                       const int64_t *shard_off, const int64_t *full_off,
                       int32_t n_params, int32_t n_ranks, int64_t S,
                       const uint16_t *grads, int64_t grad_stride, float *out,
                       float scale, int32_t accumulate)
{
    for (int32_t r = 0; r < n_ranks; ++r) {
        for (int32_t p = 0; p < n_params; ++p) {
            for (int64_t j = 0; j < shard_numel[p]; ++j) {
                int64_t i = (int64_t)r * shard_numel[p] + j;
                int64_t at = (int64_t)r * S + shard_off[p] + j;
                if (i >= numel[p]) {
                    out[at] = 0.0f;
                    continue;
                }
                float g = fold_ranks(grads, grad_stride, n_ranks,
                                     full_off[p] + i, scale);
                out[at] = accumulate ? out[at] + g : g;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* All-reduce over the unsharded tensor, element by element, with the same  */
/* rank fold.  [ZS] "Stage 2 also partitions gradients": an all-reduce is a */
/* reduce-scatter followed by an all-gather.  Used as the comparator of     */
/* that identity and of the unsharded data-parallel step.                   */
/* ------------------------------------------------------------------------ */
void or_allreduce(int64_t psi, int32_t n_ranks, const uint16_t *grads,
                  int64_t grad_stride, float *out, float scale)
{
    for (int64_t e = 0; e < psi; ++e)
        out[e] = fold_ranks(grads, grad_stride, n_ranks, e, scale);
}

/* ------------------------------------------------------------------------ */
/* Adam on a flat fp32 range (a rank's shard, or an unsharded tensor).      */
/* [ZD] s.3 "optimizer updates local shard"; [S3] the model state is fp16   */
/* (here bf16) params and grads plus fp32 master and Adam moments; [ZS]     */
/* "What stage 1 partitions" (each rank updates only its own master slice). */
/* The hyperparameters are real numbers (double); every constant the update */
/* uses is rounded once to binary32:                                        */
/*   b1 = f(beta1), c1 = f(1 - beta1), b2 = f(beta2), c2 = f(1 - beta2),    */
/*   rb1 = f(1 / (1 - beta1^t)), rb2 = f(1 / (1 - beta2^t)),                */
/*   lr = f(lr), eps = f(eps), lwd = f(lr * weight_decay).                  */
/* Update (Kingma & Ba, Algorithm 1, in binary32, in this order; the bias   */
/* corrections m/(1-beta1^t) and v/(1-beta2^t) are applied as products with */
/* their reciprocals, which is the same quantity in exact arithmetic):      */
/*   m' = b1*m + c1*g;  v' = b2*v + c2*(g*g)                                */
/*   mh = m'*rb1;  vh = v'*rb2;  u = mh / (sqrt(vh) + eps)                  */
/*   p' = (p - lwd*p) - lr*u;  bf16 = RNE(p')                               */
/* ------------------------------------------------------------------------ */
typedef struct {
    float b1, c1, b2, c2, rb1, rb2, lr, eps, lwd;
} adam_consts;

static adam_consts adam_constants(double lr, double beta1, double beta2,
                                  double eps, double weight_decay,
                                  int64_t step)
{
    adam_consts k;
    k.b1 = (float)beta1;
    k.c1 = (float)(1.0 - beta1);
    k.b2 = (float)beta2;
    k.c2 = (float)(1.0 - beta2);
    k.rb1 = (float)(1.0 / (1.0 - pow(beta1, (double)step)));
    k.rb2 = (float)(1.0 / (1.0 - pow(beta2, (double)step)));
    k.lr = (float)lr;
    k.eps = (float)eps;
    k.lwd = (float)(lr * weight_decay);
    return k;
}

/* The nine binary32 constants, in the order of the struct above. */
void or_adam_constants(double lr, double beta1, double beta2, double eps,
                       double weight_decay, int64_t step, float *out9)
{
    adam_consts k = adam_constants(lr, beta1, beta2, eps, weight_decay, step);
    out9[0] = k.b1;
    out9[1] = k.c1;
    out9[2] = k.b2;
    out9[3] = k.c2;
    out9[4] = k.rb1;
    out9[5] = k.rb2;
    out9[6] = k.lr;
    out9[7] = k.eps;
    out9[8] = k.lwd;
}

void or_adam(int64_t n, float *master, float *m, float *v, const float *grad,
             uint16_t *param_bf16, double lr, double beta1, double beta2,
             double eps, double weight_decay, int64_t step)
{
    adam_consts k = adam_constants(lr, beta1, beta2, eps, weight_decay, step);
    for (int64_t i = 0; i < n; ++i) {
        float g = grad[i];
        float p = master[i];
        float m1 = k.b1 * m[i] + k.c1 * g;
        float v1 = k.b2 * v[i] + k.c2 * (g * g);
        float mh = m1 * k.rb1;
        float vh = v1 * k.rb2;
        float u = mh / (sqrtf(vh) + k.eps);
        float pd = p - k.lwd * p;
        float p1 = pd - k.lr * u;
        m[i] = m1;
        v[i] = v1;
        master[i] = p1;
        param_bf16[i] = or_bf16_from_f32(p1);
    }
}

/* ------------------------------------------------------------------------ */
/* One layer step on the sharded state, in the order of [ZD] s.3:           */
/* forward AllGather, backward AllGather, ReduceScatter of the gradients,   */
/* then the local-shard Adam update.  Adam runs on every position of the    */
/* [N][S] shard buffers; pad positions carry g = m = v = p = 0 and stay 0.  */
/* full_fwd/full_bwd receive the two gathers; grad_shards the reduced fp32  */
/* slices.  grad_acc (may be NULL) holds micro-batch sums reduced earlier:  */
/* the reduced gradient is then grad_acc + fold (accumulate mode).          */
/* ------------------------------------------------------------------------ */
void or_step_layer(const int64_t *numel, const int64_t *shard_numel,
                   const int64_t *shard_off, const int64_t *full_off,
                   int32_t n_params, int32_t n_ranks, int64_t S,
                   uint16_t *shards_bf16, uint16_t *full_fwd,
                   uint16_t *full_bwd, const uint16_t *grads,
                   int64_t grad_stride, float scale, const float *grad_acc,
                   float *grad_shards, float *master, float *m, float *v,
                   double lr, double beta1, double beta2, double eps,
                   double weight_decay, int64_t step)
{
    int64_t total = S * (int64_t)n_ranks;
    or_allgather(numel, shard_numel, shard_off, full_off, n_params, S,
                 shards_bf16, full_fwd);
    or_allgather(numel, shard_numel, shard_off, full_off, n_params, S,
                 shards_bf16, full_bwd);
    if (grad_acc != NULL)
        for (int64_t x = 0; x < total; ++x)
            grad_shards[x] = grad_acc[x];
    or_reduce_scatter(numel, shard_numel, shard_off, full_off, n_params,
                      n_ranks, S, grads, grad_stride, grad_shards, scale,
                      grad_acc != NULL);
    or_adam(total, master, m, v, grad_shards, shards_bf16, lr, beta1, beta2,
            eps, weight_decay, step);
}

/* ------------------------------------------------------------------------ */
/* Accounting.  [S3] eq. M_Stage3: per-rank model state is 16 bytes per     */
/* owned element (2 param + 2 grad + 4 master + 4 m + 4 v), 16*Psi/N when   */
/* N divides every n_p.  [ZS] "What stage 1 partitions" counts 18 bytes     */
/* (4-byte gradients); that variant is reported beside it.                  */
/* [S3] communication list: forward AllGather 2*Psi + backward AllGather    */
/* 2*Psi + ReduceScatter 2*Psi = 6*Psi bytes per step, against 2*Psi for a  */
/* plain data-parallel all-reduce.  [ZS] table, stage-3 row: per rank about */
/* 3*Psi*(P-1)/P elements.                                                  */
/* ------------------------------------------------------------------------ */
void or_accounting(int64_t S, int64_t psi, int32_t n_ranks,
                   int64_t *state_bytes_per_rank_16,
                   int64_t *state_bytes_per_rank_18,
                   int64_t *step_volume_bytes, int64_t *dp_volume_bytes,
                   double *per_rank_ring_elems_stage3,
                   double *per_rank_ring_elems_dp)
{
    *state_bytes_per_rank_16 = (2 + 2 + 4 + 4 + 4) * S;
    *state_bytes_per_rank_18 = (2 + 4 + 4 + 4 + 4) * S;
    *step_volume_bytes = 2 * psi + 2 * psi + 2 * psi;
    *dp_volume_bytes = 2 * psi;
    double frac = (double)(n_ranks - 1) / (double)n_ranks;
    *per_rank_ring_elems_stage3 = 3.0 * (double)psi * frac;
    *per_rank_ring_elems_dp = 2.0 * (double)psi * frac;
}
