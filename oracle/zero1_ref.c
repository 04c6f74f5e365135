/*
 * zero1_ref.c -- plain, single-threaded CPU oracle for one ZeRO-1
 * data-parallel optimizer step over W emulated ranks.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this file.  It shares no code, header,
 * table or constant with the CUDA library, and the library never calls it.
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no FMA contraction, no flush-to-zero, IEEE round-to-nearest-even).
 *
 * What one step computes (sources are web pages; cited by title + section):
 *
 *  [LEC7] "Stanford CS336 Lecture 7 close reading: Parallelism (part 1)",
 *         section 5.2 (ZeRO stage 1): every rank holds a full gradient;
 *         a reduce-scatter hands rank r the sum over ranks of slice r; rank
 *         r updates slice r with its own optimizer state; an all-gather
 *         returns the updated parameters to every rank.
 *  [LEC8] "Stanford CS336 Lecture 8 close reading: Parallelism (part 2)",
 *         section 2 (all-reduce = reduce-scatter + all-gather) and section 7
 *         (data parallel: gradients are averaged, ReduceOp.AVG).
 *  [PT]   "Parallel training" (notes.cassieliang.com):
 *         section "What one card holds: mixed precision and AdamW" -- fp32
 *         master weights receive the update and are cast to bf16 each step;
 *         fp32 m and v; reductions in fp32; the AdamW update with both bias
 *         corrections folded into the step size and the decoupled decay
 *         applied after the update; 2+2+4+4+4 = 16 bytes per parameter.
 *         section "Training loop and checkpoint" -- global-norm clipping:
 *         all gradients seen as one vector; if its L2 norm exceeds the
 *         threshold the whole vector is scaled down, direction kept.
 *         section "How cards talk: collective communication" -- the 4-rank
 *         worked example and the ring send volume 2*size*(W-1)/W.
 *         section "Data parallel and ZeRO" -- the 7.5B / 64-GPU memory table.
 *
 * Precision: the pages fix fp32 for master, m, v and for reductions, and
 * write the update as in-place ops on fp32 tensors, so every element
 * operation here is one fp32 operation rounded to nearest-even, in the order
 * the update is written.  Per-step scalars are formed in double and rounded
 * once to fp32, as a Python float scalar is when it meets an fp32 tensor.
 * The pages do not fix the norm's precision: it is a compensated double sum
 * of exact double squares.
 *
 * Parity pins: every function below is pinned by the not-gpu tests against
 * the pages' printed values, closed forms, torch.optim.AdamW special cases,
 * numpy/torch library routines and brute force (see tests/test_oracle_*.py).
 * The bf16-moment variant (zref_adamw_range_ex with moments_bf16) is a
 * reading: the pages only say that some configurations store m and v in
 * bf16.  It is the page's in-place ops applied to bf16 tensors, as torch
 * performs them: each op computes in fp32 and rounds its result to bf16,
 * and a scalar added to a bf16 tensor (eps) is rounded to bf16 first.
 * The tests pin that sequence, m, v, the denominator and the master, to
 * torch running those ops.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
float zref_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even on bit 16 (IEEE 754
 * roundTiesToEven applied to an 8-bit significand).  NaN stays NaN: sign
 * kept, quiet bit forced.  Overflow rounds to +-inf as RNE requires. */
uint16_t zref_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void zref_bf16_to_f32_array(const uint16_t *b, uint64_t count, float *out)
{
    for (uint64_t i = 0; i < count; ++i) out[i] = zref_bf16_to_f32(b[i]);
}

void zref_f32_to_bf16_array(const float *x, uint64_t count, uint16_t *out)
{
    for (uint64_t i = 0; i < count; ++i) out[i] = zref_f32_to_bf16(x[i]);
}

/* -------------------------------------------------------- shard layout */

/* Equal chunks: a reduce-scatter needs the buffer to split into W equal
 * pieces (LEC8 section 2: the input carries a world-size dimension).  Rank r
 * owns [r*S, min((r+1)*S, n)); the last shard may be short or empty. */
uint64_t zref_shard_len(uint64_t n, int world)
{
    return (n + (uint64_t)world - 1u) / (uint64_t)world;
}

static void shard_range(uint64_t n, int world, int r, uint64_t *lo, uint64_t *hi)
{
    uint64_t s = zref_shard_len(n, world);
    uint64_t a = (uint64_t)r * s, b = a + s;
    if (a > n) a = n;
    if (b > n) b = n;
    *lo = a;
    *hi = b;
}

/* --------------------------------------------------- per-step scalars */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay, max_norm;
} zref_hparams;

typedef struct {
    float inv_w;          /* 1/W, the averaging factor                    */
    float beta1, one_minus_beta1;
    float beta2, one_minus_beta2;
    float step_size;      /* lr * sqrt(1 - beta2^t) / (1 - beta1^t)         */
    float decay;          /* 1 - lr * weight_decay                          */
    float eps;
} zref_scalars;

/* PT "mixed precision and AdamW": both bias corrections are folded into the
 * step size; t counts steps from 1 (PT "training loop": bias correction
 * restarts from t = 1 when m, v are lost). */
void zref_step_scalars(const zref_hparams *hp, int world, uint64_t t, zref_scalars *s)
{
    double bc1 = 1.0 - pow(hp->beta1, (double)t);
    double bc2 = 1.0 - pow(hp->beta2, (double)t);
    s->inv_w = (float)(1.0 / (double)world);
    s->beta1 = (float)hp->beta1;
    s->one_minus_beta1 = (float)(1.0 - hp->beta1);
    s->beta2 = (float)hp->beta2;
    s->one_minus_beta2 = (float)(1.0 - hp->beta2);
    s->step_size = (float)(hp->lr * sqrt(bc2) / bc1);
    s->decay = (float)(1.0 - hp->lr * hp->weight_decay);
    s->eps = (float)hp->eps;
}

/* ------------------------------------------------------ reduce-scatter */

/* Element-wise mean over ranks of `count` bf16 gradient entries: widen to
 * fp32, add in rank order 0..W-1 starting from rank 0's value, then scale
 * by fp32(1/W).  grads[q] points at rank q's entries for this range. */
void zref_rs_mean_range(const uint16_t *const *grads, int world, uint64_t count,
                        float inv_w, float *out)
{
    for (uint64_t i = 0; i < count; ++i) {
        float s = zref_bf16_to_f32(grads[0][i]);
        for (int q = 1; q < world; ++q)
            s = s + zref_bf16_to_f32(grads[q][i]);
        out[i] = s * inv_w;
    }
}

/* Reduce-scatter with averaging (LEC7 5.2 step 2, LEC8 section 7): rank r
 * receives slice r of the averaged gradient.  Slice r is stored at
 * ghat[lo_r .. hi_r), so the W slices laid end to end are ghat[0 .. n). */
void zref_reduce_scatter_mean(const uint16_t *const *grads, int world, uint64_t n,
                              float *ghat)
{
    const float inv_w = (float)(1.0 / (double)world);
    const uint16_t *g[4096];
    for (int r = 0; r < world; ++r) {
        uint64_t lo, hi;
        shard_range(n, world, r, &lo, &hi);
        for (int q = 0; q < world; ++q) g[q] = grads[q] + lo;
        zref_rs_mean_range(g, world, hi - lo, inv_w, ghat + lo);
    }
}

/* ------------------------------------------------------ global L2 norm */

/* Running sum of squares: exact double products, Neumaier-compensated
 * double sum in index order (A. Neumaier, ZAMM 54, 1974).  `plain` is the
 * uncompensated IEEE sum, used so that an inf or NaN input gives an inf or
 * NaN norm rather than a NaN from the compensation term. */
typedef struct {
    double sum, comp, plain;
} zref_norm_acc;

void zref_norm_acc_init(zref_norm_acc *a)
{
    a->sum = 0.0;
    a->comp = 0.0;
    a->plain = 0.0;
}

void zref_norm_acc_add(zref_norm_acc *a, const float *x, uint64_t count)
{
    for (uint64_t i = 0; i < count; ++i) {
        double y = (double)x[i] * (double)x[i];
        double t = a->sum + y;
        if (fabs(a->sum) >= fabs(y))
            a->comp += (a->sum - t) + y;
        else
            a->comp += (y - t) + a->sum;
        a->sum = t;
        a->plain += y;
    }
}

double zref_norm_acc_value(const zref_norm_acc *a)
{
    if (!isfinite(a->plain))
        return sqrt(a->plain);
    return sqrt(a->sum + a->comp);
}

/* PT "training loop": scale the whole gradient when its norm exceeds the
 * threshold.  Clipping is off for max_norm <= 0.  A NaN norm with clipping
 * on gives a NaN coefficient; an infinite norm gives 0 (IEEE division). */
float zref_clip_coef(double norm, double max_norm)
{
    if (!(max_norm > 0.0))
        return 1.0f;
    if (isnan(norm))
        return (float)NAN;
    if (norm > max_norm)
        return (float)(max_norm / norm);
    return 1.0f;
}

/* ------------------------------------------------------------- AdamW */

/* AdamW on one slice (PT "mixed precision and AdamW"), every line one fp32
 * operation in the order the update is written:
 *   g  = ghat * c                       clipped averaged gradient
 *   m  = beta1*m + (1-beta1)*g          first moment
 *   v  = beta2*v + ((1-beta2)*g)*g      second moment
 *   d  = sqrt(v) + eps
 *   p  = master - step_size*(m/d)       folded bias correction
 *   p  = p * (1 - lr*wd)                decoupled decay, after the update */
void zref_adamw_range(float *master, float *m, float *v, const float *ghat,
                      uint64_t count, float c, const zref_scalars *s)
{
    for (uint64_t i = 0; i < count; ++i) {
        float g = ghat[i] * c;
        float mi = s->beta1 * m[i];
        mi = mi + s->one_minus_beta1 * g;
        float vi = s->beta2 * v[i];
        float og = s->one_minus_beta2 * g;
        vi = vi + og * g;
        float d = sqrtf(vi) + s->eps;
        float u = mi / d;
        float p = master[i] - s->step_size * u;
        p = p * s->decay;
        m[i] = mi;
        v[i] = vi;
        master[i] = p;
    }
}

/* ------------------------------------------------------ step variants */

/* Variants the pages name beside the default step:
 *   decay_before_update -- torch.optim.AdamW's order, p = p*(1-lr*wd) then
 *       p = p - step_size*(m/d) ("Parallel training", "mixed precision and
 *       AdamW": PyTorch decays first, the page's code decays after);
 *   clip_eps -- c = min(1, max_norm/(norm + clip_eps)), the form
 *       torch.nn.utils.clip_grad_norm_ uses with 1e-6; 0 is the page's rule;
 *   moments_bf16 -- m and v stored in bf16 ("some configurations store m, v
 *       in bf16, 12 bytes per parameter in total"): each in-place op on a
 *       moment computes in fp32 and rounds its result to bf16, so
 *       m = bf16(bf16(b1*m) + (1-b1)*g), v likewise, d = bf16(bf16(sqrt(v))
 *       + eps); the fp32 master update reads those bf16 values. */
typedef struct {
    int decay_before_update;
    double clip_eps;
    int moments_bf16;
} zref_options;

float zref_clip_coef_ex(double norm, double max_norm, double clip_eps)
{
    if (!(max_norm > 0.0))
        return 1.0f;
    if (isnan(norm))
        return (float)NAN;
    double q = max_norm / (norm + clip_eps);
    return q < 1.0 ? (float)q : 1.0f;
}

static float bf16_round(float x) { return zref_bf16_to_f32(zref_f32_to_bf16(x)); }

/* AdamW on one slice with options.  m and v point at float arrays, or at
 * uint16_t bf16 arrays when moments_bf16. */
void zref_adamw_range_ex(float *master, void *m, void *v, const float *ghat, uint64_t count, float c,
                         const zref_scalars *s, const zref_options *o)
{
    for (uint64_t i = 0; i < count; ++i) {
        float g = ghat[i] * c;
        float mi, vi, d;
        if (o->moments_bf16) {
            uint16_t *mb = (uint16_t *)m, *vb = (uint16_t *)v;
            mi = bf16_round(s->beta1 * zref_bf16_to_f32(mb[i]));
            mi = bf16_round(mi + s->one_minus_beta1 * g);
            vi = bf16_round(s->beta2 * zref_bf16_to_f32(vb[i]));
            float og = s->one_minus_beta2 * g;
            vi = bf16_round(vi + og * g);
            /* eps joins a bf16 tensor: torch rounds the scalar to bf16 */
            d = bf16_round(bf16_round(sqrtf(vi)) + bf16_round(s->eps));
            mb[i] = zref_f32_to_bf16(mi);
            vb[i] = zref_f32_to_bf16(vi);
        } else {
            float *mf = (float *)m, *vf = (float *)v;
            mi = s->beta1 * mf[i];
            mi = mi + s->one_minus_beta1 * g;
            vi = s->beta2 * vf[i];
            float og = s->one_minus_beta2 * g;
            vi = vi + og * g;
            d = sqrtf(vi) + s->eps;
            mf[i] = mi;
            vf[i] = vi;
        }
        float u = mi / d;
        float p = master[i];
        if (o->decay_before_update) {
            p = p * s->decay;
            p = p - s->step_size * u;
        } else {
            p = p - s->step_size * u;
            p = p * s->decay;
        }
        master[i] = p;
    }
}

/* --------------------------------------------------------- all-gather */

/* bf16 cast of the fp32 master (PT: "cast a bf16 copy for the forward each
 * step") and all-gather (LEC7 5.2 step 4): every replica q receives every
 * rank r's updated slice. */
void zref_all_gather_bf16(const float *master, int world, uint64_t n,
                          uint16_t *const *replicas, int n_replicas)
{
    for (int q = 0; q < n_replicas; ++q) {
        for (int r = 0; r < world; ++r) {
            uint64_t lo, hi;
            shard_range(n, world, r, &lo, &hi);
            for (uint64_t i = lo; i < hi; ++i)
                replicas[q][i] = zref_f32_to_bf16(master[i]);
        }
    }
}

/* ---------------------------------------------------------- one step */

/* One ZeRO-1 step over W emulated ranks (LEC7 5.2 steps 2-4).
 *   grads[W]      rank q's bf16 gradient, n entries (read only)
 *   replicas[W]   rank q's bf16 parameter copy, n entries (written)
 *   master, m, v  fp32 optimizer state, n entries (updated in place)
 *   ghat          fp32 scratch, n entries (holds the reduce-scatter result)
 *   t             1-based step number
 *   use_override  nonzero: use clip_override as the clip coefficient
 *                 instead of the one from the norm (parity injection)
 * Writes the norm of the averaged gradient and the coefficient used. */
void zref_step(uint64_t n, int world, const zref_hparams *hp, uint64_t t,
               const uint16_t *const *grads, uint16_t *const *replicas,
               float *master, float *m, float *v, float *ghat,
               int use_override, float clip_override,
               double *norm_out, float *clip_out)
{
    zref_scalars s;
    zref_step_scalars(hp, world, t, &s);

    zref_reduce_scatter_mean(grads, world, n, ghat);

    zref_norm_acc acc;
    zref_norm_acc_init(&acc);
    zref_norm_acc_add(&acc, ghat, n);
    double norm = zref_norm_acc_value(&acc);
    float c = use_override ? clip_override : zref_clip_coef(norm, hp->max_norm);

    for (int r = 0; r < world; ++r) {
        uint64_t lo, hi;
        shard_range(n, world, r, &lo, &hi);
        zref_adamw_range(master + lo, m + lo, v + lo, ghat + lo, hi - lo, c, &s);
    }

    zref_all_gather_bf16(master, world, n, replicas, world);

    if (norm_out) *norm_out = norm;
    if (clip_out) *clip_out = c;
}

/* One step with options; m and v as in zref_adamw_range_ex. */
void zref_step_ex(uint64_t n, int world, const zref_hparams *hp, const zref_options *o, uint64_t t,
                  const uint16_t *const *grads, uint16_t *const *replicas,
                  float *master, void *m, void *v, float *ghat,
                  int use_override, float clip_override,
                  double *norm_out, float *clip_out)
{
    zref_scalars s;
    zref_step_scalars(hp, world, t, &s);

    zref_reduce_scatter_mean(grads, world, n, ghat);

    zref_norm_acc acc;
    zref_norm_acc_init(&acc);
    zref_norm_acc_add(&acc, ghat, n);
    double norm = zref_norm_acc_value(&acc);
    float c = use_override ? clip_override : zref_clip_coef_ex(norm, hp->max_norm, o->clip_eps);

    const size_t msz = o->moments_bf16 ? sizeof(uint16_t) : sizeof(float);
    for (int r = 0; r < world; ++r) {
        uint64_t lo, hi;
        shard_range(n, world, r, &lo, &hi);
        zref_adamw_range_ex(master + lo, (char *)m + lo * msz, (char *)v + lo * msz, ghat + lo, hi - lo, c,
                            &s, o);
    }

    zref_all_gather_bf16(master, world, n, replicas, world);

    if (norm_out) *norm_out = norm;
    if (clip_out) *clip_out = c;
}

/* ------------------------------------------------ all-reduce (sum) pins */

/* All-reduce written directly: every rank receives the full rank-ordered
 * fp32 sum, rounded to bf16 (PT "collective communication", all_reduce). */
void zref_allreduce_sum_direct(const uint16_t *const *in, int world, uint64_t n,
                               uint16_t *const *out)
{
    for (int q = 0; q < world; ++q) {
        for (uint64_t i = 0; i < n; ++i) {
            float s = zref_bf16_to_f32(in[0][i]);
            for (int k = 1; k < world; ++k)
                s = s + zref_bf16_to_f32(in[k][i]);
            out[q][i] = zref_f32_to_bf16(s);
        }
    }
}

/* The same result as reduce-scatter (sum, or mean when `average`) into
 * per-rank slices of `scratch`, then all-gather of the bf16 slices (LEC8
 * section 2: all-reduce = reduce-scatter + all-gather). */
void zref_allreduce_rs_ag(const uint16_t *const *in, int world, uint64_t n,
                          int average, float *scratch, uint16_t *const *out)
{
    const float scale = average ? (float)(1.0 / (double)world) : 1.0f;
    const uint16_t *g[4096];
    for (int r = 0; r < world; ++r) {            /* reduce-scatter */
        uint64_t lo, hi;
        shard_range(n, world, r, &lo, &hi);
        for (int q = 0; q < world; ++q) g[q] = in[q] + lo;
        if (average) {
            zref_rs_mean_range(g, world, hi - lo, scale, scratch + lo);
        } else {
            for (uint64_t i = 0; i < hi - lo; ++i) {
                float s = zref_bf16_to_f32(g[0][i]);
                for (int q = 1; q < world; ++q)
                    s = s + zref_bf16_to_f32(g[q][i]);
                scratch[lo + i] = s;
            }
        }
    }
    zref_all_gather_bf16(scratch, world, n, out, world);   /* all-gather */
}

/* fp32 all-reduce, the dtype of the pages' worked example: written
 * directly (every rank sums all ranks' values in rank order 0..W-1, then
 * scales by fp32(1/W) when `average`), ... */
void zref_allreduce_f32_direct(const float *const *in, int world, uint64_t n, int average,
                               float *const *out)
{
    const float scale = (float)(1.0 / (double)world);
    for (int q = 0; q < world; ++q) {
        for (uint64_t i = 0; i < n; ++i) {
            float s = in[0][i];
            for (int k = 1; k < world; ++k)
                s = s + in[k][i];
            out[q][i] = average ? s * scale : s;
        }
    }
}

/* ... and as reduce-scatter into per-rank slices of `scratch` followed by
 * an all-gather of the slices (the two must agree bit for bit). */
void zref_allreduce_f32_rs_ag(const float *const *in, int world, uint64_t n, int average,
                              float *scratch, float *const *out)
{
    const float scale = (float)(1.0 / (double)world);
    for (int r = 0; r < world; ++r) {            /* reduce-scatter */
        uint64_t lo, hi;
        shard_range(n, world, r, &lo, &hi);
        for (uint64_t i = lo; i < hi; ++i) {
            float s = in[0][i];
            for (int q = 1; q < world; ++q)
                s = s + in[q][i];
            scratch[i] = average ? s * scale : s;
        }
    }
    for (int q = 0; q < world; ++q) {            /* all-gather */
        for (int r = 0; r < world; ++r) {
            uint64_t lo, hi;
            shard_range(n, world, r, &lo, &hi);
            for (uint64_t i = lo; i < hi; ++i)
                out[q][i] = scratch[i];
        }
    }
}

/* All-gather of shards ("Parallel training", "How cards talk: collective
 * communication": every rank receives the concatenation of all ranks'
 * pieces; "Lecture 7 close reading" 5.4: ZeRO-3 gathers each layer's
 * sharded parameters before using them).  Rank r holds elements
 * [r*S, min((r+1)*S, n)) of an n-element buffer, elem_size bytes each;
 * every output q receives all n elements.  A byte copy: no arithmetic. */
void zref_all_gather_shards(size_t elem_size, const void *const *shards, int world, uint64_t n,
                            uint64_t shard_len, void *const *outs)
{
    for (int q = 0; q < world; ++q) {
        for (int r = 0; r < world; ++r) {
            uint64_t lo = (uint64_t)r * shard_len, hi = lo + shard_len;
            if (lo > n) lo = n;
            if (hi > n) hi = n;
            if (hi > lo)
                memcpy((char *)outs[q] + lo * elem_size, shards[r], (size_t)(hi - lo) * elem_size);
        }
    }
}

/* ------------------------------------------------------- accounting */

/* Per-rank bytes of parameter-related memory (PT "data parallel and ZeRO";
 * LEC7 5.1): psi parameters, W ranks, k optimizer-state bytes per parameter
 * (12 for fp32 master + m + v), 2-byte params and 2-byte grads.
 *   stage 0: everything replicated          (2 + 2 + k) psi
 *   stage 1: optimizer state sharded         (2 + 2) psi + k psi / W
 *   stage 2: + gradients sharded             2 psi + (2 + k) psi / W
 *   stage 3: + parameters sharded            (2 + 2 + k) psi / W          */
double zref_zero_bytes_per_rank(int stage, double psi, int world, double k)
{
    double w = (double)world;
    switch (stage) {
    case 0: return (2.0 + 2.0 + k) * psi;
    case 1: return (2.0 + 2.0) * psi + k * psi / w;
    case 2: return 2.0 * psi + (2.0 + k) * psi / w;
    case 3: return (2.0 + 2.0 + k) * psi / w;
    default: return -1.0;
    }
}

/* Ring collectives (PT "collective communication"): W-1 steps of size/W
 * each for a reduce-scatter or an all-gather; an all-reduce is both.
 * op 0 = all-reduce, 1 = reduce-scatter, 2 = all-gather. */
double zref_ring_send_bytes(double size, int world, int op)
{
    double one = size * (double)(world - 1) / (double)world;
    return op == 0 ? 2.0 * one : one;
}
