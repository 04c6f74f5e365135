/*
 * zero1.h -- C ABI of a GB300 (sm_103a) ZeRO-1 data-parallel optimizer step.
 *
 * One step of ZeRO stage 1 over W data-parallel ranks:
 *   1. reduce-scatter of the W ranks' bf16 gradients: rank r receives slice r
 *      of the rank-ordered fp32 sum, scaled by 1/W (gradient averaging);
 *   2. the global L2 norm of the averaged gradient and the clip coefficient;
 *   3. AdamW on each rank's fp32 master / m / v slice;
 *   4. bf16 cast of the updated master and all-gather into all W replicas.
 *
 * Sources (web pages, cited by title and section):
 *   "Stanford CS336 Lecture 7 close reading: Parallelism (part 1)",
 *     section 5.2 (ZeRO stage 1: reduce-scatter, per-slice update with the
 *     slice's own optimizer state, all-gather of the updated parameters).
 *   "Stanford CS336 Lecture 8 close reading: Parallelism (part 2)",
 *     section 2 (all-reduce = reduce-scatter + all-gather) and section 7
 *     (data parallel: gradients averaged with ReduceOp.AVG).
 *   "Parallel training" (notes.cassieliang.com), section "What one card
 *     holds: mixed precision and AdamW" (fp32 master, m, v; the update with
 *     folded bias correction and decoupled decay after the update; bf16 copy
 *     for the forward), section "Training loop and checkpoint" (global-norm
 *     clipping; a checkpoint holds m, v and the step count t).
 *
 * Emulation: the W ranks live in one GPU's memory.  Rank r's gradient and
 * parameter replica are caller buffers grad_ptrs[r] and param_ptrs[r]; the
 * library owns the fp32 optimizer state of all W slices.  No collective
 * library is involved: the reduce-scatter is a rank-ordered read of the W
 * gradient buffers and the all-gather is a W-way store.
 *
 * Conventions for every entry point:
 *   - Return 0 on success or a negative ZERO1_E* code; zero1_last_error()
 *     then holds a message (thread-local).  Nothing aborts the process.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued on it; calls return without waiting
 *     unless stated.
 *   - Device buffers must be 16-byte aligned (ZERO1_EALIGN otherwise).
 *   - A handle is used by one host thread and one stream at a time.
 *   - Numerics: no FMA contraction on the reduce-scatter sums and the AdamW
 *     update; every fp32 operation is IEEE round-to-nearest-even, so for a
 *     given clip coefficient the state and replicas are bit-for-bit those of
 *     the plain fp32 definition.  The norm is accumulated in compensated fp32
 *     per thread and fp64 across threads, in a fixed order (deterministic for
 *     a given n, W and device).
 */
#ifndef ZERO1_H
#define ZERO1_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO1_OK        0
#define ZERO1_EINVAL   -1   /* null pointer, n = 0, bad world size, bad hyperparameter, bad handle */
#define ZERO1_EALIGN   -2   /* a device buffer is not 16-byte aligned                             */
#define ZERO1_ENOMEM   -3   /* a device allocation failed                                         */
#define ZERO1_ECUDA    -4   /* a CUDA runtime call or a kernel launch failed                      */
#define ZERO1_ENODEV   -5   /* no CUDA device, or the device is not compute capability 10.3      */

/* Largest number of emulated ranks one handle accepts. */
#define ZERO1_MAX_WORLD 512

/* AdamW + clipping hyperparameters.
 *   lr, beta1, beta2, eps, weight_decay: the AdamW update
 *       m = beta1*m + (1-beta1)*g,  v = beta2*v + (1-beta2)*g*g,
 *       p = p - lr*sqrt(1-beta2^t)/(1-beta1^t) * m/(sqrt(v)+eps),
 *       p = p * (1 - lr*weight_decay)
 *     ("Parallel training", "mixed precision and AdamW").  0 <= beta < 1,
 *     eps >= 0, lr >= 0, weight_decay >= 0.
 *   max_norm: global-norm clipping threshold; <= 0 disables clipping
 *     ("Parallel training", "training loop and checkpoint"). */
typedef struct zero1_hparams {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    double max_norm;
} zero1_hparams;

typedef struct zero1_ctx *zero1_handle;

/* Create an optimizer for n parameters over `world` emulated ranks
 * ("Stanford CS336 Lecture 7 close reading: Parallelism (part 1)", section
 * 5.2: under ZeRO stage 1 each rank keeps the optimizer state of its own
 * slice of the parameters only).
 * Allocates the fp32 master, m and v (each W*S floats, S the shard length
 * below) plus scratch on the current CUDA device with cudaMalloc; m = v = 0,
 * master = 0, t = 0.  Load real weights with zero1_set_state.
 * Shards: rank r owns parameters [r*S, min((r+1)*S, n)) with
 * S = ceil(n/W) rounded up to a multiple of 64 (256-byte aligned shard
 * starts); the padding past n is never read or written by a step.
 * Scratch: W >= 3 keeps the fp32 reduce-scatter result (4*W*S bytes) between
 * the two kernels; W <= 2 re-reads the gradients instead (cheaper in bytes).
 * Errors: ZERO1_EINVAL (out == NULL, hp == NULL, n == 0, world outside
 * [1, ZERO1_MAX_WORLD], bad hyperparameters), ZERO1_ENODEV, ZERO1_ENOMEM.
 * On error *out is set to NULL. */
int zero1_create(uint64_t n, int world, const zero1_hparams *hp, zero1_handle *out);

/* Variants of the step the pages name beside the default (all zero = the
 * default step of zero1_create):
 *   decay_before_update: 1 = torch.optim.AdamW's order, p = p*(1-lr*wd) and
 *     then p = p - step_size*m/(sqrt(v)+eps); 0 = after the update, as the
 *     page's code does ("Parallel training", "mixed precision and AdamW").
 *   clip_eps: c = min(1, max_norm/(norm + clip_eps)); 0 is the page's rule,
 *     torch.nn.utils.clip_grad_norm_ uses 1e-6.
 *   moments_bf16: 1 = m and v stored in bf16 (the pages' note that some
 *     configurations keep them in bf16: 12 bytes per parameter in all); each
 *     moment update computes in fp32 and rounds to bf16 per operation:
 *     m = bf16(bf16(b1*m) + (1-b1)*g), v = bf16(bf16(b2*v) + (1-b2)*g*g),
 *     d = bf16(bf16(sqrt(v)) + bf16(eps)) (a scalar added to a bf16 tensor
 *     is rounded to bf16, as torch does); the fp32 master update uses
 *     those.
 *   bucket_ctas: CTAs of each zero1_bucket_reduce launch (0 = one per SM).
 *     Fewer leave SMs to a backward running alongside on another stream.
 *   small_step: the one-launch path for small n (a single thread-block
 *     cluster runs the whole step; n <= 65,536): 0 = automatic (taken when
 *     n <= 32,768 and (4W+24)*n <= 6 MiB), 1 = whenever n <= 65,536,
 *     -1 = never.  Either path computes the same update; only the order of
 *     the norm's partial sums differs (see zero1_get_grad_norm).
 *   capturable: 1 = the step counter t and the learning rate live in
 *     device memory and the kernels form each step's step size and decay
 *     there, so zero1_step (and zero1_bucket_finish) can be captured in a
 *     CUDA graph and replayed: every replay is the next step.  The bias
 *     corrections 1 - beta^t are tabulated by the host at create time with
 *     the same double operations as the host path, up to the step where
 *     both are exactly 1.0 (at most 2^22 steps: 64 MiB; beta2 = 0.99999
 *     needs 3.7M, beta2 = 0.999999 is refused), so the results equal a
 *     non-capturable handle's bit for bit.  zero1_set_lr then waits for the
 *     device; zero1_set_lr_ptr reads lr from a caller's device double
 *     (for schedules inside a graph); zero1_get_state reads t from the
 *     device; zero1_set_state writes it.  Profiling (zero1_profile_start)
 *     must not be active while a step is being captured.
 *   inject_wait_timeout: failure testing only.  1 = the update kernel's
 *     producer issues no loads, so every pipeline wait of that kernel runs
 *     out after its 1 s limit; the step returns without hanging, and
 *     zero1_get_grad_norm then reports ZERO1_ECUDA (the sticky timeout bit).
 *     Applies to the two-kernel path (set small_step = -1 for small n).
 *   host_chunk: parameters per chunk of the host-buffer steps
 *     (zero1_step_host, zero1_step_host_async); 0 = the default, which makes
 *     one ring slot (W ranks' bf16 slices of a chunk) 256 MiB.  Rounded down
 *     to a multiple of 2048 (at least 2048); at most 65,536 chunks.
 *   load_phase_gbs: load phasing of the update kernel.  Where the replica
 *     stores far outweigh the loads (the fp32-scratch step with fp32
 *     moments at W >= 16: 16 bytes loaded against 12 + 2W stored per
 *     parameter), loads issued one tile at a time by each SM reach DRAM
 *     scattered among the stores and cost more than their bytes.  Phased,
 *     each CTA issues a tile's loads only at the next boundary of a period
 *     that every SM shares (the global nanosecond clock), so the grid's
 *     loads arrive together (measured on GB300: the update 3.7% faster at
 *     W = 16, 4-6% at 20 to 32, 9% at 48, 8-13% at 64 to 256, 6% at 512;
 *     below W = 16 every period tried was slower, so it stays off).  The
 *     period is the time one tile's bytes take when the grid moves them at
 *     a device-wide rate: 0 = the built-in rule (14000 GB/s, half a tile's
 *     time, at 16 <= W < 20; 7000 GB/s from W = 20; off below W = 16; and
 *     17500 GB/s, about 0.4 of a tile's time, for the W <= 2 step that
 *     re-reads the gradients, 16 bytes in and 16 out per parameter, where
 *     it measured 1.2% faster), > 0 = this rate in GB/s for any W on
 *     either path, < 0 = never.  Only update
 *     launches that have the device to themselves and span every SM are
 *     phased: zero1_step's and zero1_bucket_finish's, not
 *     zero1_bucket_update's (beside a backward) nor the host-buffer steps'
 *     pieces (beside the next step's reduces and the copies).  Timing
 *     only: results are the same bit for bit.  Must be finite, and a
 *     positive rate at least 1000 GB/s (a slower one would only stretch
 *     the step).
 *   size: sizeof(zero1_options) (lets the struct grow). */
typedef struct zero1_options {
    uint32_t size;
    int32_t decay_before_update;
    double clip_eps;
    int32_t moments_bf16;
    int32_t bucket_ctas;
    int32_t small_step;
    int32_t capturable;
    int32_t inject_wait_timeout;
    uint64_t host_chunk;
    double load_phase_gbs;
} zero1_options;

/* zero1_create with step variants (opts may be NULL: the default step).
 * Errors as zero1_create, plus ZERO1_EINVAL for a bad opts->size, a
 * negative or non-finite clip_eps, a negative bucket_ctas, small_step
 * outside {-1, 0, 1}, capturable or inject_wait_timeout outside {0, 1}, a
 * non-finite load_phase_gbs or one in (0, 1000), and a capturable handle
 * whose bias corrections would need more than 2^22 table entries.  All
 * option checks come before any device call. */
int zero1_create_ex(uint64_t n, int world, const zero1_hparams *hp, const zero1_options *opts,
                    zero1_handle *out);

/* Free the handle and its device memory after synchronizing the device.
 * NULL is accepted and ignored.  Returns ZERO1_OK or ZERO1_ECUDA. */
int zero1_destroy(zero1_handle h);

/* One ZeRO-1 step (t -> t+1) on `stream`, fully asynchronous, allocation-free
 * ("Stanford CS336 Lecture 7 close reading: Parallelism (part 1)", section
 * 5.2: reduce-scatter the gradients, update each rank's slice with its own
 * optimizer state, all-gather the updated parameters; the update itself as
 * "Parallel training", "What one card holds: mixed precision and AdamW").
 *   grad_ptrs:  host array of W device pointers; rank r's bf16 gradient,
 *               n entries, 16-byte aligned.  Only read.
 *   param_ptrs: host array of W device pointers; rank r's bf16 parameter
 *               replica, n entries, 16-byte aligned.  Only written: every
 *               replica receives bf16(master) of all n parameters.
 * The pointer arrays themselves are copied into the launch; the buffers must
 * stay valid until the stream reaches the step.  Gradient and replica
 * buffers must not overlap each other or the library's state.
 * Launches two kernels, the reduce-scatter + norm kernel and the clip +
 * AdamW + bf16 + all-gather kernel, or, for small n (zero1_options
 * small_step), one kernel that does all of it (zero1_step_launches).
 * Errors: ZERO1_EINVAL (NULL handle / array / entry), ZERO1_EALIGN,
 * ZERO1_ECUDA (launch failure; t is then left unchanged). */
int zero1_step(zero1_handle h, const void *const *grad_ptrs, void *const *param_ptrs, void *stream);

/* The same step for callers whose gradients and replicas live in host
 * memory, and waits for it: the W host gradients are uploaded, reduced,
 * updated and the W replicas downloaded chunk by chunk (zero1_options
 * host_chunk) through two bounded device rings, so the device memory the
 * host path needs does not grow with n:
 *   - rings: 2 x 8 slots of W x chunk bf16 (4 GiB at the default chunk),
 *     each direction's chunks dealt over 4 copy streams;
 *   - for W <= 2, an fp32 reduce-scatter scratch of 4*W*S bytes (the plain
 *     step re-reads the gradients instead, which the host path cannot).
 * Per step, every chunk is uploaded and reduce-scattered (with its norm
 * partial) on an internal stream; after the last chunk the norm and clip
 * coefficient are formed from the partials in chunk order, and every chunk
 * is updated, cast, all-gathered into a download slot and copied back.
 *   host_grads:  W host pointers, n bf16 each (pinned memory recommended).
 *   host_params: W host pointers, n bf16 each, written.
 * The step starts after earlier work on `stream`, and later work on
 * `stream` starts after it.  The first call allocates the rings (and the
 * W <= 2 scratch) and creates the internal streams and events;
 * zero1_destroy frees them.  For a given clip coefficient the result equals
 * zero1_step's bit for bit; the norm is summed in a chunking-dependent
 * (fixed) order.  No profile events are recorded.  Refused while a
 * bucketed step is open.  Errors as zero1_step, plus ZERO1_ENOMEM. */
int zero1_step_host(zero1_handle h, const void *const *host_grads, void *const *host_params, void *stream);

/* A ZeRO-2-style bucketed step ("Lecture 7 close reading", section 5.3:
 * each layer's gradients are reduced to their owner as soon as the backward
 * produces them and then freed; "Parallel training", "data parallel and
 * ZeRO": buckets, and communication overlapped with the backward).  The
 * same step as zero1_step, delivered in pieces:
 *   zero1_bucket_begin(h): open a step.  The first call allocates the
 *     bucket bookkeeping (64 KB) and, for W <= 2, an fp32 reduce-scatter
 *     scratch of 4*W*S bytes.
 *   zero1_bucket_reduce(h, offset, count, grad_ptrs, stream): reduce-scatter
 *     parameters [offset, offset+count) -- grad_ptrs[r] points at rank r's
 *     gradient for exactly that range (16-byte aligned; offset a multiple of
 *     8) -- into the handle's fp32 scratch and record the range's norm
 *     partial.  The gradient buffers may be reused once `stream` passes the
 *     call.  Issue all of one step's buckets on one stream (they share
 *     per-launch scratch); that stream may run alongside the caller's
 *     backward on another.  At most 4096 buckets, in any order; they may
 *     not overlap, and only the bucket that ends at n may have a count that
 *     is not a multiple of 8.
 *   zero1_bucket_update(h, offset, count, grad_ptrs, param_ptrs, stream):
 *     for handles without clipping (max_norm <= 0), where no step of the
 *     update waits for the global norm: the bucket's reduce-scatter and,
 *     right after it, the AdamW + bf16 + all-gather of the bucket's own
 *     parameters.  param_ptrs[r] points at rank r's replica for exactly
 *     that range.  So the whole optimizer step runs beside the backward.
 *     One step uses zero1_bucket_reduce or zero1_bucket_update, not both;
 *     not available on capturable handles.
 *   zero1_bucket_finish(h, param_ptrs, stream): the buckets must cover
 *     [0, n) exactly once (else ZERO1_EINVAL and the step is abandoned;
 *     buckets already updated by zero1_bucket_update stay updated); forms
 *     the norm from the buckets' partials in call order, clips, runs the
 *     AdamW + bf16 + all-gather kernel over all n, t -> t+1.  After
 *     zero1_bucket_update buckets it launches nothing (param_ptrs may be
 *     NULL) and only advances t; the norm was recorded with the last
 *     bucket.
 * The result equals zero1_step's for the same clip coefficient bit for bit;
 * the norm itself is summed in a bucketing-dependent (but fixed) order.
 * zero1_step is refused while a bucketed step is open. */
int zero1_bucket_begin(zero1_handle h);
int zero1_bucket_reduce(zero1_handle h, uint64_t offset, uint64_t count, const void *const *grad_ptrs,
                        void *stream);
int zero1_bucket_update(zero1_handle h, uint64_t offset, uint64_t count, const void *const *grad_ptrs,
                        void *const *param_ptrs, void *stream);
int zero1_bucket_finish(zero1_handle h, void *const *param_ptrs, void *stream);

/* The host-buffer step, pipelined: enqueue and return.  The same chunked
 * step as zero1_step_host, on the handle's internal streams: step t+1's
 * chunk i is reduced as soon as step t's update of chunk i has read the
 * scratch it overwrites, so one step's replica downloads overlap the next
 * step's gradient uploads (the two directions of the host link run at
 * once).  The step starts after earlier work on `stream`; any later call on
 * the handle that touches its state (zero1_step, the state copies, the
 * norm, the bucketed step) is ordered after it on that call's stream.  The
 * caller must keep host_grads unchanged and must not read host_params until
 * zero1_host_sync(h) returns (host buffers may be the same every call).
 * Errors as zero1_step_host. */
int zero1_step_host_async(zero1_handle h, const void *const *host_grads, void *const *host_params, void *stream);

/* Wait for all work of the handle's host-buffer steps (copies and kernels).
 * Errors: ZERO1_EINVAL, ZERO1_ECUDA. */
int zero1_host_sync(zero1_handle h);

/* Checkpoint restore ("Parallel training", "training loop and checkpoint":
 * a checkpoint carries m, v and t).  master, m, v: arrays of n entries in
 * device or host memory (copied with cudaMemcpyDefault): master fp32, m and
 * v fp32, or bf16 for a handle created with moments_bf16; m or v may be
 * NULL, meaning zeros.  t: the number of steps already taken (the next step
 * uses t+1).  Enqueued on `stream`; a pageable host source is consumed
 * before the call returns.  On a capturable handle t is also written to the
 * device counter, and the call waits for `stream`.
 * Errors: ZERO1_EINVAL, ZERO1_ECUDA. */
int zero1_set_state(zero1_handle h, const float *master, const void *m, const void *v,
                    uint64_t t, void *stream);

/* Checkpoint save ("Parallel training", "Training loop and checkpoint": a
 * checkpoint must hold m, v and the step count t, or bias correction
 * restarts from t = 1 without the moments): copies master (n fp32), m and
 * v (n fp32 each, or bf16 on a moments_bf16 handle) into device or host
 * arrays (any may be NULL to skip it) and writes the step count to *t (may
 * be NULL).  Enqueued on `stream`; synchronize it before reading a host
 * destination.  On a capturable handle t is read from the device counter
 * (replayed graphs advance it), which waits for `stream`. */
int zero1_get_state(zero1_handle h, float *master, void *m, void *v, uint64_t *t, void *stream);

/* The same two copies for parameters [offset, offset+count) only -- one
 * rank's shard is offset = r*S, count = min(S, n - r*S) -- so that each rank
 * can save or load its own slice.  The step count is untouched.
 * Errors: ZERO1_EINVAL (range outside [0, n), NULL master for set). */
int zero1_set_state_range(zero1_handle h, uint64_t offset, uint64_t count, const float *master,
                          const void *m, const void *v, void *stream);
int zero1_get_state_range(zero1_handle h, uint64_t offset, uint64_t count, float *master,
                          void *m, void *v, void *stream);

/* Change the learning rate used by later steps (schedules such as warmup +
 * cosine, "Parallel training", "training loop and checkpoint").  On a
 * capturable handle it writes the handle's device lr slot after waiting for
 * the whole device (steps already enqueued keep the old rate).
 * Errors: ZERO1_EINVAL for a NULL handle or lr < 0 or not finite,
 * ZERO1_ECUDA. */
int zero1_set_lr(zero1_handle h, double lr);

/* Capturable handles only: later steps (and replays of captured steps)
 * read the learning rate from the device double at device_lr, which the
 * caller may update on the step's stream (e.g. a schedule kernel captured
 * in the same graph); it must stay valid while such steps run.  NULL goes
 * back to the handle's own slot (set by zero1_set_lr).
 * Errors: ZERO1_EINVAL (no handle, or a non-capturable one), ZERO1_EALIGN
 * (not 8-byte aligned). */
int zero1_set_lr_ptr(zero1_handle h, const double *device_lr);

/* Norm of the averaged gradient of the latest step and the clip coefficient
 * it applied (1 when not clipped) ("Parallel training", "Training loop and
 * checkpoint": the gradient is clipped by its global L2 norm, scaled down
 * when the norm exceeds max_norm).  The norm is returned in double because
 * the kernels finish it in fp64; the coefficient is the fp32 value the
 * update multiplied into every gradient element, so a caller (or a test)
 * can repeat the update exactly.  Both live in device memory written by the
 * step's kernels, so the read is ordered on `stream`, the stream the step
 * ran on, and waits for it.  Either output may
 * be NULL.  Before the first step both read 0.  Returns ZERO1_ECUDA if any
 * step of this handle had a kernel pipeline wait give up (each wait is
 * bounded to 1 s so that a fault cannot hang the GPU); the state is then not
 * valid. */
int zero1_get_grad_norm(zero1_handle h, double *norm, float *clip_coef, void *stream);

/* Layout facts: the shard length S, the padded state length W*S, and the
 * bytes of device memory the handle holds (state + scratch, excluding the
 * host-buffer steps' rings and scratch).  Any output may be NULL. */
int zero1_layout(zero1_handle h, uint64_t *shard_len, uint64_t *padded_len, uint64_t *device_bytes);

/* Per-kernel timing.  After zero1_profile_start, each of the next
 * `capacity` steps records three CUDA events on its stream (before the
 * reduce-scatter + norm kernel, between the kernels, after the update +
 * all-gather kernel).  zero1_profile_stop waits for the last recorded event
 * and returns the summed kernel times in milliseconds and the number of
 * steps recorded; it frees the events.  Either kernel's average launch
 * duration is its sum divided by *steps.  On the one-launch path the first
 * interval is the whole kernel and the second is empty.  Outputs may be
 * NULL.  Errors: ZERO1_EINVAL (capacity < 1, or stop without start),
 * ZERO1_ECUDA. */
int zero1_profile_start(zero1_handle h, int capacity);
int zero1_profile_stop(zero1_handle h, double *rs_norm_ms, double *update_ms, uint64_t *steps);

/* Kernel launches one zero1_step makes with this handle: 2, or 1 on the
 * one-launch small-n path.  Errors: ZERO1_EINVAL. */
int zero1_step_launches(zero1_handle h, int *launches);

/* The per-step kernel times recorded so far, before zero1_profile_stop:
 * waits for the last recorded event, then writes step i's reduce-scatter +
 * norm and update + all-gather durations (ms) to rs_norm_ms[i] and
 * update_ms[i] for i < min(recorded, capacity) and the number recorded to
 * *steps.  Arrays are caller-owned host memory and may be NULL.  The events
 * stay alive.  Errors: ZERO1_EINVAL (no profiling started), ZERO1_ECUDA. */
int zero1_profile_read(zero1_handle h, float *rs_norm_ms, float *update_ms, uint64_t capacity, uint64_t *steps);

/* Host-only planning (no device needed).  The shard length S = ceil(n/W)
 * rounded up to 64 and the padded state length W*S for n parameters over
 * `world` ranks.  Errors: ZERO1_EINVAL (n == 0 or world out of range). */
int zero1_shard_plan(uint64_t n, int world, uint64_t *shard_len, uint64_t *padded_len);

/* Host-only: the fp32 scalars step number t (1-based) multiplies with,
 * formed in double and rounded once ("Parallel training", "mixed precision
 * and AdamW"): out[0..7] = 1/W, beta1, 1-beta1, beta2, 1-beta2,
 * lr*sqrt(1-beta2^t)/(1-beta1^t), 1-lr*weight_decay, eps.
 * Errors: ZERO1_EINVAL (NULL pointer, t == 0, bad world or hyperparameter). */
int zero1_step_scalars(const zero1_hparams *hp, int world, uint64_t t, float out[8]);

/* One step that allocates no device memory, for callers that cannot call
 * cudaMalloc: a framework whose caching allocator has reserved the device's
 * memory, a plug-in whose host fixes its device memory up front, or a loop
 * that cannot take the device synchronisation cudaMalloc/cudaFree imply.
 * The pages have no counterpart to this entry point; it is the same two
 * kernels as zero1_step with the caller owning all state (and the built-in
 * load-phasing rule of zero1_options.load_phase_gbs = 0).
 *   n, world, hp: as zero1_create; n is limited to 4,194,304 parameters
 *     (larger n: ZERO1_EINVAL with a message; use zero1_create/zero1_step).
 *   t: this step's number, 1-based (the caller keeps the count).
 *   grad_ptrs, param_ptrs: as zero1_step.
 *   master, m, v: caller-owned device fp32 arrays of n entries, 16-byte
 *     aligned, updated in place (m = v = 0 before the first step).
 * Scratch (the fp32 reduce-scatter result, norm partials and status) is a
 * fixed ~16.1 MiB array inside the library image, held by every GPU that
 * loads the library until the process exits.  The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress) with the
 * device current; make that first call before any stream capture.  The
 * address is kept with the identity of the CUDA context it belongs to, and
 * a call made in another context (for instance after cudaDeviceReset)
 * looks it up again.  Each call clears the scratch status on `stream`
 * first.  All calls share the one array: calls whose GPU work overlaps
 * (other streams or threads) race.  The norm is not read back by this
 * call, and neither is the bit a kernel pipeline wait sets when it gives up
 * after its 1 s limit: a timeout on this path is not reported (the next
 * call clears it).
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ENODEV, ZERO1_ECUDA. */
int zero1_step_noalloc(uint64_t n, int world, const zero1_hparams *hp, uint64_t t,
                       const void *const *grad_ptrs, void *const *param_ptrs,
                       float *master, float *m, float *v, void *stream);

/* Element types and reductions of zero1_allreduce. */
#define ZERO1_DTYPE_BF16 0
#define ZERO1_DTYPE_F32  1
#define ZERO1_OP_SUM     0
#define ZERO1_OP_AVG     1

/* The data-parallel (DDP) all-reduce of W emulated ranks' buffers
 * ("Parallel training", "How cards talk: collective communication": every
 * rank receives the element-wise sum; "Stanford CS336 Lecture 8 close
 * reading: Parallelism (part 2)", section 7: DDP averages gradients with
 * all_reduce(op=AVG)).  out_ptrs[q][i] = (in_ptrs[0][i] + in_ptrs[1][i] +
 * ... + in_ptrs[W-1][i]), summed in fp32 in rank order 0..W-1, times fp32(1/W)
 * for ZERO1_OP_AVG, rounded to the element type (bf16: nearest even).  Equal
 * bit for bit to a reduce-scatter followed by an all-gather.
 *   n: elements per rank (>= 1); world: 1..ZERO1_MAX_WORLD;
 *   dtype: ZERO1_DTYPE_BF16 or ZERO1_DTYPE_F32; op: ZERO1_OP_SUM or _AVG;
 *   in_ptrs, out_ptrs: host arrays of W device pointers, 16-byte aligned;
 *     out_ptrs[r] may equal in_ptrs[r] (in place); other overlaps are not
 *     allowed.
 *   errors: optional device word (NULL = none); bit 0 is set if a kernel
 *     pipeline wait gave up (1 s limit), in which case the outputs are not
 *     valid.
 * Asynchronous on `stream`; allocates nothing.  One kernel launch.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_allreduce(uint64_t n, int world, int dtype, int op, const void *const *in_ptrs,
                    void *const *out_ptrs, unsigned *errors, void *stream);

/* The all-reduce over a handle's W emulated ranks: zero1_allreduce(n, W,
 * ZERO1_DTYPE_BF16, ZERO1_OP_SUM, in_ptrs, out_ptrs, NULL, stream) with the
 * handle's n and W ("Stanford CS336 Lecture 8 close reading: Parallelism
 * (part 2)", section 2: all-reduce = reduce-scatter + all-gather; the
 * pages' worked example sums [0,1,2,3] + rank over 4 ranks to [6,10,14,18]).
 * in_ptrs, out_ptrs: W device pointers to n bf16 each (16-byte aligned;
 * out may equal in).  Touches none of the handle's optimizer state.
 * Errors: as zero1_allreduce, and ZERO1_EINVAL for an unknown handle. */
int zero1_allreduce_sum(zero1_handle h, const void *const *in_ptrs, void *const *out_ptrs, void *stream);

/* The ZeRO-3 / FSDP parameter all-gather ("Lecture 7 close reading:
 * Parallelism (part 1)", section 5.4: before a layer runs, its sharded
 * parameters are all-gathered onto every rank; "Parallel training", "How
 * cards talk: collective communication": all-gather concatenates every
 * rank's piece onto all ranks).  Rank r's shard_ptrs[r] holds elements
 * [r*S, min((r+1)*S, n)) of an n-element buffer (S = shard_len, a multiple
 * of 8, S*W >= n; ranks past n hold nothing and may pass any pointer);
 * every out_ptrs[q] receives all n elements.  A byte copy, bf16 or fp32.
 * In place is allowed: shard_ptrs[r] may be out_ptrs[r] + r*S elements.
 * Buffers 16-byte aligned; `errors` as zero1_allreduce.  Asynchronous on
 * `stream`; allocates nothing; one kernel launch.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_allgather(uint64_t n, int world, uint64_t shard_len, int dtype, const void *const *shard_ptrs,
                    void *const *out_ptrs, unsigned *errors, void *stream);

/* Two streams on disjoint groups of the current device's SMs, for running
 * the bucketed step beside a backward ("Lecture 7 close reading", section
 * 5.3; "Parallel training", "data parallel and ZeRO": communication hidden
 * behind the backward).  The library GEMMs of a backward are persistent
 * kernels that hold every SM until they end, so bucket reduces issued on
 * another stream find no SM free; kernels launched on stream_a run only on
 * the first group's SMs and kernels on stream_b only on the rest (each
 * group is a green context of the device).  Run the backward on one stream
 * and zero1_bucket_reduce / zero1_bucket_update on the other; order them
 * with events as with any two streams.
 *   sms_a: SMs wanted in the first group, 1 <= sms_a < the device's SM
 *     count; the driver rounds it up to its partition granularity, and
 *     sms_a / sms_b report the counts granted.
 * The streams are cudaStream_t values passed as void*; they belong to the
 * partition and stay valid until zero1_sm_partition_destroy, which waits
 * for the work queued on both to finish and then releases the green
 * contexts (ZERO1_ECUDA if that wait fails; the partition is released and
 * *part cleared either way).  Creating a partition changes no device
 * setting.
 * Errors: ZERO1_EINVAL (NULL out, sms_a out of range, nothing left for
 * the second group), ZERO1_ENODEV, ZERO1_ENOMEM, ZERO1_ECUDA (the driver
 * has no green contexts or refused the split). */
typedef struct zero1_sm_partition {
    void *stream_a;
    void *stream_b;
    int sms_a;
    int sms_b;
    void *opaque;
} zero1_sm_partition;

int zero1_sm_partition_create(int sms_a, zero1_sm_partition *out);
int zero1_sm_partition_destroy(zero1_sm_partition *part);

/* Message for the last error on this thread ("" if none). */
const char *zero1_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO1_H */
