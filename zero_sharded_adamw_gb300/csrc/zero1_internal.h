// zero1_internal.h -- declarations shared by the C-ABI host code
// (zero1_host.cu, zero1_noalloc.cu, zero1_allreduce.cu) and the step's
// kernels (zero1_kernels.cu).  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zero1 {

constexpr int kVec = 8;          // parameters per 16-byte vector of bf16
constexpr int kShardAlign = 64;  // shard length multiple (256-byte fp32 shard starts)
// Automatic one-launch path: at most this many parameters and bytes per step
// (measured crossover against the two-kernel path on GB300).
constexpr uint64_t kSmallAutoMaxN = 32768;
constexpr uint64_t kSmallAutoBytes = 6ull << 20;

// Device-resident result of the norm pass and, for capturable handles, the
// step counter and learning rate (library-owned).
struct DevStatus {
    double nsq;        // sum of squares of the averaged gradient
    double norm;       // sqrt(nsq)
    float clip;        // coefficient the update kernel multiplies into g
    unsigned ticket;   // last-CTA election counter; 0 between launches
    unsigned flags;    // bit 0: the norm is not finite (rewritten every step)
    unsigned errors;   // sticky: bit 0 = a pipeline wait gave up (1 s limit)
    unsigned long long t;  // capturable: steps taken (the update kernel's last CTA advances it)
    double lr;             // capturable: the handle's own learning-rate slot
    unsigned ticket2;      // capturable: update-kernel CTA counter; 0 between launches
    unsigned pad;
};

// Capturable steps: the step size and decay are formed on the device from
// the step counter in DevStatus, a learning rate read through lr, and the
// bias corrections (1 - beta1^t, 1 - beta2^t) tabulated by the host for
// t = 1..tab_len (both are exactly 1.0 in double from t = tab_len on).
struct DevScalars {
    const double2 *bc;     // nullptr: the launch's host-formed scalars are used
    uint64_t tab_len;
    const double *lr;
    double weight_decay;
};
constexpr unsigned kFlagNonFinite = 1u;
constexpr unsigned kErrWaitTimeout = 1u;

// Per-step fp32 scalars, formed on the host in double and rounded once.
struct StepScalars {
    float inv_w;       // 1/W
    float beta1, omb1; // beta1, 1 - beta1
    float beta2, omb2; // beta2, 1 - beta2
    float step_size;   // lr * sqrt(1 - beta2^t) / (1 - beta1^t)
    float decay;       // 1 - lr * weight_decay
    float eps;
};

// Everything one step's two launches need.
struct StepLaunch {
    const void *const *grads;   // W device pointers (bf16, n entries)
    void *const *params;        // W device pointers (bf16, n entries)
    int world;
    uint64_t n;
    float *master;              // fp32 master, n (padded) entries, 256-B aligned
    void *m, *v;                // fp32 moments, or bf16 when moments_bf16
    float *ghat;                // fp32 reduce-scatter result, or nullptr: re-read grads
    double *partials;           // 2 * grid_rs doubles
    DevStatus *status;
    StepScalars sc;
    double max_norm;
    int grid_rs;                // CTAs of the reduce-scatter + norm kernel
    int grid_update;            // CTAs of the update + all-gather kernel
    // step variants (defaults: the pages' step)
    bool moments_bf16 = false;  // m, v stored in bf16 (then m, v point at bf16 arrays)
    bool decay_first = false;   // torch.optim.AdamW's order
    double clip_eps = 0.0;      // c = min(1, max_norm / (norm + clip_eps))
    // bucketed (ZeRO-2 style) step
    int phase = 0;                  // 0: both kernels, 1: reduce-scatter only, 2: update only
    double *bucket_sums = nullptr;  // phase 1: written at [2*bucket_index]; phase 2: read
    int bucket_index = 0;
    int nbuckets = 0;
    // small steps: > 0 selects the one-launch cluster kernel with this many
    // 8-parameter vectors per thread (see small_step_vpt)
    int small_vpt = 0;
    DevScalars dev{};       // capturable handles
    bool advance_t = true;  // capturable: the update launch advances the device step counter
    bool stall_test = false; // failure test: the update kernel's waits run out (zero1_options)
    double load_rate_gbs = 0.0;  // > 0: the update kernel's loads phased for this device-wide rate
};

// The one-launch path for small n: a cluster of kSmallCtas CTAs of
// kSmallThreads threads, each thread holding up to kSmallMaxVpt vectors.
#ifndef ZERO1_SMALL_CTAS
#define ZERO1_SMALL_CTAS 8
#define ZERO1_SMALL_THREADS 256
#endif
constexpr int kSmallCtas = ZERO1_SMALL_CTAS;        // 8 is the portable cluster maximum
constexpr int kSmallThreads = ZERO1_SMALL_THREADS;
constexpr int kSmallMaxVpt = 4;
constexpr uint64_t kSmallCap = (uint64_t)kSmallCtas * kSmallThreads * kVec * kSmallMaxVpt;   // 65,536

// Vectors per thread (1, 2 or 4) for the one-launch path, or 0 for the
// two-kernel path.  mode: 0 = automatic (n and the bytes it moves both
// small), 1 = whenever n fits (n <= kSmallCap), -1 = never.
inline int small_step_vpt(uint64_t n, int world, int mode)
{
    if (mode < 0 || n > kSmallCap) return 0;
    if (mode == 0 && (n > kSmallAutoMaxN || n * (4ull * (uint64_t)world + 24ull) > kSmallAutoBytes)) return 0;
    const uint64_t per = (uint64_t)kSmallCtas * kSmallThreads * kVec;
    return n <= per ? 1 : n <= 2 * per ? 2 : 4;
}

// Enqueue the reduce-scatter + norm kernel, then the update + all-gather
// kernel (or, when small_vpt > 0, the one-launch kernel).  `ev`, when not
// null, holds three events recorded before, between and after the two
// kernels (before, after and after the one-launch kernel).
cudaError_t launch_step(const StepLaunch &s, cudaStream_t stream, cudaEvent_t *ev);

// cudaFuncSetAttribute(kernel, max dynamic shared memory, bytes) once per
// (kernel, device): the attribute stays with the context, and skipping the
// call keeps a step's host path short and free of non-stream calls (so a
// step can be captured in a CUDA graph after one uncaptured step).
cudaError_t allow_dynamic_smem(const void *kernel, int bytes);
// The same once-per-(kernel, device, attribute) rule for any function attribute.
cudaError_t set_func_attribute_once(const void *kernel, cudaFuncAttribute attr, int value);

// Grid sizes: one wave of resident CTAs on this device, capped by the work.
void plan_grids(uint64_t n, bool reread, int num_sms, int *grid_rs, int *grid_update);

// Set the message zero1_last_error() returns on this thread.
void set_error_message(const char *msg);

}  // namespace zero1
