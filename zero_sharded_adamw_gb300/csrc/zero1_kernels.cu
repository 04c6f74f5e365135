// zero1_kernels.cu -- the sm_103a kernels of one ZeRO-1 step.
//
//  K1  zero1_rs_norm_kernel   reduce-scatter (rank-ordered fp32 sum of the W
//                             bf16 gradients, times 1/W) fused with the
//                             squared L2 norm: per-thread compensated fp32,
//                             warp shuffles, one fp64 grid pass by the last
//                             CTA, which also forms the clip coefficient.
//  K2  zero1_adamw_ag_kernel  clip scale + AdamW on fp32 master/m/v + bf16
//                             cast + all-gather (W-way store of each tile).
//  K0  zero1_small_step_kernel  all of the above in one launch of one
//                             8-CTA thread-block cluster, for small n.
//
// Sources (web pages, cited by title and section):
//  "Stanford CS336 Lecture 7 close reading: Parallelism (part 1)", 5.2: the
//    ZeRO-1 step (reduce-scatter, per-slice update, all-gather).
//  "Stanford CS336 Lecture 8 close reading: Parallelism (part 2)", 2 and 7:
//    all-reduce = reduce-scatter + all-gather; gradients averaged.
//  "Parallel training" (notes.cassieliang.com), "mixed precision and AdamW":
//    fp32 master/m/v, reductions in fp32, the update with folded bias
//    correction and decay after it, bf16 copy of the master; "training loop
//    and checkpoint": clip the concatenated gradient to max_norm.
//
// Both kernels are HBM streams (no contraction, so no tensor cores) built as
// persistent, warp-specialised TMA pipelines, one CTA per SM:
//  - a producer warp moves tiles (2048-8192 parameters, per kernel and
//    path; see the configurations below) from HBM into a 3-4 stage
//    shared-memory ring with 1-D bulk copies (cp.async.bulk) that complete
//    on an mbarrier per stage;
//  - 8 or 16 consumer warps compute out of shared memory;
//  - K2 has a store warp whose lanes write the tile's master, m, v and W
//    bf16 replicas back with bulk stores, so the W-way all-gather costs the
//    SM one bulk instruction per replica per tile;
//  - where the stores far outweigh the loads (W >= 16), K2's producer
//    issues each tile's loads at the next boundary of a clock period that
//    every SM shares, so the grid's loads reach DRAM together instead of
//    one tile at a time among the stores (load phasing); the W <= 2
//    re-read path uses the same gate with a period of about 0.4 tile.
// Every mbarrier wait gives up after 1 s of global time: it raises the CTA's
// abort flag and a sticky error bit in the status the host reads; a producer
// that stops lets its loads in flight land before exiting.
//
// Every fp32 operation of the sum and the update is an explicit _rn
// intrinsic: no FMA contraction, IEEE round-to-nearest-even, no FTZ, so the
// results are those of the plain fp32 definition bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zero1_internal.h"
#include "zero1_ptx.cuh"

namespace zero1 {
namespace {

using namespace ptx;

// The reduce-scatter kernel's tiles, per path: each rank's slice of a tile
// is one bulk load of tile * 2 bytes, a stage holds `ranks` ranks' slices of
// one tile, and `stages` stages are in flight.  The size of each bulk copy
// sets the read rate (measured on GB300 with 152 CTAs streaming 8 GiB:
// 7.43-7.54 TB/s in 16 KB copies, 6.20 TB/s in 4 KB copies).  Measured
// per path in interleaved repeats on one box:
//  - gradients only read (W <= 2): 8192-parameter tiles, 2 ranks per stage
//    (16 KB copies, 128 KB in flight): the 7B step's reduce 4.23 -> 3.77 ms
//    against 2048-parameter tiles of 4 tiles x 2 ranks per stage;
//  - fp32 scratch written (W >= 3): 4096-parameter tiles, 4 ranks per stage
//    (8 KB copies), 0.1-0.4% faster than 2048 x 8 ranks and than 8192 x 2;
//    8192 x 1 x 8 stages and 8192 x 4 x 3 are 1-3% slower, and deeper rings
//    (192 KB in flight: 8192 x 2 x 6, 4096 x 4 x 6, 16384 x 1 x 6) 3-8%
//    slower, at W = 8 and at W = 64 alike.
struct RsConfig {
    int tile, ranks, stages;
};
#ifndef ZERO1_RS_SPILL_TILE
#define ZERO1_RS_SPILL_TILE 4096
#define ZERO1_RS_SPILL_RANKS 4
#define ZERO1_RS_SPILL_STAGES 4
#endif
#ifndef ZERO1_RS_READ_TILE
#define ZERO1_RS_READ_TILE 8192
#define ZERO1_RS_READ_RANKS 2
#define ZERO1_RS_READ_STAGES 4
#endif
constexpr RsConfig kRsSpill{ZERO1_RS_SPILL_TILE, ZERO1_RS_SPILL_RANKS, ZERO1_RS_SPILL_STAGES};
constexpr RsConfig kRsRead{ZERO1_RS_READ_TILE, ZERO1_RS_READ_RANKS, ZERO1_RS_READ_STAGES};
// 1: whole steps launch their two kernels with programmatic dependencies
// (programmatic dependent launch).  Off by default: measured in 50-step CUDA
// graphs on GB300 it was mixed -- 7% faster at 65,536 parameters (W = 4),
// 0.1% at 124M (W = 8), but 3% slower at 1M and 2% at 4M (W = 8).
#ifndef ZERO1_PDL
#define ZERO1_PDL 0
#endif
// The update kernel's tile, ring depth, consumer warps and tile order, per
// path (measured on GB300, gpt2_small / ragged / 7B / W = 64 / bf16-moment
// workloads):
//  - fp32 scratch, fp32 moments: write-heavy (16 B read, 12 + 2W written per
//    parameter); fastest with 2048-parameter tiles, 3 stages in flight and 16
//    consumer warps, tiles grid-strided;
//  - fp32 scratch, bf16 moments: 2048-parameter tiles, 4 stages, 8 warps;
//  - gradient re-read (W <= 2): 4096-parameter tiles, 3 stages, 8 warps, and
//    each CTA walking one contiguous run of tiles (1.5% faster than 2048 x 4
//    grid-strided at 2B parameters; the other paths lose 1-2% with runs).
// Tile order: grid-strided = CTA b takes tiles ntiles-1-b, ntiles-1-b-G, ...;
// runs = CTA b takes [b*ntiles/G, (b+1)*ntiles/G), from the top down.
struct UpdConfig {
    int tile, stages, warps;
    bool runs;
};
// (-D overrides for tuning: ZERO1_UPD_<PATH>_TILE / _STAGES / _WARPS / _RUNS.)
#ifndef ZERO1_UPD_SPILL_F32_STAGES
#define ZERO1_UPD_SPILL_F32_TILE 2048
#define ZERO1_UPD_SPILL_F32_STAGES 3
#define ZERO1_UPD_SPILL_F32_WARPS 16
#define ZERO1_UPD_SPILL_F32_RUNS false
#endif
#ifndef ZERO1_UPD_SPILL_BF16_STAGES
#define ZERO1_UPD_SPILL_BF16_TILE 2048
#define ZERO1_UPD_SPILL_BF16_STAGES 4
#define ZERO1_UPD_SPILL_BF16_WARPS 8
#define ZERO1_UPD_SPILL_BF16_RUNS false
#endif
#ifndef ZERO1_UPD_REREAD_STAGES
#define ZERO1_UPD_REREAD_TILE 4096
#define ZERO1_UPD_REREAD_STAGES 3
#define ZERO1_UPD_REREAD_WARPS 8
#define ZERO1_UPD_REREAD_RUNS true
#endif
constexpr UpdConfig kUpdSpillF32{ZERO1_UPD_SPILL_F32_TILE, ZERO1_UPD_SPILL_F32_STAGES, ZERO1_UPD_SPILL_F32_WARPS,
                                 ZERO1_UPD_SPILL_F32_RUNS};      // fp32 scratch, fp32 moments
constexpr UpdConfig kUpdSpillBf16{ZERO1_UPD_SPILL_BF16_TILE, ZERO1_UPD_SPILL_BF16_STAGES, ZERO1_UPD_SPILL_BF16_WARPS,
                                  ZERO1_UPD_SPILL_BF16_RUNS};   // fp32 scratch, bf16 moments
constexpr UpdConfig kUpdReread{ZERO1_UPD_REREAD_TILE, ZERO1_UPD_REREAD_STAGES, ZERO1_UPD_REREAD_WARPS,
                               ZERO1_UPD_REREAD_RUNS};          // gradients re-read (W <= 2)
constexpr int kConsumers = 256;                  // consumer threads of the reduce-scatter kernel
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kRsThreads = kConsumers + 32;      // + producer warp
static_assert(kRsSpill.tile % (kConsumers * kVec) == 0 && kRsRead.tile % (kConsumers * kVec) == 0,
              "consumers must tile the reduce-scatter tiles");

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// --------------------------------------------------------- kernel params

// Pointer tables live in the launch parameters (CAP slots, W used).
template <int CAP>
struct RsParams {
    const uint16_t *grads[CAP];
    float *ghat;              // nullptr: norm only
    double *partials;         // [2 * gridDim.x]
    DevStatus *status;
    uint64_t nvec;            // n / 8
    uint64_t n;
    int world;
    float inv_w;
    double max_norm;
    double clip_eps;          // c = min(1, max_norm / (norm + clip_eps))
    double *bucket_sums;      // bucketed step: this launch's (sum, plain sum) go to
    int bucket;               // bucket_sums[2*bucket .. +1] instead of forming c
};

template <int CAP>
struct UpdParams {
    const uint16_t *grads[CAP];  // re-read mode only
    uint16_t *params[CAP];
    const float *ghat;           // spill mode only
    float *master;
    void *m, *v;                 // fp32, or bf16 in the bf16-moment variant
    DevStatus *status;
    uint64_t nvec, n;
    int world;
    int decay_first;             // torch.optim.AdamW's decay order
    StepScalars sc;
    const double *bucket_sums;   // bucketed step: c comes from these nbuckets pairs
    int nbuckets;
    double max_norm, clip_eps;
    DevScalars dev;              // capturable: scalars formed from the device step counter
    int advance_t;               // capturable: this launch ends the step (advances the counter)
    int stall_test;              // failure test: the producer issues nothing, so every wait runs out
    unsigned long long load_period_ns;  // > 0: each tile's loads wait for the next boundary of this period
};

// Scalar rank-ordered sum for the last n % 8 parameters.
__device__ __forceinline__ float rank_sum1(const uint16_t *const *grads, int world, uint64_t e)
{
    float s = __uint_as_float((unsigned)grads[0][e] << 16);
    for (int r = 1; r < world; ++r) s = __fadd_rn(s, __uint_as_float((unsigned)grads[r][e] << 16));
    return s;
}

// ------------------------------------------------------- norm reduction

// Kahan-compensated fp32 running sum (W. Kahan, CACM 8(1), 1965): `hi - lo`
// carries the sum to about one fp32 rounding regardless of the count.
struct Kahan {
    float hi = 0.f, lo = 0.f, plain = 0.f;
    __device__ __forceinline__ void add(float x)
    {
        float y = __fsub_rn(x, lo);
        float t = __fadd_rn(hi, y);
        lo = __fsub_rn(__fsub_rn(t, hi), y);
        hi = t;
        plain = __fadd_rn(plain, x);
    }
};

__device__ __forceinline__ float sumsq8(const float g[8])
{
    float q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = __fmul_rn(g[k], g[k]);
    return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                     __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
}

// Fixed-order sum of two doubles over the consumer threads (warp shuffle
// tree, then warp 0); the result is valid in consumer thread 0.
__device__ __forceinline__ void consumer_sum2(double &a, double &b, double *sa, double *sb)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_down_sync(0xFFFFFFFFu, a, off);
        b += __shfl_down_sync(0xFFFFFFFFu, b, off);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sa[warp] = a;
        sb[warp] = b;
    }
    consumer_sync();
    if (warp == 0) {
        a = lane < kConsumerWarps ? sa[lane] : 0.0;
        b = lane < kConsumerWarps ? sb[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_down_sync(0xFFFFFFFFu, a, off);
            b += __shfl_down_sync(0xFFFFFFFFu, b, off);
        }
    }
    consumer_sync();
}

// The norm and clip coefficient from the sum of squares `x` and its
// uncompensated companion `y` (which carries inf/NaN): c = min(1,
// max_norm/(norm + clip_eps)) when clipping is on, NaN for a NaN norm.
__device__ __forceinline__ void finish_norm(double x, double y, double max_norm, double clip_eps, DevStatus *status,
                                            float *clip_out)
{
    const double nsq = isfinite(y) ? x : y;
    const double norm = sqrt(nsq);
    float c = 1.0f;
    if (max_norm > 0.0) {
        if (isnan(norm))
            c = __int_as_float(0x7FC00000);
        else if (max_norm / (norm + clip_eps) < 1.0)
            c = (float)(max_norm / (norm + clip_eps));
    }
    if (status) {
        status->nsq = nsq;
        status->norm = norm;
        status->clip = c;
        status->flags = isfinite(norm) ? 0u : kFlagNonFinite;
    }
    *clip_out = c;
}

// The step's scalars on a capturable handle: the host-formed constants with
// the step size lr * sqrt(1 - beta2^t) / (1 - beta1^t) and the decay
// 1 - lr * weight_decay formed here for step t, in the same double
// operations, in the same order, as the host forms them (so both give the
// same fp32 values bit for bit).
__device__ __forceinline__ StepScalars form_scalars(const StepScalars &base, const DevScalars &d, unsigned long long t)
{
    const uint64_t i = (t < d.tab_len ? t : d.tab_len) - 1;
    const double2 bc = d.bc[i];
    const double lr = *d.lr;
    StepScalars s = base;
    s.step_size = __double2float_rn(__ddiv_rn(__dmul_rn(lr, __dsqrt_rn(bc.y)), bc.x));
    s.decay = __double2float_rn(__dsub_rn(1.0, __dmul_rn(lr, d.weight_decay)));
    return s;
}

// ------------------------------------------------------------------- K1

// Parameters of tile j (of `tile` parameters) that lie in the 8-aligned
// vector part [0, nel).
__device__ __forceinline__ uint32_t rs_tile_count(uint64_t nel, uint64_t j, uint64_t tile)
{
    const uint64_t base = j * tile;
    return (uint32_t)(nel - base < tile ? nel - base : tile);
}

template <int TILE, int RANKS, int STAGES>
struct RsSmem {
    uint16_t g[STAGES][RANKS][TILE];   // 128 KB: RANKS (rank, tile) slices per stage
    uint64_t full[STAGES], empty[STAGES];
    double red_a[kConsumerWarps], red_b[kConsumerWarps];
    int abort;
    int last;
};

// Warps 0..7 consume, warp 8 produces.  A CTA's tiles are j = blockIdx.x,
// +gridDim.x, ... in increasing order; work item k of a CTA is (tile, rank
// group grp), the rank groups of a tile in increasing order, so each
// consumer thread's fp32 sums run over the ranks strictly in order 0..W-1.
// Consumer thread t owns the 8-parameter vectors q * 2048 + 8 t (q <
// tile / 2048) of every tile: a warp's 16-byte shared-memory reads are
// consecutive.
template <int W, int CAP, bool SPILL>
__global__ void __launch_bounds__(kRsThreads, 1)
zero1_rs_norm_kernel(const __grid_constant__ RsParams<CAP> p)
{
    constexpr RsConfig kCfg = SPILL ? kRsSpill : kRsRead;
    constexpr int kRsTile = kCfg.tile, kRsRanks = kCfg.ranks, kStages = kCfg.stages;
    constexpr int kRsVecs = kRsTile / (kConsumers * kVec);   // 8-parameter vectors per consumer thread per tile
    extern __shared__ __align__(128) unsigned char smem_raw[];
    RsSmem<kRsTile, kRsRanks, kStages> &sm = *reinterpret_cast<RsSmem<kRsTile, kRsRanks, kStages> *>(smem_raw);
    const int nw = W > 0 ? W : p.world;
    const int ngroups = (nw + kRsRanks - 1) / kRsRanks;
    const uint64_t nel = p.nvec * kVec;
    const uint64_t ntiles = (nel + kRsTile - 1) / kRsTile;
    // This CTA's tiles: blockIdx.x + i * gridDim.x for i < tcta.
    const uint32_t tcta = blockIdx.x < ntiles ? (uint32_t)((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0u;
    auto tile_of = [&](uint32_t i) -> uint64_t { return blockIdx.x + (uint64_t)i * gridDim.x; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort = &sm.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Launched with a programmatic dependency (whole steps without
    // profiling events): the update kernel may launch now; this kernel reads
    // nothing (the gradients may come from the kernel before it) until the
    // previous grid has completed.
    launch_dependents();
    grid_dependency_wait();

    if (warp == kConsumerWarps) {                                 // producer
        if (lane == 0) {
            // With a scratch ĝ, gradients go first out of L2 so that the ĝ
            // written last stays resident for the update kernel; when the
            // update kernel re-reads the gradients they keep normal priority.
            const uint64_t pol = SPILL ? policy_evict_first() : 0;
            uint32_t k = 0;
            for (uint32_t i = 0; i < tcta && !*abort; ++i) {
                const uint64_t base = tile_of(i) * kRsTile;
                const uint32_t cnt = rs_tile_count(nel, tile_of(i), kRsTile);
                for (int grp = 0; grp < ngroups; ++grp, ++k) {
                    const int s = k % kStages;
                    if (k >= kStages && !mbar_wait(&sm.empty[s], ((k / kStages) & 1u) ^ 1u, abort, &p.status->errors))
                        break;
                    const int r0 = grp * kRsRanks;
                    const int rn = nw - r0 < kRsRanks ? nw - r0 : kRsRanks;
                    mbar_arrive_expect_tx(&sm.full[s], (uint32_t)rn * cnt * 2u);
                    for (int r = 0; r < rn; ++r) {
                        if (SPILL)
                            tma_load_hint(sm.g[s][r], p.grads[r0 + r] + base, cnt * 2u, &sm.full[s], pol);
                        else
                            tma_load(sm.g[s][r], p.grads[r0 + r] + base, cnt * 2u, &sm.full[s]);
                    }
                }
            }
            if (*abort) drain_loads<kStages>(sm.full, k);
        }
        return;
    }

    // Consumers.
    Kahan acc;
    const uint64_t keep = policy_evict_last();
    uint32_t k = 0;
    float s[kRsVecs][8];
    for (uint32_t i = 0; i < tcta; ++i) {
        if (__any_sync(0xFFFFFFFFu, *abort != 0)) break;
        const uint64_t base = tile_of(i) * kRsTile;
        const uint32_t cnt = rs_tile_count(nel, tile_of(i), kRsTile);
        bool ok = true;
        for (int grp = 0; grp < ngroups; ++grp, ++k) {
            const int st = k % kStages;
            const bool got = mbar_wait(&sm.full[st], (k / kStages) & 1u, abort, &p.status->errors);
            if (!__all_sync(0xFFFFFFFFu, got)) {      // warp-uniform: no lane left behind
                ok = false;
                break;
            }
            const int rn = nw - grp * kRsRanks < kRsRanks ? nw - grp * kRsRanks : kRsRanks;
#pragma unroll
            for (int q = 0; q < kRsVecs; ++q) {
                const uint32_t e0 = (uint32_t)q * (kConsumers * kVec) + threadIdx.x * kVec;
                if (e0 < cnt) {
#pragma unroll
                    for (int r = 0; r < kRsRanks; ++r) {
                        if (r < rn) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(&sm.g[st][r][e0]);
                            if (grp == 0 && r == 0)
                                set_widened(s[q], raw);
                            else
                                add_widened(s[q], raw);
                        }
                    }
                    if (grp == ngroups - 1) {          // all W ranks summed: finish the vector
                        float g[8];
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) g[c8] = __fmul_rn(s[q][c8], p.inv_w);
                        if (SPILL) {
                            st_hint(p.ghat + base + e0, make_float4(g[0], g[1], g[2], g[3]), keep);
                            st_hint(p.ghat + base + e0 + 4, make_float4(g[4], g[5], g[6], g[7]), keep);
                        }
                        acc.add(sumsq8(g));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[st]);
        }
        if (!ok) break;
    }
    // The last n % 8 parameters, one per thread of CTA 0.
    const uint64_t e = nel + threadIdx.x;
    if (blockIdx.x == 0 && threadIdx.x < kVec && e < p.n) {
        const float g = __fmul_rn(rank_sum1(p.grads, nw, e), p.inv_w);
        if (SPILL) p.ghat[e] = g;
        acc.add(__fmul_rn(g, g));
    }

    double a = (double)acc.hi - (double)acc.lo;
    double b = (double)acc.plain;
    consumer_sum2(a, b, sm.red_a, sm.red_b);
    if (threadIdx.x == 0) {
        p.partials[blockIdx.x] = a;
        p.partials[gridDim.x + blockIdx.x] = b;
        __threadfence();
        sm.last = atomicAdd(&p.status->ticket, 1u) == gridDim.x - 1;
    }
    consumer_sync();
    if (!sm.last) return;

    // Last CTA: sum the per-CTA partials in a fixed order (deterministic).
    __threadfence();
    double x = 0.0, y = 0.0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += kConsumers) {
        x += __ldcg(p.partials + i);
        y += __ldcg(p.partials + gridDim.x + i);
    }
    consumer_sum2(x, y, sm.red_a, sm.red_b);
    if (threadIdx.x == 0) {
        if (p.bucket_sums) {            // one bucket of a bucketed step
            p.bucket_sums[2 * p.bucket] = x;
            p.bucket_sums[2 * p.bucket + 1] = y;
        } else {
            float c;
            finish_norm(x, y, p.max_norm, p.clip_eps, p.status, &c);
        }
        p.status->ticket = 0u;
    }
}

// ------------------------------------------------------------------- K2

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// One parameter of the AdamW update, in the order the update is written.
// MV16: the moments are bf16 tensors, so each operation on them rounds its
// fp32 result to bf16.  decay_first: torch.optim.AdamW's order.
template <bool MV16>
__device__ __forceinline__ void adamw1(float gh, float c, const StepScalars &s, bool decay_first, float &master,
                                       float &m, float &v)
{
    const float g = __fmul_rn(gh, c);
    float mi, vi, d;
    if (MV16) {
        mi = bf16_round(__fmul_rn(s.beta1, m));
        mi = bf16_round(__fadd_rn(mi, __fmul_rn(s.omb1, g)));
        vi = bf16_round(__fmul_rn(s.beta2, v));
        vi = bf16_round(__fadd_rn(vi, __fmul_rn(__fmul_rn(s.omb2, g), g)));
        d = bf16_round(__fadd_rn(bf16_round(__fsqrt_rn(vi)), s.eps));
    } else {
        mi = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
        vi = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
        d = __fadd_rn(__fsqrt_rn(vi), s.eps);
    }
    const float u = __fdiv_rn(mi, d);
    float pm = master;
    if (decay_first) {
        pm = __fmul_rn(pm, s.decay);
        pm = __fsub_rn(pm, __fmul_rn(s.step_size, u));
    } else {
        pm = __fsub_rn(pm, __fmul_rn(s.step_size, u));
        pm = __fmul_rn(pm, s.decay);
    }
    master = pm;
    m = mi;
    v = vi;
}

template <int TILE, int STAGES>
struct UpdSmem {
    float in[STAGES][4][TILE];     // 16*TILE bytes per stage: ghat (or the W <= 2 bf16 grads), master, m, v
                                   // (m, v use half their slot when stored in bf16)
    uint16_t b16[STAGES][TILE];    // 2*TILE bytes per stage: the tile's bf16 parameters
    uint64_t full[STAGES], done[STAGES], empty[STAGES];
    int abort;
    float clip;
    StepScalars sc;
};

// Four consecutive parameters at offset o of stage s: AdamW in place on the
// staged master, m, v and the bf16 values into the replica tile.
template <bool REREAD, bool MV16, int TILE, int STAGES>
__device__ __forceinline__ void update4(UpdSmem<TILE, STAGES> &sm, int s, uint32_t o, int nw, float c, const StepScalars &sc,
                                        bool decay_first)
{
    float gh[4];
    if (REREAD) {
        const uint16_t *g = reinterpret_cast<const uint16_t *>(sm.in[s][0]);
        uint2 raw = *reinterpret_cast<const uint2 *>(g + o);
        gh[0] = __uint_as_float(raw.x << 16);
        gh[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        gh[2] = __uint_as_float(raw.y << 16);
        gh[3] = __uint_as_float(raw.y & 0xFFFF0000u);
        for (int r = 1; r < nw; ++r) {
            raw = *reinterpret_cast<const uint2 *>(g + r * TILE + o);
            gh[0] = __fadd_rn(gh[0], __uint_as_float(raw.x << 16));
            gh[1] = __fadd_rn(gh[1], __uint_as_float(raw.x & 0xFFFF0000u));
            gh[2] = __fadd_rn(gh[2], __uint_as_float(raw.y << 16));
            gh[3] = __fadd_rn(gh[3], __uint_as_float(raw.y & 0xFFFF0000u));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) gh[q] = __fmul_rn(gh[q], sc.inv_w);
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(&sm.in[s][0][o]);
        gh[0] = a.x;
        gh[1] = a.y;
        gh[2] = a.z;
        gh[3] = a.w;
    }
    float4 *w4 = reinterpret_cast<float4 *>(&sm.in[s][1][o]);
    float4 w = *w4, m, v;
    if (MV16) {
        const uint2 rm = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(sm.in[s][2]) + o);
        const uint2 rv = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(sm.in[s][3]) + o);
        m = make_float4(__uint_as_float(rm.x << 16), __uint_as_float(rm.x & 0xFFFF0000u),
                        __uint_as_float(rm.y << 16), __uint_as_float(rm.y & 0xFFFF0000u));
        v = make_float4(__uint_as_float(rv.x << 16), __uint_as_float(rv.x & 0xFFFF0000u),
                        __uint_as_float(rv.y << 16), __uint_as_float(rv.y & 0xFFFF0000u));
    } else {
        m = *reinterpret_cast<const float4 *>(&sm.in[s][2][o]);
        v = *reinterpret_cast<const float4 *>(&sm.in[s][3][o]);
    }
    adamw1<MV16>(gh[0], c, sc, decay_first, w.x, m.x, v.x);
    adamw1<MV16>(gh[1], c, sc, decay_first, w.y, m.y, v.y);
    adamw1<MV16>(gh[2], c, sc, decay_first, w.z, m.z, v.z);
    adamw1<MV16>(gh[3], c, sc, decay_first, w.w, m.w, v.w);
    *w4 = w;
    if (MV16) {   // the values are bf16 already: the packing is exact
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(sm.in[s][2]) + o) =
            make_uint2(pack2(m.x, m.y), pack2(m.z, m.w));
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(sm.in[s][3]) + o) =
            make_uint2(pack2(v.x, v.y), pack2(v.z, v.w));
    } else {
        *reinterpret_cast<float4 *>(&sm.in[s][2][o]) = m;
        *reinterpret_cast<float4 *>(&sm.in[s][3][o]) = v;
    }
    *reinterpret_cast<uint2 *>(&sm.b16[s][o]) = make_uint2(pack2(w.x, w.y), pack2(w.z, w.w));
}

// Warps 0..7 consume, warp 8 produces, warp 9 stores.  Tiles are walked
// from the highest down (the reduce-scatter kernel wrote those last, so
// they are the likeliest to still be in L2).  master, m, v are updated in
// place in the stage and written back from there.
template <int W, int CAP, bool REREAD, bool MV16, int TILE, int STAGES, int CWARPS, bool RUNS>
__global__ void __launch_bounds__(CWARPS * 32 + 64, 1)
zero1_adamw_ag_kernel(const __grid_constant__ UpdParams<CAP> p)
{
    constexpr uint32_t kMomBytes = MV16 ? 2u : 4u;   // bytes per stored moment
    constexpr int kUpdTile = TILE;
    constexpr int kUpdStages = STAGES;
    constexpr int kUpdConsumerWarps = CWARPS;
    constexpr int kUpdConsumers = CWARPS * 32;
    constexpr int kUpdQuads = kUpdTile / (4 * kUpdConsumers);   // 4-parameter groups per consumer thread per tile
    static_assert(kUpdQuads >= 1 && kUpdQuads * 4 * kUpdConsumers == kUpdTile, "update consumers must tile kUpdTile");
    static_assert(kUpdTile / 32 <= kUpdConsumers, "one discarded scratch line per consumer thread");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    UpdSmem<TILE, STAGES> &sm = *reinterpret_cast<UpdSmem<TILE, STAGES> *>(smem_raw);
    const int nw = W > 0 ? W : p.world;
    const uint64_t nel = p.nvec * kVec;
    const int64_t ntiles = (int64_t)((nel + kUpdTile - 1) / kUpdTile);
    // This CTA's tiles, k = 0 .. ncta-1, highest first: one contiguous run
    // (RUNS), or every gridDim.x-th tile.
    const int64_t run_hi = RUNS ? (int64_t)(((uint64_t)blockIdx.x + 1) * (uint64_t)ntiles / gridDim.x)
                                : ntiles - 1 - (int64_t)blockIdx.x;
    const int64_t run_lo = (int64_t)((uint64_t)blockIdx.x * (uint64_t)ntiles / gridDim.x);
    const uint32_t ncta = RUNS ? (uint32_t)(run_hi - run_lo)
                               : (run_hi >= 0 ? (uint32_t)(run_hi / gridDim.x + 1) : 0u);
    auto tile_at = [&](uint32_t k) -> int64_t {
        return RUNS ? run_hi - 1 - (int64_t)k : run_hi - (int64_t)k * gridDim.x;
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort = &sm.abort;

    // Programmatic dependency on the reduce-scatter kernel: the next step's
    // kernel may launch now; ĝ and the clip coefficient are read only after
    // the reduce-scatter grid has completed.
    launch_dependents();
    grid_dependency_wait();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kUpdStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.done[s], kUpdConsumerWarps);
            mbar_init(&sm.empty[s], 1);
        }
        sm.abort = 0;
        if (p.bucket_sums) {
            // Bucketed step: every CTA forms c from the buckets' sums in
            // call order (the same value everywhere); CTA 0 records it.
            double x = 0.0, y = 0.0;
            for (int b = 0; b < p.nbuckets; ++b) {
                x += p.bucket_sums[2 * b];
                y += p.bucket_sums[2 * b + 1];
            }
            finish_norm(x, y, p.max_norm, p.clip_eps, blockIdx.x == 0 ? p.status : nullptr, &sm.clip);
        } else {
            sm.clip = p.status->clip;
        }
        if (p.dev.bc) {
            // Capturable: this step is t + 1.  The CTA that counts in last
            // (every CTA has read t by then) advances the counter, unless
            // later launches of the same step (a step cut into pieces)
            // still have to read it.
            const unsigned long long t = p.status->t + 1;
            sm.sc = form_scalars(p.sc, p.dev, t);
            __threadfence();
            if (atomicAdd(&p.status->ticket2, 1u) == gridDim.x - 1) {
                if (p.advance_t) p.status->t = t;
                p.status->ticket2 = 0u;
            }
        } else {
            sm.sc = p.sc;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Every byte this kernel moves is touched once per step: lowest L2 priority.
    const uint64_t once = policy_evict_first();

    if (warp == kUpdConsumerWarps) {                              // producer
        if (lane == 0 && !p.stall_test) {
            uint32_t k = 0;
            for (; k < ncta && !*abort; ++k) {
                const int64_t j = tile_at(k);
                const int s = k % kUpdStages;
                if (k >= kUpdStages && !mbar_wait(&sm.empty[s], ((k / kUpdStages) & 1u) ^ 1u, abort, &p.status->errors)) break;
                if (p.load_period_ns && k >= kUpdStages) {
                    // Load phasing: once the ring is primed, a tile's loads go
                    // out only at the next boundary of a period shared by every
                    // SM (the global nanosecond clock), so the whole grid's
                    // loads reach DRAM together rather than one by one among
                    // the stores.  The boundary is at most one period away;
                    // the iteration cap only guards against a stopped clock.
                    const unsigned long long next = (global_ns() / p.load_period_ns + 1) * p.load_period_ns;
                    for (uint32_t it = 0; global_ns() < next && it < (1u << 20); ++it) {
                    }
                }
                const uint64_t base = (uint64_t)j * kUpdTile;
                const uint32_t cnt = (uint32_t)(nel - base < (uint64_t)kUpdTile ? nel - base : kUpdTile);
                const uint32_t gbytes = REREAD ? (uint32_t)nw * cnt * 2u : cnt * 4u;
                mbar_arrive_expect_tx(&sm.full[s], gbytes + 4u * cnt + 2u * kMomBytes * cnt);
                if (REREAD) {
                    uint16_t *g = reinterpret_cast<uint16_t *>(sm.in[s][0]);
                    for (int r = 0; r < nw; ++r)
                        tma_load_hint(g + r * kUpdTile, p.grads[r] + base, cnt * 2u, &sm.full[s], once);
                }
                tma_load_hint(sm.in[s][1], p.master + base, cnt * 4u, &sm.full[s], once);
                tma_load_hint(sm.in[s][2], static_cast<const unsigned char *>(p.m) + base * kMomBytes,
                              cnt * kMomBytes, &sm.full[s], once);
                tma_load_hint(sm.in[s][3], static_cast<const unsigned char *>(p.v) + base * kMomBytes,
                              cnt * kMomBytes, &sm.full[s], once);
                // ĝ last: master, m, v come from DRAM, while the ĝ written last by
                // the reduce-scatter kernel is partly still in L2, so the
                // misses start first (measured 0.2% faster on gpt2_small).
                if (!REREAD) tma_load_hint(sm.in[s][0], p.ghat + base, cnt * 4u, &sm.full[s], once);
            }
            if (*abort) drain_loads<kUpdStages>(sm.full, k);
        }
        return;
    }

    if (warp == kUpdConsumerWarps + 1) {                          // stores
        uint32_t k = 0;
        for (; k < ncta; ++k) {
            const int64_t j = tile_at(k);
            const int s = k % kUpdStages;
            const bool got = mbar_wait(&sm.done[s], (k / kUpdStages) & 1u, abort, &p.status->errors);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            const uint64_t base = (uint64_t)j * kUpdTile;
            const uint32_t cnt = (uint32_t)(nel - base < (uint64_t)kUpdTile ? nel - base : kUpdTile);
            // Targets 0..2 are master, m, v; 3.. are the W replicas (the
            // all-gather).  Lane L issues targets L, L+32, ...
            for (int t = lane; t < nw + 3; t += 32) {
                if (t == 0) {
                    tma_store_hint(p.master + base, sm.in[s][1], cnt * 4u, once);
                } else if (t < 3) {
                    unsigned char *dst = static_cast<unsigned char *>(t == 1 ? p.m : p.v);
                    tma_store_hint(dst + base * kMomBytes, sm.in[s][1 + t], cnt * kMomBytes, once);
                } else {
                    tma_store_hint(p.params[t - 3] + base, sm.b16[s], cnt * 2u, once);
                }
            }
            tma_commit();
            if (k >= 1) {                      // the previous tile's stores have read its stage
                tma_wait_read<1>();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[(k - 1) % kUpdStages]);
            }
        }
        tma_wait_all();
        return;
    }

    // Consumers: thread t owns parameters [4t + 4qC, 4t + 4qC + 4) of every
    // tile (C consumer threads, q < kUpdQuads), so a warp's 16-byte
    // shared-memory accesses are consecutive (no bank conflicts).
    const float c = sm.clip;
    const StepScalars sc = sm.sc;
    // Discards act on whole 128-byte L2 lines, so only when ĝ starts on a
    // line: a bucket that begins mid-line (a multiple of 8 parameters, not
    // of 32) must not drop its neighbour's unread values.
    const bool discard = !REREAD && (reinterpret_cast<uintptr_t>(p.ghat) & 127u) == 0;
    for (uint32_t k = 0; k < ncta; ++k) {
        const int64_t j = tile_at(k);
        const int s = k % kUpdStages;
        const bool got = mbar_wait(&sm.full[s], (k / kUpdStages) & 1u, abort, &p.status->errors);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        const uint64_t base = (uint64_t)j * kUpdTile;
        const uint32_t cnt = (uint32_t)(nel - base < (uint64_t)kUpdTile ? nel - base : kUpdTile);
        if (discard && threadIdx.x < cnt / 32u) {
            // This tile's ĝ is in shared memory now and dead in HBM: drop its
            // whole 128-byte lines from L2 unwritten (a partly covered last
            // line may hold the n % 8 tail and is left alone).
            discard_l2_line(p.ghat + base + threadIdx.x * 32u);
        }
#pragma unroll
        for (int q = 0; q < kUpdQuads; ++q) {
            const uint32_t o = threadIdx.x * 4u + (uint32_t)q * 4u * kUpdConsumers;
            if (o < cnt) update4<REREAD, MV16, TILE, STAGES>(sm, s, o, nw, c, sc, p.decay_first != 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.done[s]);
    }

    // The last n % 8 parameters, one per thread of CTA 0, straight from HBM.
    const uint64_t e = nel + threadIdx.x;
    if (blockIdx.x == 0 && threadIdx.x < kVec && e < p.n) {
        const float gh = REREAD ? __fmul_rn(rank_sum1(p.grads, nw, e), p.sc.inv_w) : p.ghat[e];
        float w = p.master[e], m, v;
        if (MV16) {
            m = __uint_as_float((unsigned)static_cast<const uint16_t *>(p.m)[e] << 16);
            v = __uint_as_float((unsigned)static_cast<const uint16_t *>(p.v)[e] << 16);
        } else {
            m = static_cast<const float *>(p.m)[e];
            v = static_cast<const float *>(p.v)[e];
        }
        adamw1<MV16>(gh, c, sc, p.decay_first != 0, w, m, v);
        p.master[e] = w;
        if (MV16) {
            static_cast<__nv_bfloat16 *>(p.m)[e] = __float2bfloat16_rn(m);
            static_cast<__nv_bfloat16 *>(p.v)[e] = __float2bfloat16_rn(v);
        } else {
            static_cast<float *>(p.m)[e] = m;
            static_cast<float *>(p.v)[e] = v;
        }
        const __nv_bfloat16 bw = __float2bfloat16_rn(w);
        for (int r = 0; r < nw; ++r) reinterpret_cast<__nv_bfloat16 *>(p.params[r])[e] = bw;
    }
}

// ------------------------------------------------------------------- K0

// Small steps: the whole step in one launch of one thread-block cluster.
// Each thread owns up to VPT 8-parameter vectors (vector i of thread g of
// the cluster is g + i * kSmallCtas * kSmallThreads, threads numbered with
// the warps interleaved over the CTAs).  It loads their master, m, v and
// their W gradients (in batches of loads issued before any add), forms the
// rank-ordered mean and its squares, and keeps both in registers.  Each
// CTA pushes its fixed-order partial sums into every CTA's shared memory
// (distributed shared memory), one cluster barrier makes them visible,
// every CTA adds the kSmallCtas partials in rank order (so all form the
// same c), and each thread then updates its vectors and stores master, m,
// v and the W replicas.  The cluster barriers are hardware barriers that
// every thread reaches: nothing returns early.
template <int CAP>
struct SmallParams {
    const uint16_t *grads[CAP];
    uint16_t *params[CAP];
    float *master;
    void *m, *v;
    DevStatus *status;
    uint64_t nvec, n;
    int world;
    int decay_first;
    StepScalars sc;
    double max_norm, clip_eps;
    DevScalars dev;
};

template <bool MV16>
__device__ __forceinline__ void load_moment8(float out[8], const void *base, uint64_t e)
{
    if (MV16) {
        set_widened(out, *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + e));
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e);
        const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e + 4);
        out[0] = a.x, out[1] = a.y, out[2] = a.z, out[3] = a.w;
        out[4] = b.x, out[5] = b.y, out[6] = b.z, out[7] = b.w;
    }
}

template <bool MV16>
__device__ __forceinline__ void store_moment8(void *base, uint64_t e, const float x[8])
{
    if (MV16) {   // the values are bf16 already: the packing is exact
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + e) =
            make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
    } else {
        float *f = static_cast<float *>(base) + e;
        *reinterpret_cast<float4 *>(f) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4 *>(f + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
}

template <int W, int CAP, int CTAS, int THREADS, int VPT, bool MV16>
__global__ void __launch_bounds__(THREADS, 1)
zero1_small_step_kernel(const __grid_constant__ SmallParams<CAP> p)
{
    constexpr int kWarps = THREADS / 32;
    constexpr uint32_t kStride = CTAS * THREADS;
    __shared__ double red_a[kWarps], red_b[kWarps];
    __shared__ double part[2 * CTAS];      // (sum, plain sum) of every CTA, in cluster rank order
    __shared__ float clip;
    __shared__ StepScalars ssc;
    const int nw = W > 0 ? W : p.world;
    const uint64_t nel = p.nvec * kVec;
    // Warps are dealt round-robin over the CTAs (warp i of CTA b is global
    // warp i * CTAS + b), so even a few vectors' worth of work spreads over
    // every SM of the cluster; each warp still covers 32 consecutive vectors.
    const uint32_t gt = ((threadIdx.x >> 5) * CTAS + blockIdx.x) * 32u + (threadIdx.x & 31u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Every CTA of the cluster must have started before any thread writes
    // into another CTA's shared memory: arrive now, wait just before the
    // pushes below (by then the wait is free).
    cluster_arrive_relaxed();
    // Capturable: this step is t + 1; every CTA reads t here, before the
    // cluster barrier, and CTA 0 advances it after it.
    const unsigned long long tnext = p.dev.bc ? p.status->t + 1 : 0ull;
    if (threadIdx.x == 0) ssc = p.dev.bc ? form_scalars(p.sc, p.dev, tnext) : p.sc;

    float gh[VPT][8], w[VPT][8], m[VPT][8], v[VPT][8];
    uint64_t ev[VPT];
    bool has[VPT];
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        ev[q] = (uint64_t)(gt + q * kStride) * kVec;
        has[q] = ev[q] < nel;
        if (has[q]) {              // state first: in flight while the gradients are summed
            load_moment8<false>(w[q], p.master, ev[q]);
            load_moment8<MV16>(m[q], p.m, ev[q]);
            load_moment8<MV16>(v[q], p.v, ev[q]);
        }
    }
    // Rank-ordered sum.  The gradient loads go out in batches (8 16-byte
    // loads per thread) before the adds consume them, so a batch costs one
    // memory latency rather than one per rank.
    constexpr int kBatch = 8 / VPT;
    for (int r0 = 0; r0 < nw; r0 += kBatch) {
        uint4 buf[kBatch][VPT];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
            for (int q = 0; q < VPT; ++q)
                if (r0 + k < nw && has[q]) buf[k][q] = __ldg(reinterpret_cast<const uint4 *>(p.grads[r0 + k] + ev[q]));
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
            for (int q = 0; q < VPT; ++q)
                if (r0 + k < nw && has[q]) {
                    if (r0 + k == 0)
                        set_widened(gh[q], buf[k][q]);
                    else
                        add_widened(gh[q], buf[k][q]);
                }
    }
    Kahan acc;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        if (has[q]) {
#pragma unroll
            for (int k = 0; k < 8; ++k) gh[q][k] = __fmul_rn(gh[q][k], p.sc.inv_w);
            acc.add(sumsq8(gh[q]));
        }
    }
    // The last n % 8 parameters, one per thread of CTA 0.
    const uint64_t et = nel + threadIdx.x;
    const bool tail = blockIdx.x == 0 && threadIdx.x < kVec && et < p.n;
    float tg = 0.f, tw = 0.f, tm = 0.f, tv = 0.f;
    if (tail) {
        tg = __fmul_rn(rank_sum1(p.grads, nw, et), p.sc.inv_w);
        acc.add(__fmul_rn(tg, tg));
        tw = p.master[et];
        if (MV16) {
            tm = __uint_as_float((unsigned)static_cast<const uint16_t *>(p.m)[et] << 16);
            tv = __uint_as_float((unsigned)static_cast<const uint16_t *>(p.v)[et] << 16);
        } else {
            tm = static_cast<const float *>(p.m)[et];
            tv = static_cast<const float *>(p.v)[et];
        }
    }

    // CTA partials in a fixed order: warp shuffle tree, then warp 0.
    double a = (double)acc.hi - (double)acc.lo;
    double b = (double)acc.plain;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_down_sync(0xFFFFFFFFu, a, off);
        b += __shfl_down_sync(0xFFFFFFFFu, b, off);
    }
    if (lane == 0) {
        red_a[warp] = a;
        red_b[warp] = b;
    }
    __syncthreads();
    cluster_wait();            // every CTA has started (the arrive at the top)
    if (threadIdx.x == 0) {
        double x = 0.0, y = 0.0;
        for (int i = 0; i < kWarps; ++i) {
            x += red_a[i];
            y += red_b[i];
        }
        // Push this CTA's pair into slot blockIdx.x (its cluster rank) of
        // every CTA's table, this CTA's own included.
        for (uint32_t r = 0; r < (uint32_t)CTAS; ++r) {
            st_cluster_f64(&part[2 * blockIdx.x], r, x);
            st_cluster_f64(&part[2 * blockIdx.x + 1], r, y);
        }
    }
    static_assert(CTAS > 1 && CTAS <= 32, "a cluster of 2..32 CTAs");
    // The pushes (released before this barrier) are visible after it, and
    // no CTA touches another's shared memory afterwards, so a CTA may finish
    // while the others still work.
    cluster_sync();
    if (threadIdx.x == 0) {
        double x = 0.0, y = 0.0;
        for (int r = 0; r < CTAS; ++r) {       // rank order: every CTA forms the same c
            x += part[2 * r];
            y += part[2 * r + 1];
        }
        float c;
        finish_norm(x, y, p.max_norm, p.clip_eps, blockIdx.x == 0 ? p.status : nullptr, &c);
        clip = c;
    }
    __syncthreads();
    const float c = clip;
    const StepScalars sc = ssc;
    const bool decay_first = p.decay_first != 0;
    if (p.dev.bc && blockIdx.x == 0 && threadIdx.x == 0) p.status->t = tnext;

#pragma unroll
    for (int q = 0; q < VPT; ++q) {
        const uint64_t e = (uint64_t)(gt + q * kStride) * kVec;
        if (e < nel) {
#pragma unroll
            for (int k = 0; k < 8; ++k) adamw1<MV16>(gh[q][k], c, sc, decay_first, w[q][k], m[q][k], v[q][k]);
            store_moment8<false>(p.master, e, w[q]);
            store_moment8<MV16>(p.m, e, m[q]);
            store_moment8<MV16>(p.v, e, v[q]);
            const uint4 bw = make_uint4(pack2(w[q][0], w[q][1]), pack2(w[q][2], w[q][3]), pack2(w[q][4], w[q][5]),
                                        pack2(w[q][6], w[q][7]));
            for (int r = 0; r < nw; ++r) *reinterpret_cast<uint4 *>(p.params[r] + e) = bw;
        }
    }
    if (tail) {
        adamw1<MV16>(tg, c, sc, decay_first, tw, tm, tv);
        p.master[et] = tw;
        if (MV16) {
            static_cast<__nv_bfloat16 *>(p.m)[et] = __float2bfloat16_rn(tm);
            static_cast<__nv_bfloat16 *>(p.v)[et] = __float2bfloat16_rn(tv);
        } else {
            static_cast<float *>(p.m)[et] = tm;
            static_cast<float *>(p.v)[et] = tv;
        }
        const __nv_bfloat16 bw = __float2bfloat16_rn(tw);
        for (int r = 0; r < nw; ++r) reinterpret_cast<__nv_bfloat16 *>(p.params[r])[et] = bw;
    }
}

// ------------------------------------------------------------- launchers

template <typename Kernel>
cudaError_t allow_smem(Kernel kernel, size_t bytes)
{
    return allow_dynamic_smem(reinterpret_cast<const void *>(kernel), (int)bytes);
}

template <int W, int CAP, int CTAS, int THREADS, int VPT, bool MV16>
cudaError_t launch_small_v(const StepLaunch &s, cudaStream_t stream)
{
    SmallParams<CAP> sp{};
    for (int r = 0; r < s.world; ++r) {
        sp.grads[r] = static_cast<const uint16_t *>(s.grads[r]);
        sp.params[r] = static_cast<uint16_t *>(s.params[r]);
    }
    sp.master = s.master;
    sp.m = s.m;
    sp.v = s.v;
    sp.status = s.status;
    sp.nvec = s.n / kVec;
    sp.n = s.n;
    sp.world = s.world;
    sp.decay_first = s.decay_first ? 1 : 0;
    sp.sc = s.sc;
    sp.max_norm = s.max_norm;
    sp.clip_eps = s.clip_eps;
    sp.dev = s.dev;
    // One thread-block cluster of CTAS CTAs (distributed shared memory and
    // the cluster barrier need them co-scheduled).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CTAS, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CTAS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = zero1_small_step_kernel<W, CAP, CTAS, THREADS, VPT, MV16>;
    if (CTAS > 8) {   // past the portable cluster size
        cudaError_t e = set_func_attribute_once(reinterpret_cast<const void *>(kern),
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kern, sp);
}

template <int W, int CAP>
cudaError_t launch_small(const StepLaunch &s, cudaStream_t stream)
{
    constexpr int C = kSmallCtas, T = kSmallThreads;
    switch (s.small_vpt * 2 + (s.moments_bf16 ? 1 : 0)) {
    case 2: return launch_small_v<W, CAP, C, T, 1, false>(s, stream);
    case 3: return launch_small_v<W, CAP, C, T, 1, true>(s, stream);
    case 4: return launch_small_v<W, CAP, C, T, 2, false>(s, stream);
    case 5: return launch_small_v<W, CAP, C, T, 2, true>(s, stream);
    case 8: return launch_small_v<W, CAP, C, T, 4, false>(s, stream);
    case 9: return launch_small_v<W, CAP, C, T, 4, true>(s, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int W, int CAP>
cudaError_t launch_w(const StepLaunch &s, cudaStream_t stream, cudaEvent_t *ev)
{
    cudaError_t e;
    if (s.small_vpt > 0 && s.phase == 0 && !s.bucket_sums) {
        // One launch; the profile's second interval is empty.
        if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
        if ((e = launch_small<0, CAP>(s, stream)) != cudaSuccess) return e;   // runtime W: latency-bound anyway
        if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
        if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;
        return cudaSuccess;
    }
    RsParams<CAP> rp{};
    UpdParams<CAP> up{};
    for (int r = 0; r < s.world; ++r) {
        rp.grads[r] = s.grads ? static_cast<const uint16_t *>(s.grads[r]) : nullptr;
        up.grads[r] = s.grads ? static_cast<const uint16_t *>(s.grads[r]) : nullptr;
        up.params[r] = s.params ? static_cast<uint16_t *>(s.params[r]) : nullptr;
    }
    rp.ghat = s.ghat;
    rp.partials = s.partials;
    rp.status = s.status;
    rp.nvec = s.n / kVec;
    rp.n = s.n;
    rp.world = s.world;
    rp.inv_w = s.sc.inv_w;
    rp.max_norm = s.max_norm;
    rp.clip_eps = s.clip_eps;
    rp.bucket_sums = s.bucket_sums;
    rp.bucket = s.bucket_index;

    up.ghat = s.ghat;
    up.master = s.master;
    up.m = s.m;
    up.v = s.v;
    up.status = s.status;
    up.nvec = s.n / kVec;
    up.n = s.n;
    up.world = s.world;
    up.sc = s.sc;
    up.decay_first = s.decay_first ? 1 : 0;
    up.bucket_sums = s.bucket_sums;
    up.nbuckets = s.nbuckets;
    up.max_norm = s.max_norm;
    up.clip_eps = s.clip_eps;
    up.dev = s.dev;
    up.advance_t = s.advance_t ? 1 : 0;
    up.stall_test = s.stall_test ? 1 : 0;

    const bool spill = s.ghat != nullptr;
    if (!spill && s.world > 2) return cudaErrorInvalidValue;   // the re-read stage holds two ranks
    auto k1 = spill ? zero1_rs_norm_kernel<W, CAP, true> : zero1_rs_norm_kernel<W, CAP, false>;
    constexpr UpdConfig U1 = kUpdSpillF32, U2 = kUpdSpillBf16, U0 = kUpdReread;
    constexpr int C1 = U1.warps, C2 = U2.warps, C0 = U0.warps;
    const size_t k1_smem = spill ? sizeof(RsSmem<kRsSpill.tile, kRsSpill.ranks, kRsSpill.stages>)
                                 : sizeof(RsSmem<kRsRead.tile, kRsRead.ranks, kRsRead.stages>);
    if ((e = allow_smem(k1, k1_smem)) != cudaSuccess) return e;
    const int path = spill ? (s.moments_bf16 ? 2 : 1) : 0;
    auto k2 = path == 1   ? zero1_adamw_ag_kernel<W, CAP, false, false, U1.tile, U1.stages, C1, U1.runs>
              : path == 2 ? zero1_adamw_ag_kernel<W, CAP, false, true, U2.tile, U2.stages, C2, U2.runs>
                          : (s.moments_bf16 ? zero1_adamw_ag_kernel<W, CAP, true, true, U0.tile, U0.stages, C0, U0.runs>
                                            : zero1_adamw_ag_kernel<W, CAP, true, false, U0.tile, U0.stages, C0, U0.runs>);
    const size_t k2_smem = path == 1   ? sizeof(UpdSmem<U1.tile, U1.stages>)
                           : path == 2 ? sizeof(UpdSmem<U2.tile, U2.stages>)
                                       : sizeof(UpdSmem<U0.tile, U0.stages>);
    const int k2_threads = (path == 1 ? C1 : path == 2 ? C2 : C0) * 32 + 64;
    if ((e = allow_smem(k2, k2_smem)) != cudaSuccess) return e;
    // Load phasing (fp32 moments; the scratch path or the gradient re-read
    // path): the period is the time one tile's bytes per CTA take when the
    // whole grid moves them at the given device-wide rate (bytes / (GB/s) =
    // ns).  A tile moves 28 + 2W bytes per parameter on the scratch path
    // (ĝ, master, m, v in; master, m, v, W replicas out) and 24 + 4W on the
    // re-read path (W gradients in instead of ĝ).
    if (path != 2 && s.load_rate_gbs > 0.0) {
        const double tile_bytes = path == 1 ? (28.0 + 2.0 * s.world) * U1.tile : (24.0 + 4.0 * s.world) * U0.tile;
        up.load_period_ns = (unsigned long long)(tile_bytes * s.grid_update / s.load_rate_gbs + 0.5);
    }
    // A whole step without profiling events between its kernels launches
    // both with a programmatic dependency on the kernel before them in the
    // stream: each may launch while its predecessor drains and waits for it
    // in grid_dependency_wait before touching memory.
    const bool pdl = ZERO1_PDL && !ev && s.phase == 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c1 = {};
    c1.gridDim = dim3(s.grid_rs);
    c1.blockDim = dim3(kRsThreads);
    c1.dynamicSmemBytes = k1_smem;
    c1.stream = stream;
    c1.attrs = attr;
    c1.numAttrs = pdl ? 1 : 0;
    cudaLaunchConfig_t c2 = c1;
    c2.gridDim = dim3(s.grid_update);
    c2.blockDim = dim3(k2_threads);
    c2.dynamicSmemBytes = k2_smem;
    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    if (s.phase != 2 && (e = cudaLaunchKernelEx(&c1, k1, rp)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
    if (s.phase != 1 && (e = cudaLaunchKernelEx(&c2, k2, up)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_step(const StepLaunch &s, cudaStream_t stream, cudaEvent_t *ev)
{
    switch (s.world) {
    case 1: return launch_w<1, 8>(s, stream, ev);
    case 2: return launch_w<2, 8>(s, stream, ev);
    case 4: return launch_w<4, 8>(s, stream, ev);
    case 8: return launch_w<8, 8>(s, stream, ev);
    case 16: return launch_w<16, 64>(s, stream, ev);
    case 32: return launch_w<32, 64>(s, stream, ev);
    case 64: return launch_w<64, 64>(s, stream, ev);
    default: break;
    }
    if (s.world <= 8) return launch_w<0, 8>(s, stream, ev);
    if (s.world <= 64) return launch_w<0, 64>(s, stream, ev);
    return launch_w<0, 512>(s, stream, ev);
}

void plan_grids(uint64_t n, bool reread, int num_sms, int *grid_rs, int *grid_update)
{
    // Persistent kernels: one CTA per SM (each holds ~130-220 KB of shared
    // memory), never more CTAs than tiles, at least one (the n % 8 tail).
    // The update kernel's tile depends on its path (re-read or scratch).
    const uint64_t rs_tile = (uint64_t)(reread ? kRsRead.tile : kRsSpill.tile);
    const uint64_t ntiles = (n / kVec * kVec + rs_tile - 1) / rs_tile;
    uint64_t g = (uint64_t)num_sms;
    if (ntiles < g) g = ntiles;
    if (g < 1) g = 1;
    *grid_rs = (int)g;
    const uint64_t upd_tile = (uint64_t)(reread ? kUpdReread.tile : kUpdSpillF32.tile);
    static_assert(kUpdSpillF32.tile == kUpdSpillBf16.tile, "the scratch paths share one tile size");
    const uint64_t ntiles_upd = (n / kVec * kVec + upd_tile - 1) / upd_tile;
    uint64_t gu = (uint64_t)num_sms;
    if (ntiles_upd < gu) gu = ntiles_upd;
    if (gu < 1) gu = 1;
    *grid_update = (int)gu;
}

}  // namespace zero1
