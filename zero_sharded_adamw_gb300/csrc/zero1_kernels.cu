// zero1_kernels.cu -- the two sm_103a kernels of one ZeRO-1 step.
//
//  K1  zero1_rs_norm_kernel   reduce-scatter (rank-ordered fp32 sum of the W
//                             bf16 gradients, times 1/W) fused with the
//                             squared L2 norm: per-thread compensated fp32,
//                             warp shuffles, one fp64 grid pass by the last
//                             CTA, which also forms the clip coefficient.
//  K2  zero1_adamw_ag_kernel  clip scale + AdamW on fp32 master/m/v + bf16
//                             cast + all-gather (W-way store of each vector).
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
// Both kernels are HBM-bound streams (no contraction, so no tensor cores).
// Every fp32 operation of the sum and the update is an explicit _rn
// intrinsic: no FMA contraction, IEEE round-to-nearest-even, no FTZ, so the
// results are those of the plain fp32 definition bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zero1_internal.h"

namespace zero1 {
namespace {

// ------------------------------------------------------------ memory ops

// 16-byte read-only streaming load: no L1 allocation (each byte is read once
// per kernel).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ float4 ld_stream_f4(const float4 *p)
{
    float4 r;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p));
    return r;
}

// Read-write state: plain 16-byte load (the kernel writes the same address).
__device__ __forceinline__ float4 ld_f4(const float4 *p) { return *p; }

// ------------------------------------------------------------ bf16 pack

// bf16 -> fp32 widening is exact: the bf16 bits are the top half.
__device__ __forceinline__ void add_widened(float s[8], uint4 raw)
{
    const unsigned w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        s[2 * k] = __fadd_rn(s[2 * k], __uint_as_float(w[k] << 16));
        s[2 * k + 1] = __fadd_rn(s[2 * k + 1], __uint_as_float(w[k] & 0xFFFF0000u));
    }
}

__device__ __forceinline__ void set_widened(float s[8], uint4 raw)
{
    const unsigned w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        s[2 * k] = __uint_as_float(w[k] << 16);
        s[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ unsigned pack2(float lo, float hi)
{
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // .x (lo) -> low 16 bits
    return *reinterpret_cast<unsigned *>(&b);
}

// --------------------------------------------------------- kernel params

// Pointer tables live in the launch parameters (CAP slots, W used).
template <int CAP>
struct RsParams {
    const uint4 *grads[CAP];
    float4 *ghat;             // nullptr: norm only
    double *partials;         // [2 * gridDim.x]
    DevStatus *status;
    uint64_t nvec;            // n / 8
    uint64_t n;
    int world;
    float inv_w;
    double max_norm;
};

template <int CAP>
struct UpdParams {
    const uint4 *grads[CAP];  // re-read mode only
    uint4 *params[CAP];
    const float4 *ghat;       // spill mode only
    float4 *master, *m, *v;
    const DevStatus *status;
    uint64_t nvec, n;
    int world;
    StepScalars sc;
};

// ------------------------------------------------- rank-ordered sum of 8

// s[k] = ((g_0 + g_1) + g_2) + ... + g_{W-1} for the 8 parameters of vector
// `vec`, in fp32.  W > 0: compile-time world size; W == 0: `world` at run
// time.  Ranks are loaded in groups of 8 so that a group's loads are all in
// flight together; the sum itself stays strictly in rank order.
template <int W>
__device__ __forceinline__ void rank_sum8(const uint4 *const *grads, int world, uint64_t vec, float s[8])
{
    constexpr int G = 8;
    const int nw = W > 0 ? W : world;
    {
        uint4 raw[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            if (j < nw) raw[j] = ld_stream(grads[j] + vec);
        set_widened(s, raw[0]);
#pragma unroll
        for (int j = 1; j < G; ++j)
            if (j < nw) add_widened(s, raw[j]);
    }
#pragma unroll 1
    for (int r0 = G; r0 < nw; r0 += G) {
        uint4 raw[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            if (r0 + j < nw) raw[j] = ld_stream(grads[r0 + j] + vec);
#pragma unroll
        for (int j = 0; j < G; ++j)
            if (r0 + j < nw) add_widened(s, raw[j]);
    }
}

// Scalar version for the last n % 8 parameters.
__device__ __forceinline__ float rank_sum1(const uint4 *const *grads, int world, uint64_t e)
{
    const unsigned short *g0 = reinterpret_cast<const unsigned short *>(grads[0]);
    float s = __uint_as_float((unsigned)g0[e] << 16);
    for (int r = 1; r < world; ++r) {
        const unsigned short *gr = reinterpret_cast<const unsigned short *>(grads[r]);
        s = __fadd_rn(s, __uint_as_float((unsigned)gr[e] << 16));
    }
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

// Fixed-order block sum of two doubles (warp shuffle tree, then warp 0).
__device__ __forceinline__ void block_sum2(double &a, double &b)
{
    __shared__ double sa[kThreads / 32], sb[kThreads / 32];
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
    __syncthreads();
    if (warp == 0) {
        a = lane < kThreads / 32 ? sa[lane] : 0.0;
        b = lane < kThreads / 32 ? sb[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_down_sync(0xFFFFFFFFu, a, off);
            b += __shfl_down_sync(0xFFFFFFFFu, b, off);
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------- K1

template <int W, int CAP, bool SPILL>
__global__ void __launch_bounds__(kThreads)
zero1_rs_norm_kernel(const __grid_constant__ RsParams<CAP> p)
{
    Kahan acc;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    for (uint64_t vec = tid; vec < p.nvec; vec += stride) {
        float s[8];
        rank_sum8<W>(p.grads, p.world, vec, s);
        float g[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) g[k] = __fmul_rn(s[k], p.inv_w);
        if (SPILL) {
            p.ghat[2 * vec] = make_float4(g[0], g[1], g[2], g[3]);
            p.ghat[2 * vec + 1] = make_float4(g[4], g[5], g[6], g[7]);
        }
        acc.add(sumsq8(g));
    }
    // The last n % 8 parameters, one per thread of the first CTA.
    const uint64_t e = p.nvec * kVec + tid;
    if (tid < kVec && e < p.n) {
        float g = __fmul_rn(rank_sum1(p.grads, p.world, e), p.inv_w);
        if (SPILL) reinterpret_cast<float *>(p.ghat)[e] = g;
        acc.add(__fmul_rn(g, g));
    }

    double a = (double)acc.hi - (double)acc.lo;
    double b = (double)acc.plain;
    block_sum2(a, b);

    __shared__ bool last;
    if (threadIdx.x == 0) {
        p.partials[blockIdx.x] = a;
        p.partials[gridDim.x + blockIdx.x] = b;
        __threadfence();
        last = atomicAdd(&p.status->ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;

    // Last CTA: sum the per-CTA partials in a fixed order (deterministic).
    __threadfence();
    double x = 0.0, y = 0.0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += kThreads) {
        x += __ldcg(p.partials + i);
        y += __ldcg(p.partials + gridDim.x + i);
    }
    block_sum2(x, y);
    if (threadIdx.x == 0) {
        const double nsq = isfinite(y) ? x : y;
        const double norm = sqrt(nsq);
        float c = 1.0f;
        if (p.max_norm > 0.0) {
            if (isnan(norm))
                c = __int_as_float(0x7FC00000);
            else if (norm > p.max_norm)
                c = (float)(p.max_norm / norm);
        }
        p.status->nsq = nsq;
        p.status->norm = norm;
        p.status->clip = c;
        p.status->flags = isfinite(norm) ? 0u : kFlagNonFinite;
        p.status->ticket = 0u;
    }
}

// ------------------------------------------------------------------- K2

// One parameter of the AdamW update, in the order the update is written.
__device__ __forceinline__ void adamw1(float gh, float c, const StepScalars &s,
                                       float &master, float &m, float &v)
{
    const float g = __fmul_rn(gh, c);
    const float mi = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
    const float vi = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
    const float d = __fadd_rn(__fsqrt_rn(vi), s.eps);
    const float u = __fdiv_rn(mi, d);
    float pm = __fsub_rn(master, __fmul_rn(s.step_size, u));
    pm = __fmul_rn(pm, s.decay);
    master = pm;
    m = mi;
    v = vi;
}

template <int W, int CAP, bool REREAD>
__global__ void __launch_bounds__(kThreads)
zero1_adamw_ag_kernel(const __grid_constant__ UpdParams<CAP> p)
{
    const float c = p.status->clip;
    const int nw = W > 0 ? W : p.world;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    if (tid < p.nvec) {
        // Walk this thread's vectors from the highest address down: the
        // reduce-scatter kernel wrote those last, so they are the likeliest
        // to still sit in L2.
        uint64_t k = (p.nvec - 1 - tid) / stride;
        for (;;) {
            const uint64_t vec = tid + k * stride;
            float gh[8];
            if (REREAD) {
                rank_sum8<W>(p.grads, p.world, vec, gh);
#pragma unroll
                for (int j = 0; j < 8; ++j) gh[j] = __fmul_rn(gh[j], p.sc.inv_w);
            } else {
                const float4 a = ld_stream_f4(p.ghat + 2 * vec);
                const float4 b = ld_stream_f4(p.ghat + 2 * vec + 1);
                gh[0] = a.x; gh[1] = a.y; gh[2] = a.z; gh[3] = a.w;
                gh[4] = b.x; gh[5] = b.y; gh[6] = b.z; gh[7] = b.w;
            }
            float4 w0 = ld_f4(p.master + 2 * vec), w1 = ld_f4(p.master + 2 * vec + 1);
            float4 m0 = ld_f4(p.m + 2 * vec), m1 = ld_f4(p.m + 2 * vec + 1);
            float4 v0 = ld_f4(p.v + 2 * vec), v1 = ld_f4(p.v + 2 * vec + 1);
            adamw1(gh[0], c, p.sc, w0.x, m0.x, v0.x);
            adamw1(gh[1], c, p.sc, w0.y, m0.y, v0.y);
            adamw1(gh[2], c, p.sc, w0.z, m0.z, v0.z);
            adamw1(gh[3], c, p.sc, w0.w, m0.w, v0.w);
            adamw1(gh[4], c, p.sc, w1.x, m1.x, v1.x);
            adamw1(gh[5], c, p.sc, w1.y, m1.y, v1.y);
            adamw1(gh[6], c, p.sc, w1.z, m1.z, v1.z);
            adamw1(gh[7], c, p.sc, w1.w, m1.w, v1.w);
            p.master[2 * vec] = w0; p.master[2 * vec + 1] = w1;
            p.m[2 * vec] = m0;      p.m[2 * vec + 1] = m1;
            p.v[2 * vec] = v0;      p.v[2 * vec + 1] = v1;
            const uint4 b16 = make_uint4(pack2(w0.x, w0.y), pack2(w0.z, w0.w),
                                         pack2(w1.x, w1.y), pack2(w1.z, w1.w));
            // All-gather: every rank's replica receives the same 16 bytes.
#pragma unroll 8
            for (int r = 0; r < nw; ++r) __stcs(p.params[r] + vec, b16);
            if (k == 0) break;
            --k;
        }
    }
    const uint64_t e = p.nvec * kVec + tid;
    if (tid < kVec && e < p.n) {
        float gh;
        if (REREAD)
            gh = __fmul_rn(rank_sum1(p.grads, p.world, e), p.sc.inv_w);
        else
            gh = reinterpret_cast<const float *>(p.ghat)[e];
        float *mw = reinterpret_cast<float *>(p.master);
        float *mm = reinterpret_cast<float *>(p.m);
        float *mv = reinterpret_cast<float *>(p.v);
        float w = mw[e], m = mm[e], v = mv[e];
        adamw1(gh, c, p.sc, w, m, v);
        mw[e] = w;
        mm[e] = m;
        mv[e] = v;
        const __nv_bfloat16 b = __float2bfloat16_rn(w);
        for (int r = 0; r < nw; ++r)
            reinterpret_cast<__nv_bfloat16 *>(p.params[r])[e] = b;
    }
}

// ------------------------------------------------------------- launchers

template <int W, int CAP>
cudaError_t launch_w(const StepLaunch &s, cudaStream_t stream, cudaEvent_t *ev)
{
    const uint64_t nvec = s.n / kVec;
    RsParams<CAP> rp{};
    UpdParams<CAP> up{};
    for (int r = 0; r < s.world; ++r) {
        rp.grads[r] = static_cast<const uint4 *>(s.grads[r]);
        up.grads[r] = static_cast<const uint4 *>(s.grads[r]);
        up.params[r] = static_cast<uint4 *>(s.params[r]);
    }
    rp.ghat = reinterpret_cast<float4 *>(s.ghat);
    rp.partials = s.partials;
    rp.status = s.status;
    rp.nvec = nvec;
    rp.n = s.n;
    rp.world = s.world;
    rp.inv_w = s.sc.inv_w;
    rp.max_norm = s.max_norm;

    up.ghat = reinterpret_cast<const float4 *>(s.ghat);
    up.master = reinterpret_cast<float4 *>(s.master);
    up.m = reinterpret_cast<float4 *>(s.m);
    up.v = reinterpret_cast<float4 *>(s.v);
    up.status = s.status;
    up.nvec = nvec;
    up.n = s.n;
    up.world = s.world;
    up.sc = s.sc;

    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    if (s.ghat)
        zero1_rs_norm_kernel<W, CAP, true><<<s.grid_rs, kThreads, 0, stream>>>(rp);
    else
        zero1_rs_norm_kernel<W, CAP, false><<<s.grid_rs, kThreads, 0, stream>>>(rp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
    if (s.ghat)
        zero1_adamw_ag_kernel<W, CAP, false><<<s.grid_update, kThreads, 0, stream>>>(up);
    else
        zero1_adamw_ag_kernel<W, CAP, true><<<s.grid_update, kThreads, 0, stream>>>(up);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
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

void plan_grids(int world, uint64_t n, bool reread, int num_sms, int *grid_rs, int *grid_update)
{
    (void)world;
    (void)reread;
    // 256-thread CTAs; 4 resident per SM keeps ~64 KB of loads in flight per
    // SM for the 16-byte streams, and both kernels fit that at their register
    // budgets.  Never more CTAs than there are vectors to process.
    const uint64_t nvec = n / kVec;
    const uint64_t need = (nvec + kThreads - 1) / kThreads;
    uint64_t g = (uint64_t)num_sms * 4;
    if (need < g) g = need;
    if (g < 1) g = 1;
    *grid_rs = (int)g;
    *grid_update = (int)g;
}

}  // namespace zero1
