// zero1_ptx.cuh -- inline-PTX building blocks shared by the sm_103a kernels:
// 1-D TMA bulk copies with mbarrier completion, bulk-store groups, L2
// eviction-priority hints, time-bounded mbarrier waits, bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zero1_internal.h"

namespace zero1 {
namespace ptx {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s per wait

// ------------------------------------------------------ PTX: TMA, mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Global -> shared bulk copy; `bytes` (multiple of 16) are counted on `bar`.
__device__ __forceinline__ void tma_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void tma_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tma_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 eviction-priority policies for the cache-hinted copies below.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_hint(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared -> global bulk copy in this thread's current bulk group.
__device__ __forceinline__ void tma_store_hint(void *gdst, const void *smem_src, uint32_t bytes, uint64_t policy)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes), "l"(policy)
                 : "memory");
}

// 16-byte global store with an L2 eviction-priority hint.
__device__ __forceinline__ void st_hint(float *dst, float4 v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(policy)
                 : "memory");
}

// Drop one 128-byte L2 line without writing it back (dead scratch only).
__device__ __forceinline__ void discard_l2_line(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


// Bounded wait on an mbarrier phase.  Gives up when another thread of the
// CTA has raised `abort`, or after kWaitLimitNs, raising `abort` and the
// sticky error bit.  Returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, unsigned *errors)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(errors, kErrWaitTimeout);
                return false;
            }
        }
    }
}

// After an abort, let the producer's last loads land before it exits (the
// CTA's shared memory must outlive them).  Item k used stage k % kStages,
// phase (k / kStages) & 1.
template <int kStages>
__device__ __forceinline__ void drain_loads(uint64_t *full, uint32_t issued)
{
    for (uint32_t k = issued > kStages ? issued - kStages : 0; k < issued; ++k) {
        const unsigned long long t0 = global_ns();
        while (!mbar_test(&full[k % kStages], (k / kStages) & 1u) && global_ns() - t0 < kWaitLimitNs) {
        }
    }
}

// ------------------------------------------ programmatic dependent launch

// Let the next kernel of the stream launch now, if it was launched with a
// programmatic dependency on this one (it still waits for this grid in its
// own grid_dependency_wait).  No-op otherwise.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Wait until the grid this one programmatically depends on has completed
// and its memory is visible.  No-op for a launch without that dependency.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------ thread-block cluster

// All threads of all CTAs of the cluster arrive and wait (the non-.aligned
// form: threads need not be converged when they reach it); the release /
// acquire pair orders every CTA's shared-memory writes before the barrier
// against reads after it, anywhere in the cluster.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// The two halves of a cluster barrier, for work between them: arrive
// (relaxed: no memory ordering), and later wait for every thread of every
// CTA of the cluster to have arrived.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }

// Store a double at the same shared-memory offset as `local`, in the CTA of
// cluster rank `rank` (distributed shared memory).
__device__ __forceinline__ void st_cluster_f64(double *local, uint32_t rank, double v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(remote), "d"(v) : "memory");
}

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

}  // namespace ptx
}  // namespace zero1
