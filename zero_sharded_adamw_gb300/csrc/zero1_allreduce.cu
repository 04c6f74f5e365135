// zero1_allreduce.cu -- the data-parallel (DDP) all-reduce of W emulated
// ranks' buffers: every output receives the rank-ordered fp32 sum (or mean)
// of the W inputs, in bf16 or fp32, in one pass over HBM.
//
// Sources (web pages, cited by title and section):
//  "Parallel training" (notes.cassieliang.com), "How cards talk: collective
//    communication": the 4-rank gloo example (arange(4) + rank -> all-reduce
//    [6, 10, 14, 18]) and all-reduce = reduce-scatter + all-gather.
//  "Stanford CS336 Lecture 8 close reading: Parallelism (part 2)", section 5
//    (the four-rank experiment), section 6 (the benchmark: 1e8 fp32 elements,
//    world size 4) and section 7 (DDP: all_reduce(param.grad, op=AVG)).
//
// The kernel is the reduce-scatter half of the ZeRO-1 step fused with the
// all-gather half: a persistent, warp-specialised TMA pipeline, one CTA per
// SM.  A producer warp streams (rank, tile) slices of 2048 elements into a
// 4-stage, 32 KB-per-stage shared-memory ring (8 bf16 or 4 fp32 slices per
// stage: a rank group of one tile, or several tiles of all ranks when W is
// small); 8 consumer warps add the ranks in order 0..W-1 in fp32, scale by
// fp32(1/W) for the mean, round to the output type and write the result in
// place into the stage; a store warp's lanes bulk-store each finished tile
// to all W outputs.  Inputs and outputs may alias rank by rank (in place):
// a tile's outputs are stored only after all its inputs have been read.
// Every mbarrier wait gives up after 1 s and sets bit 0 of `errors`.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "zero1.h"
#include "zero1_internal.h"
#include "zero1_ptx.cuh"

namespace zero1 {
namespace {

using namespace ptx;

constexpr int kTile = 2048;
constexpr int kStages = 4;
constexpr int kStageBytes = 32768;
constexpr int kConsumers = 256;
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kThreads = kConsumers + 64;          // + producer warp + store warp

template <typename T>
struct Slots {
    static constexpr int n = kStageBytes / (kTile * (int)sizeof(T));   // bf16: 8, fp32: 4
};

template <int CAP>
struct ArParams {
    const unsigned char *in[CAP];
    unsigned char *out[CAP];
    unsigned *errors;          // may be null
    uint64_t nvec, n;
    int world;
    int average;
    float scale;               // fp32(1/W)
};

struct ArSmem {
    unsigned char stage[kStages][kStageBytes];
    uint64_t full[kStages], done[kStages], empty[kStages];
    int abort;
    unsigned local_errors;
};

__device__ __forceinline__ uint32_t count_of(uint64_t nel, uint64_t j)
{
    const uint64_t base = j * kTile;
    return (uint32_t)(nel - base < (uint64_t)kTile ? nel - base : kTile);
}

// Element offsets of consumer thread t inside a tile, as two groups of 4:
// bf16 takes 8 contiguous elements (one 16-byte access), fp32 takes 4 from
// each half of the tile (two 16-byte accesses, consecutive across lanes).
template <typename T>
__device__ __forceinline__ void offsets(uint32_t t, uint32_t &o0, uint32_t &o1)
{
    if (sizeof(T) == 2) {
        o0 = 8u * t;
        o1 = 8u * t + 4u;
    } else {
        o0 = 4u * t;
        o1 = kTile / 2 + 4u * t;
    }
}

template <typename T>
__device__ __forceinline__ void load8(const unsigned char *slice, uint32_t o0, uint32_t o1, bool v0, bool v1,
                                      float x[8])
{
    if (sizeof(T) == 2) {
        if (v0) set_widened(x, *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(slice) + o0));
    } else {
        const float *f = reinterpret_cast<const float *>(slice);
        if (v0) {
            const float4 a = *reinterpret_cast<const float4 *>(f + o0);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        }
        if (v1) {
            const float4 b = *reinterpret_cast<const float4 *>(f + o1);
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
    }
}

template <typename T>
__device__ __forceinline__ void store8(unsigned char *slice, uint32_t o0, uint32_t o1, bool v0, bool v1,
                                       const float x[8])
{
    if (sizeof(T) == 2) {
        if (v0)
            *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(slice) + o0) =
                make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
    } else {
        float *f = reinterpret_cast<float *>(slice);
        if (v0) *reinterpret_cast<float4 *>(f + o0) = make_float4(x[0], x[1], x[2], x[3]);
        if (v1) *reinterpret_cast<float4 *>(f + o1) = make_float4(x[4], x[5], x[6], x[7]);
    }
}

template <typename T>
__device__ __forceinline__ float load1(const unsigned char *p, uint64_t e)
{
    if (sizeof(T) == 2) return __uint_as_float((unsigned)reinterpret_cast<const uint16_t *>(p)[e] << 16);
    return reinterpret_cast<const float *>(p)[e];
}

template <typename T>
__device__ __forceinline__ void store1(unsigned char *p, uint64_t e, float x)
{
    if (sizeof(T) == 2)
        reinterpret_cast<__nv_bfloat16 *>(p)[e] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(p)[e] = x;
}

template <typename T, int CAP>
__global__ void __launch_bounds__(kThreads, 1) zero1_allreduce_kernel(const __grid_constant__ ArParams<CAP> p)
{
    constexpr int kSlots = Slots<T>::n;
    constexpr uint32_t kSlice = kTile * sizeof(T);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    ArSmem &sm = *reinterpret_cast<ArSmem *>(smem_raw);
    const int nw = p.world;
    const int ngroups = (nw + kSlots - 1) / kSlots;
    const int sub = nw >= kSlots ? 1 : kSlots / nw;
    const uint64_t nel = p.nvec * kVec;
    const uint64_t ntiles = (nel + kTile - 1) / kTile;
    const uint32_t tcta = blockIdx.x < ntiles ? (uint32_t)((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0u;
    auto tile_of = [&](uint32_t i) -> uint64_t { return blockIdx.x + (uint64_t)i * gridDim.x; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort = &sm.abort;
    unsigned *errors = p.errors ? p.errors : &sm.local_errors;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.done[s], kConsumerWarps);
            mbar_init(&sm.empty[s], 1);
        }
        sm.abort = 0;
        sm.local_errors = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint64_t once = policy_evict_first();

    if (warp == kConsumerWarps) {                                 // producer
        if (lane == 0) {
            uint32_t k = 0;
            for (uint32_t b = 0; b * sub < tcta && !*abort; ++b) {
                for (int grp = 0; grp < ngroups; ++grp, ++k) {
                    const int s = k % kStages;
                    if (k >= kStages && !mbar_wait(&sm.empty[s], ((k / kStages) & 1u) ^ 1u, abort, errors)) break;
                    const int r0 = grp * kSlots;
                    const int rn = nw - r0 < kSlots ? nw - r0 : kSlots;
                    uint32_t bytes = 0;
                    for (int q = 0; q < sub && b * sub + q < tcta; ++q)
                        bytes += (uint32_t)rn * count_of(nel, tile_of(b * sub + q)) * (uint32_t)sizeof(T);
                    mbar_arrive_expect_tx(&sm.full[s], bytes);
                    for (int q = 0; q < sub && b * sub + q < tcta; ++q) {
                        const uint64_t j = tile_of(b * sub + q);
                        const uint32_t cnt = count_of(nel, j);
                        for (int r = 0; r < rn; ++r)
                            tma_load_hint(sm.stage[s] + (q * rn + r) * kSlice, p.in[r0 + r] + j * kSlice,
                                          cnt * (uint32_t)sizeof(T), &sm.full[s], once);
                    }
                }
            }
            if (*abort) drain_loads<kStages>(sm.full, k);
        }
        return;
    }

    if (warp == kConsumerWarps + 1) {                             // stores
        uint32_t k = 0;
        bool stop = false;
        for (uint32_t b = 0; b * sub < tcta && !stop; ++b) {
            for (int grp = 0; grp < ngroups; ++grp, ++k) {
                const int s = k % kStages;
                const bool got = mbar_wait(&sm.done[s], (k / kStages) & 1u, abort, errors);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    stop = true;
                    break;
                }
                if (grp == ngroups - 1) {                      // finished tiles: fan out to every rank
                    const int rn = nw - grp * kSlots < kSlots ? nw - grp * kSlots : kSlots;
                    for (int q = 0; q < sub && b * sub + q < tcta; ++q) {
                        const uint64_t j = tile_of(b * sub + q);
                        const uint32_t cnt = count_of(nel, j);
                        for (int r = lane; r < nw; r += 32)
                            tma_store_hint(p.out[r] + j * kSlice, sm.stage[s] + (q * rn) * kSlice,
                                           cnt * (uint32_t)sizeof(T), once);
                    }
                }
                tma_commit();
                if (k >= 1) {
                    tma_wait_read<1>();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.empty[(k - 1) % kStages]);
                }
            }
        }
        tma_wait_all();
        return;
    }

    // Consumers.
    uint32_t o0, o1;
    offsets<T>(threadIdx.x, o0, o1);
    uint32_t k = 0;
    float acc[8];
    for (uint32_t b = 0; b * sub < tcta; ++b) {
        bool ok = true;
        for (int grp = 0; grp < ngroups; ++grp, ++k) {
            const int s = k % kStages;
            const bool got = mbar_wait(&sm.full[s], (k / kStages) & 1u, abort, errors);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                ok = false;
                break;
            }
            const int rn = nw - grp * kSlots < kSlots ? nw - grp * kSlots : kSlots;
            for (int q = 0; q < sub && b * sub + q < tcta; ++q) {
                const uint32_t cnt = count_of(nel, tile_of(b * sub + q));
                const bool v0 = o0 < cnt, v1 = o1 < cnt;
#pragma unroll
                for (int r = 0; r < kSlots; ++r) {
                    if (r < rn) {
                        float x[8];
                        load8<T>(sm.stage[s] + (q * rn + r) * kSlice, o0, o1, v0, v1, x);
                        if (grp == 0 && r == 0) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) acc[c] = x[c];
                        } else {
#pragma unroll
                            for (int c = 0; c < 8; ++c) acc[c] = __fadd_rn(acc[c], x[c]);
                        }
                    }
                }
                if (grp == ngroups - 1) {
                    float y[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) y[c] = p.average ? __fmul_rn(acc[c], p.scale) : acc[c];
                    store8<T>(sm.stage[s] + (q * rn) * kSlice, o0, o1, v0, v1, y);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.done[s]);
        }
        if (!ok) break;
    }

    // The last n % 8 elements, one per thread of CTA 0: read every rank's
    // element, then write every rank's (safe in place).
    const uint64_t e = nel + threadIdx.x;
    if (blockIdx.x == 0 && threadIdx.x < kVec && e < p.n) {
        float s = load1<T>(p.in[0], e);
        for (int r = 1; r < nw; ++r) s = __fadd_rn(s, load1<T>(p.in[r], e));
        if (p.average) s = __fmul_rn(s, p.scale);
        for (int r = 0; r < nw; ++r) store1<T>(p.out[r], e, s);
    }
}

template <typename T, int CAP>
cudaError_t launch_ar(uint64_t n, int world, int average, const void *const *in, void *const *out,
                      unsigned *errors, int num_sms, cudaStream_t stream)
{
    ArParams<CAP> p{};
    for (int r = 0; r < world; ++r) {
        p.in[r] = static_cast<const unsigned char *>(in[r]);
        p.out[r] = static_cast<unsigned char *>(out[r]);
    }
    p.errors = errors;
    p.nvec = n / kVec;
    p.n = n;
    p.world = world;
    p.average = average;
    p.scale = (float)(1.0 / (double)world);
    const uint64_t ntiles = (p.nvec * kVec + kTile - 1) / kTile;
    uint64_t grid = (uint64_t)num_sms;
    if (ntiles < grid) grid = ntiles;
    if (grid < 1) grid = 1;
    auto kern = zero1_allreduce_kernel<T, CAP>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kern), (int)sizeof(ArSmem));
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads, sizeof(ArSmem), stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_ar_t(uint64_t n, int world, int average, const void *const *in, void *const *out,
                        unsigned *errors, int num_sms, cudaStream_t stream)
{
    if (world <= 8) return launch_ar<T, 8>(n, world, average, in, out, errors, num_sms, stream);
    if (world <= 64) return launch_ar<T, 64>(n, world, average, in, out, errors, num_sms, stream);
    return launch_ar<T, 512>(n, world, average, in, out, errors, num_sms, stream);
}

// ------------------------------------------------------------ all-gather

// The ZeRO-3 / FSDP parameter all-gather ("Lecture 7 close reading" 5.4:
// before a layer runs, its sharded parameters are gathered onto every rank).
// Rank r's shard holds elements [r*S, min((r+1)*S, n)); every output q
// receives all n.  A byte copy with W-way fan-out.  One 32-thread CTA per
// 16 KB tile: lane 0 bulk-loads the tile into shared memory, the lanes
// bulk-store it to the W outputs, the CTA waits for the stores to have read
// shared memory and exits.  Per-layer gathers are short, so instead of a
// persistent pipeline many small CTAs (about 13 per SM) keep ~200 KB per
// SM in flight.  The last CTA copies every shard's sub-16-byte tail.
constexpr int kAgBytes = 16384;

template <int CAP>
struct AgParams {
    const unsigned char *shards[CAP];
    unsigned char *out[CAP];
    unsigned *errors;
    uint64_t n, shard_len;
    uint64_t tiles_per_shard;
    int world;
    int esize;
};

struct AgSmem {
    unsigned char tile[kAgBytes];
    uint64_t full;
};

// Elements of shard r, and of its 16-byte vector part.
__device__ __forceinline__ void shard_extent(uint64_t n, uint64_t s, int r, int esize, uint64_t &len, uint64_t &vlen)
{
    const uint64_t lo = (uint64_t)r * s;
    len = lo >= n ? 0 : (n - lo < s ? n - lo : s);
    const uint64_t per16 = 16u / (uint64_t)esize;
    vlen = len / per16 * per16;
}

template <int CAP>
__global__ void __launch_bounds__(32) zero1_allgather_kernel(const __grid_constant__ AgParams<CAP> p)
{
    __shared__ __align__(128) AgSmem sm;
    const int lane = threadIdx.x;
    const uint64_t tile_elems = (uint64_t)(kAgBytes / p.esize);
    const uint64_t item = blockIdx.x;
    if (item == (uint64_t)p.world * p.tiles_per_shard) {          // the tails
        if (lane == 0) {
            for (int r = 0; r < p.world; ++r) {
                uint64_t len, vlen;
                shard_extent(p.n, p.shard_len, r, p.esize, len, vlen);
                for (uint64_t i = vlen; i < len; ++i) {
                    const uint64_t dst = ((uint64_t)r * p.shard_len + i) * p.esize;
                    for (int q = 0; q < p.world; ++q) {
                        if (p.esize == 2)
                            *reinterpret_cast<uint16_t *>(p.out[q] + dst) =
                                reinterpret_cast<const uint16_t *>(p.shards[r])[i];
                        else
                            *reinterpret_cast<uint32_t *>(p.out[q] + dst) =
                                reinterpret_cast<const uint32_t *>(p.shards[r])[i];
                    }
                }
            }
        }
        return;
    }
    const int r = (int)(item / p.tiles_per_shard);
    const uint64_t e0 = (item % p.tiles_per_shard) * tile_elems;
    uint64_t len, vlen;
    shard_extent(p.n, p.shard_len, r, p.esize, len, vlen);
    if (e0 >= vlen) return;                                       // past a short or empty shard
    const uint32_t bytes = (uint32_t)((vlen - e0 < tile_elems ? vlen - e0 : tile_elems) * p.esize);
    int abort_flag = 0;
    volatile int *abort = &abort_flag;
    unsigned *errors = p.errors;
    unsigned local = 0;
    if (!errors) errors = &local;
    if (lane == 0) {
        mbar_init(&sm.full, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const uint64_t once = policy_evict_first();
    if (lane == 0) {
        mbar_arrive_expect_tx(&sm.full, bytes);
        tma_load_hint(sm.tile, p.shards[r] + e0 * p.esize, bytes, &sm.full, once);
    }
    const bool got = mbar_wait(&sm.full, 0, abort, errors);
    if (!__all_sync(0xFFFFFFFFu, got)) {
        // Let the load land (bounded) before the CTA's shared memory goes away.
        if (lane == 0) drain_loads<1>(&sm.full, 1);
        return;
    }
    const uint64_t dst = ((uint64_t)r * p.shard_len + e0) * p.esize;
    for (int q = lane; q < p.world; q += 32) tma_store_hint(p.out[q] + dst, sm.tile, bytes, once);
    tma_commit();
    tma_wait_read<0>();
}

template <int CAP>
cudaError_t launch_ag(uint64_t n, int world, uint64_t shard_len, int esize, const void *const *shards,
                      void *const *out, unsigned *errors, cudaStream_t stream)
{
    AgParams<CAP> p{};
    for (int r = 0; r < world; ++r) {
        p.shards[r] = static_cast<const unsigned char *>(shards[r]);
        p.out[r] = static_cast<unsigned char *>(out[r]);
    }
    const uint64_t tile_elems = kAgBytes / esize;
    p.errors = errors;
    p.n = n;
    p.shard_len = shard_len;
    p.tiles_per_shard = (shard_len + tile_elems - 1) / tile_elems;
    p.world = world;
    p.esize = esize;
    const uint64_t grid = (uint64_t)world * p.tiles_per_shard + 1;
    if (grid > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    zero1_allgather_kernel<CAP><<<(unsigned)grid, 32, 0, stream>>>(p);
    return cudaGetLastError();
}

int afail(int code, const char *msg)
{
    set_error_message(msg);
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace zero1

extern "C" int zero1_allreduce(uint64_t n, int world, int dtype, int op, const void *const *in_ptrs,
                               void *const *out_ptrs, unsigned *errors, void *stream)
{
    using namespace zero1;
    if (n == 0) return afail(ZERO1_EINVAL, "zero1_allreduce: n must be > 0");
    if (world < 1 || world > ZERO1_MAX_WORLD) return afail(ZERO1_EINVAL, "zero1_allreduce: bad world size");
    if (dtype != ZERO1_DTYPE_BF16 && dtype != ZERO1_DTYPE_F32) return afail(ZERO1_EINVAL, "zero1_allreduce: bad dtype");
    if (op != ZERO1_OP_SUM && op != ZERO1_OP_AVG) return afail(ZERO1_EINVAL, "zero1_allreduce: bad op");
    if (!in_ptrs || !out_ptrs) return afail(ZERO1_EINVAL, "zero1_allreduce: pointer array is NULL");
    for (int r = 0; r < world; ++r) {
        if (!in_ptrs[r] || !out_ptrs[r]) return afail(ZERO1_EINVAL, "zero1_allreduce: a rank buffer is NULL");
        if (!aligned16(in_ptrs[r]) || !aligned16(out_ptrs[r]))
            return afail(ZERO1_EALIGN, "zero1_allreduce: rank buffers must be 16-byte aligned");
    }
    if (errors && (reinterpret_cast<uintptr_t>(errors) & 3u))
        return afail(ZERO1_EALIGN, "zero1_allreduce: errors must be 4-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return afail(ZERO1_ECUDA, cudaGetErrorString(e));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = dtype == ZERO1_DTYPE_BF16
            ? launch_ar_t<uint16_t>(n, world, op == ZERO1_OP_AVG, in_ptrs, out_ptrs, errors, sms, st)
            : launch_ar_t<float>(n, world, op == ZERO1_OP_AVG, in_ptrs, out_ptrs, errors, sms, st);
    if (e != cudaSuccess) return afail(ZERO1_ECUDA, cudaGetErrorString(e));
    return ZERO1_OK;
}

extern "C" int zero1_allgather(uint64_t n, int world, uint64_t shard_len, int dtype, const void *const *shard_ptrs,
                               void *const *out_ptrs, unsigned *errors, void *stream)
{
    using namespace zero1;
    if (n == 0) return afail(ZERO1_EINVAL, "zero1_allgather: n must be > 0");
    if (world < 1 || world > ZERO1_MAX_WORLD) return afail(ZERO1_EINVAL, "zero1_allgather: bad world size");
    if (dtype != ZERO1_DTYPE_BF16 && dtype != ZERO1_DTYPE_F32) return afail(ZERO1_EINVAL, "zero1_allgather: bad dtype");
    if (shard_len == 0 || shard_len % 8 || shard_len > ((uint64_t)1 << 50) || shard_len * (uint64_t)world < n)
        return afail(ZERO1_EINVAL, "zero1_allgather: shard_len must be a multiple of 8 with shard_len*world >= n");
    if (!shard_ptrs || !out_ptrs) return afail(ZERO1_EINVAL, "zero1_allgather: pointer array is NULL");
    for (int r = 0; r < world; ++r) {
        const bool empty = (uint64_t)r * shard_len >= n;
        if (!out_ptrs[r] || (!empty && !shard_ptrs[r]))
            return afail(ZERO1_EINVAL, "zero1_allgather: a rank buffer is NULL");
        if (!aligned16(out_ptrs[r]) || (!empty && !aligned16(shard_ptrs[r])))
            return afail(ZERO1_EALIGN, "zero1_allgather: rank buffers must be 16-byte aligned");
    }
    if (errors && (reinterpret_cast<uintptr_t>(errors) & 3u))
        return afail(ZERO1_EALIGN, "zero1_allgather: errors must be 4-byte aligned");
    const int esize = dtype == ZERO1_DTYPE_BF16 ? 2 : 4;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (world <= 8)
        e = launch_ag<8>(n, world, shard_len, esize, shard_ptrs, out_ptrs, errors, st);
    else if (world <= 64)
        e = launch_ag<64>(n, world, shard_len, esize, shard_ptrs, out_ptrs, errors, st);
    else
        e = launch_ag<512>(n, world, shard_len, esize, shard_ptrs, out_ptrs, errors, st);
    if (e != cudaSuccess) return afail(ZERO1_ECUDA, cudaGetErrorString(e));
    return ZERO1_OK;
}
