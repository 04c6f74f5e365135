// zero1_host.cu -- the C ABI declared in include/zero1.h: argument checks,
// the shard plan, per-step scalars, device memory, and the launches.
//
// Shard plan ("Stanford CS336 Lecture 7 close reading: Parallelism (part 1)",
// 5.2; equal chunks as "Stanford CS336 Lecture 8 close reading: Parallelism
// (part 2)", section 2, requires of a reduce-scatter): S = ceil(n/W) rounded
// up to 64, rank r owns [r*S, min((r+1)*S, n)).  In one GPU's memory the W
// fp32 shards of master, m and v sit end to end, so parameter i's state is
// at index i of each array and a launch covers all ranks' shards at once.
//
// Per-step scalars ("Parallel training", "mixed precision and AdamW"):
// formed in double, rounded once to fp32 -- step_size = lr*sqrt(1-beta2^t)/
// (1-beta1^t), decay = 1 - lr*wd, 1-beta1, 1-beta2, 1/W.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <tuple>
#include <unordered_set>
#include <algorithm>
#include <utility>
#include <vector>

#include "zero1.h"
#include "zero1_internal.h"
#include "zero1_policy.h"

// Slots in each of the host path's two device rings (uploads, downloads),
// and the copy streams each direction's chunks are dealt over, so that
// several copies are in flight (the driver maps the streams onto the
// device's copy engines; GB300 reports three).  Measured on the 7B
// workload: 8 or 16 slots with 2 or 4 streams ran within 7% of one another
// (the host link sets the rate); 8 slots with 3 streams were about 10%
// slower.
#ifndef ZERO1_HOST_SLOTS
#define ZERO1_HOST_SLOTS 8
#define ZERO1_HOST_COPY_STREAMS 4
#endif
constexpr int kHostSlots = ZERO1_HOST_SLOTS;
constexpr int kHostCopyStreams = ZERO1_HOST_COPY_STREAMS;
// Device bytes of one slot by default: the W ranks' bf16 slices of one chunk
// (256 MiB: measured on GB300 hosts at 1.6-2x the host-link rate of 64 MiB
// slots; 8 copy streams per direction with 64 MiB slots gained nothing).
constexpr uint64_t kHostSlotBytes = 256ull << 20;
constexpr uint64_t kHostChunkAlign = 2048;   // chunks start on whole update tiles

// The host-buffer steps (zero1_step_host, zero1_step_host_async): gradients
// and replicas live in host memory and pass through two bounded device rings
// chunk by chunk.  Per step, every chunk's W gradient slices are uploaded
// into a ring slot and reduce-scattered into the fp32 scratch (with the
// chunk's norm partial) on the reduce stream; once the last chunk's partial
// is in, the update stream runs each chunk's clip + AdamW + bf16 cast +
// all-gather into a download slot, which a download stream copies to the W
// host replicas.  Step t+1's chunk i reduce waits only for step t's chunk i
// update (the scratch it overwrites), so one step's downloads overlap the
// next step's uploads.  The norm partials alternate between two sets by
// step parity, since step t's updates still read step t's set while step
// t+1's reduces fill the other.
struct HostPath {
    bool ready = false;
    uint64_t chunk = 0;            // parameters per chunk (a multiple of kHostChunkAlign)
    int nchunks = 0;
    uint64_t rank_stride = 0;      // bytes between ranks' slices in a slot (256-byte rounded)
    void *staging = nullptr;       // kHostSlots upload slots, then kHostSlots download slots
    double *sums = nullptr;        // 2 parity sets x nchunks x (sum, plain sum)
    cudaStream_t rs = nullptr, upd = nullptr, up[kHostCopyStreams] = {}, down[kHostCopyStreams] = {};
    cudaEvent_t fork = nullptr, norm_done = nullptr, last = nullptr;
    cudaEvent_t up_ready[kHostSlots] = {}, up_free[kHostSlots] = {};
    cudaEvent_t down_ready[kHostSlots] = {}, down_free[kHostSlots] = {};
    bool up_used[kHostSlots] = {}, down_used[kHostSlots] = {};
    std::vector<cudaEvent_t> upd_done;   // per chunk: the latest step's update of it has read the scratch
    std::vector<char> upd_recorded;
    uint64_t up_count = 0, down_count = 0;
    int parity = 0;
    bool pending = false;          // steps enqueued on the internal streams and not yet joined
};

struct zero1_ctx {
    uint64_t n = 0;
    int world = 0;
    zero1_hparams hp{};
    uint64_t t = 0;              // steps taken
    uint64_t shard = 0;          // S
    uint64_t padded = 0;         // W * S
    int device = 0;
    int num_sms = 0;
    int grid_rs = 0, grid_update = 0;
    bool reread = false;         // W <= 2: the update kernel re-reads the gradients
    void *block = nullptr;       // one cudaMalloc holding everything below
    uint64_t block_bytes = 0;
    float *master = nullptr, *ghat = nullptr;
    unsigned char *m = nullptr, *v = nullptr;   // fp32 or bf16 elements (msz bytes each)
    zero1_options opts{};
    size_t msz = sizeof(float);
    double *partials = nullptr;
    zero1::DevStatus *status = nullptr;
    // host-buffer steps (zero1_step_host, zero1_step_host_async): rings,
    // streams and events, set up on first use
    HostPath host;
    // capturable handles: bias-correction table (1 - beta1^t, 1 - beta2^t)
    // for t = 1..tab_len on the device, and where the kernels read lr
    double2 *bctab = nullptr;
    uint64_t tab_len = 0;
    const double *lr_ptr = nullptr;
    // per-kernel timing (zero1_profile_start/stop): 3 events per step
    std::vector<cudaEvent_t> prof;
    int prof_capacity = 0, prof_used = 0;
    // bucketed step (zero1_bucket_*): buckets in call order, their norm sums,
    // and a reduce-scatter scratch for W <= 2 (whose plain step re-reads;
    // the host-buffer steps use it too)
    bool bucket_open = false;
    int bucket_mode = 0;         // 0: no bucket yet, 1: reduce-only buckets, 2: reduce + update buckets
    std::vector<std::pair<uint64_t, uint64_t>> buckets;
    double *bucket_sums = nullptr;
    float *ghat_bucket = nullptr;
};

constexpr int kMaxBuckets = 4096;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    if (e == cudaErrorMemoryAllocation)
        return fail(ZERO1_ENOMEM, "%s: %s", what, cudaGetErrorString(e));
    return fail(ZERO1_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::mutex g_mu;
std::unordered_set<zero1_ctx *> g_live;

bool live(zero1_ctx *h)
{
    std::lock_guard<std::mutex> lk(g_mu);
    return h != nullptr && g_live.count(h) != 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

bool finite_nonneg(double x) { return std::isfinite(x) && x >= 0.0; }

int check_hparams(const zero1_hparams *hp)
{
    if (!finite_nonneg(hp->lr)) return fail(ZERO1_EINVAL, "lr must be finite and >= 0");
    if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0)) return fail(ZERO1_EINVAL, "beta1 must be in [0, 1)");
    if (!(hp->beta2 >= 0.0 && hp->beta2 < 1.0)) return fail(ZERO1_EINVAL, "beta2 must be in [0, 1)");
    if (!finite_nonneg(hp->eps)) return fail(ZERO1_EINVAL, "eps must be finite and >= 0");
    if (!finite_nonneg(hp->weight_decay)) return fail(ZERO1_EINVAL, "weight_decay must be finite and >= 0");
    if (std::isnan(hp->max_norm)) return fail(ZERO1_EINVAL, "max_norm must not be NaN");
    return ZERO1_OK;
}

zero1::StepScalars step_scalars(const zero1_hparams &hp, int world, uint64_t t)
{
    const double bc1 = 1.0 - std::pow(hp.beta1, (double)t);
    const double bc2 = 1.0 - std::pow(hp.beta2, (double)t);
    zero1::StepScalars s;
    s.inv_w = (float)(1.0 / (double)world);
    s.beta1 = (float)hp.beta1;
    s.omb1 = (float)(1.0 - hp.beta1);
    s.beta2 = (float)hp.beta2;
    s.omb2 = (float)(1.0 - hp.beta2);
    s.step_size = (float)(hp.lr * std::sqrt(bc2) / bc1);
    s.decay = (float)(1.0 - hp.lr * hp.weight_decay);
    s.eps = (float)hp.eps;
    return s;
}

// Round-to-nearest-even float -> bf16 -> float (finite values).
float round_to_bf16(float x)
{
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    float r;
    std::memcpy(&r, &u, sizeof r);
    return r;
}

// The scalars one launch of this handle uses for step t.  With bf16
// moments, d = sqrt(v) + eps is an in-place add of the scalar eps to a bf16
// tensor, which torch performs with eps rounded to bf16; the step does
// the same.
zero1::StepScalars launch_scalars(const zero1_ctx *h, uint64_t t)
{
    zero1::StepScalars s = step_scalars(h->hp, h->world, t);
    if (h->opts.moments_bf16) s.eps = round_to_bf16(s.eps);
    return s;
}

constexpr uint64_t kMaxBiasTable = 1ull << 22;   // entries (64 MiB) a capturable handle may tabulate

// The step's scalars as a capturable launch forms them on the device.
zero1::DevScalars dev_scalars(const zero1_ctx *h)
{
    zero1::DevScalars d{};
    if (h->bctab) {
        d.bc = h->bctab;
        d.tab_len = h->tab_len;
        d.lr = h->lr_ptr;
        d.weight_decay = h->hp.weight_decay;
    }
    return d;
}

// Make the handle's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

// Work a host-buffer step left on the handle's internal streams comes
// before anything the caller enqueues on `st` afterwards (the steps share
// the state, the scratch and the status).
int join_host(zero1_ctx *h, cudaStream_t st)
{
    if (!h->host.pending) return ZERO1_OK;
    cudaError_t e = cudaStreamWaitEvent(st, h->host.last, 0);
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e, "cudaStreamWaitEvent");
}

void release_host_path(HostPath &P)
{
    for (cudaStream_t x : {P.rs, P.upd})
        if (x) cudaStreamDestroy(x);
    for (int i = 0; i < kHostCopyStreams; ++i)
        for (cudaStream_t x : {P.up[i], P.down[i]})
            if (x) cudaStreamDestroy(x);
    for (cudaEvent_t x : {P.fork, P.norm_done, P.last})
        if (x) cudaEventDestroy(x);
    for (int i = 0; i < kHostSlots; ++i)
        for (cudaEvent_t x : {P.up_ready[i], P.up_free[i], P.down_ready[i], P.down_free[i]})
            if (x) cudaEventDestroy(x);
    for (cudaEvent_t x : P.upd_done)
        if (x) cudaEventDestroy(x);
    if (P.sums) cudaFree(P.sums);
    P = HostPath{};
}

}  // namespace

void zero1::set_error_message(const char *msg)
{
    snprintf(g_err, sizeof g_err, "%s", msg);
}

cudaError_t zero1::set_func_attribute_once(const void *kernel, cudaFuncAttribute attr, int value)
{
    static std::mutex mu;
    static std::set<std::tuple<const void *, int, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(kernel, dev, (int)attr);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (done.count(key)) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kernel, attr, value);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lk(mu);
        done.insert(key);
    }
    return e;
}

cudaError_t zero1::allow_dynamic_smem(const void *kernel, int bytes)
{
    return set_func_attribute_once(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

extern "C" {

const char *zero1_last_error(void) { return g_err; }

int zero1_create(uint64_t n, int world, const zero1_hparams *hp, zero1_handle *out)
{
    return zero1_create_ex(n, world, hp, nullptr, out);
}

// Capturable handles: tabulate the two bias corrections exactly as
// step_scalars forms them, up to the first t at which both are 1.0 in
// double (they stay 1.0 after it), and seed the device lr slot and t = 0.
static int build_bias_table(zero1_ctx *h)
{
    std::vector<double2> tab;
    for (uint64_t t = 1;; ++t) {
        if (t > kMaxBiasTable)
            return fail(ZERO1_EINVAL, "capturable: the bias corrections do not reach 1.0 within %llu steps",
                        (unsigned long long)kMaxBiasTable);
        const double bc1 = 1.0 - std::pow(h->hp.beta1, (double)t);
        const double bc2 = 1.0 - std::pow(h->hp.beta2, (double)t);
        tab.push_back(make_double2(bc1, bc2));
        if (bc1 == 1.0 && bc2 == 1.0) break;
    }
    cudaError_t e;
    if ((e = cudaMalloc(&h->bctab, tab.size() * sizeof(double2))) != cudaSuccess) {
        h->bctab = nullptr;
        return cuda_fail(e, "cudaMalloc of the bias-correction table");
    }
    if ((e = cudaMemcpy(h->bctab, tab.data(), tab.size() * sizeof(double2), cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(&h->status->lr, &h->hp.lr, sizeof(double), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(h->bctab);
        h->bctab = nullptr;
        return cuda_fail(e, "bias-correction table upload");
    }
    h->tab_len = tab.size();
    h->lr_ptr = &h->status->lr;
    return ZERO1_OK;
}

int zero1_create_ex(uint64_t n, int world, const zero1_hparams *hp, const zero1_options *opts, zero1_handle *out)
{
    g_err[0] = '\0';
    if (out == nullptr) return fail(ZERO1_EINVAL, "out is NULL");
    *out = nullptr;
    if (hp == nullptr) return fail(ZERO1_EINVAL, "hparams is NULL");
    if (n == 0) return fail(ZERO1_EINVAL, "n must be > 0");
    if (world < 1 || world > ZERO1_MAX_WORLD)
        return fail(ZERO1_EINVAL, "world must be in [1, %d], got %d", ZERO1_MAX_WORLD, world);
    if (n > (uint64_t)1 << 50) return fail(ZERO1_EINVAL, "n too large");
    int rc = check_hparams(hp);
    if (rc) return rc;
    zero1_options o{};
    o.size = sizeof(zero1_options);
    if (opts) {
        if (opts->size != sizeof(zero1_options)) return fail(ZERO1_EINVAL, "opts->size must be sizeof(zero1_options)");
        if (!finite_nonneg(opts->clip_eps)) return fail(ZERO1_EINVAL, "clip_eps must be finite and >= 0");
        if (opts->bucket_ctas < 0) return fail(ZERO1_EINVAL, "bucket_ctas must be >= 0");
        if (opts->small_step < -1 || opts->small_step > 1) return fail(ZERO1_EINVAL, "small_step must be -1, 0 or 1");
        if (opts->capturable != 0 && opts->capturable != 1) return fail(ZERO1_EINVAL, "capturable must be 0 or 1");
        if (opts->inject_wait_timeout != 0 && opts->inject_wait_timeout != 1)
            return fail(ZERO1_EINVAL, "inject_wait_timeout must be 0 or 1");
        if (!std::isfinite(opts->load_phase_gbs)) return fail(ZERO1_EINVAL, "load_phase_gbs must be finite");
        if (opts->load_phase_gbs > 0.0 && opts->load_phase_gbs < 1000.0)
            return fail(ZERO1_EINVAL, "load_phase_gbs must be <= 0 or at least 1000 (GB/s), got %g", opts->load_phase_gbs);
        o = *opts;
    }

    int dev = 0, count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess || count == 0)
        return fail(ZERO1_ENODEV, "no CUDA device (%s)", cudaGetErrorString(e));
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(ZERO1_ENODEV, "device %d is sm_%d%d; this library is built for sm_103a", dev, prop.major, prop.minor);

    zero1_ctx *h = new (std::nothrow) zero1_ctx;
    if (!h) return fail(ZERO1_ENOMEM, "host allocation failed");
    h->n = n;
    h->world = world;
    h->hp = *hp;
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->opts = o;
    h->msz = o.moments_bf16 ? 2 : sizeof(float);
    zero1_shard_plan(n, world, &h->shard, &h->padded);
    h->reread = world <= 2;
    zero1::plan_grids(n, h->reread, h->num_sms, &h->grid_rs, &h->grid_update);

    // One allocation: master | m | v | ghat (W >= 3) | partials | status,
    // every section 256-byte aligned.
    const uint64_t state_bytes = round_up(h->padded * sizeof(float), 256);
    const uint64_t mom_bytes = round_up(h->padded * h->msz, 256);
    const uint64_t ghat_bytes = h->reread ? 0 : state_bytes;
    const uint64_t part_bytes = round_up(2 * (uint64_t)h->grid_rs * sizeof(double), 256);
    const uint64_t status_bytes = 256;
    const uint64_t st3 = state_bytes + 2 * mom_bytes;
    h->block_bytes = st3 + ghat_bytes + part_bytes + status_bytes;
    if ((e = cudaMalloc(&h->block, h->block_bytes)) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaMalloc of optimizer state");
    }
    char *base = static_cast<char *>(h->block);
    h->master = reinterpret_cast<float *>(base);
    h->m = reinterpret_cast<unsigned char *>(base + state_bytes);
    h->v = reinterpret_cast<unsigned char *>(base + state_bytes + mom_bytes);
    h->ghat = h->reread ? nullptr : reinterpret_cast<float *>(base + st3);
    h->partials = reinterpret_cast<double *>(base + st3 + ghat_bytes);
    h->status = reinterpret_cast<zero1::DevStatus *>(base + st3 + ghat_bytes + part_bytes);
    if ((e = cudaMemset(h->block, 0, h->block_bytes)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        cudaFree(h->block);
        delete h;
        return cuda_fail(e, "cudaMemset of optimizer state");
    }
    if (o.capturable) {
        rc = build_bias_table(h);
        if (rc) {
            cudaFree(h->block);
            delete h;
            return rc;
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_live.insert(h);
    }
    *out = h;
    return ZERO1_OK;
}

int zero1_destroy(zero1_handle h)
{
    if (h == nullptr) return ZERO1_OK;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_live.erase(h)) return fail(ZERO1_EINVAL, "unknown or already destroyed handle");
    }
    DeviceGuard g(h->device);
    cudaError_t e1 = cudaDeviceSynchronize();
    cudaError_t e2 = cudaFree(h->block);
    cudaError_t e3 = h->host.staging ? cudaFree(h->host.staging) : cudaSuccess;
    if (h->bucket_sums) cudaFree(h->bucket_sums);
    if (h->ghat_bucket) cudaFree(h->ghat_bucket);
    for (cudaEvent_t ev : h->prof) cudaEventDestroy(ev);
    release_host_path(h->host);
    if (h->bctab) cudaFree(h->bctab);
    delete h;
    if (e1 != cudaSuccess) return cuda_fail(e1, "cudaDeviceSynchronize in destroy");
    if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree");
    if (e3 != cudaSuccess) return cuda_fail(e3, "cudaFree staging");
    return ZERO1_OK;
}

int zero1_step(zero1_handle h, const void *const *grad_ptrs, void *const *param_ptrs, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (h->bucket_open) return fail(ZERO1_EINVAL, "a bucketed step is open; finish it first");
    if (!grad_ptrs || !param_ptrs) return fail(ZERO1_EINVAL, "pointer array is NULL");
    for (int r = 0; r < h->world; ++r) {
        if (!grad_ptrs[r] || !param_ptrs[r]) return fail(ZERO1_EINVAL, "rank %d buffer is NULL", r);
        if (!aligned16(grad_ptrs[r]) || !aligned16(param_ptrs[r]))
            return fail(ZERO1_EALIGN, "rank %d buffer is not 16-byte aligned", r);
    }
    DeviceGuard g(h->device);
    int rc = join_host(h, static_cast<cudaStream_t>(stream));
    if (rc) return rc;
    zero1::StepLaunch s;
    s.grads = grad_ptrs;
    s.params = param_ptrs;
    s.world = h->world;
    s.n = h->n;
    s.master = h->master;
    s.m = h->m;
    s.v = h->v;
    s.ghat = h->ghat;
    s.partials = h->partials;
    s.status = h->status;
    s.sc = launch_scalars(h, h->t + 1);
    s.max_norm = h->hp.max_norm;
    s.grid_rs = h->grid_rs;
    s.grid_update = h->grid_update;
    s.moments_bf16 = h->opts.moments_bf16 != 0;
    s.decay_first = h->opts.decay_before_update != 0;
    s.clip_eps = h->opts.clip_eps;
    s.small_vpt = zero1::small_step_vpt(h->n, h->world, h->opts.small_step);
    s.dev = dev_scalars(h);
    s.stall_test = h->opts.inject_wait_timeout != 0;
    s.load_rate_gbs = zero1::load_rate_gbs(h->opts.load_phase_gbs, h->world, s.moments_bf16, h->ghat == nullptr,
                                           s.grid_update, h->num_sms);
    cudaEvent_t *ev = nullptr;
    if (h->prof_used < h->prof_capacity) ev = &h->prof[3 * (size_t)h->prof_used];
    cudaError_t e = zero1::launch_step(s, static_cast<cudaStream_t>(stream), ev);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    if (ev) h->prof_used += 1;
    h->t += 1;
    return ZERO1_OK;
}

namespace {

// The reduce-scatter + norm partial of parameters [offset, offset+count)
// (the reduce kernel in bucket mode): the gradients come from grad_ptrs,
// whose entries point at that range; the fp32 result goes to ghat + offset
// and the range's partial (sum, plain sum) to sums[2*index].  max_ctas > 0
// caps the grid.
int launch_rs_piece(zero1_ctx *h, uint64_t offset, uint64_t count, const void *const *grad_ptrs, float *ghat,
                    double *sums, int index, int max_ctas, cudaStream_t st)
{
    zero1::StepLaunch s;
    s.grads = grad_ptrs;
    s.params = nullptr;
    s.world = h->world;
    s.n = count;
    s.master = h->master;
    s.m = h->m;
    s.v = h->v;
    s.ghat = ghat + offset;
    s.partials = h->partials;
    s.status = h->status;
    s.sc = launch_scalars(h, h->t + 1);
    s.max_norm = h->hp.max_norm;
    s.clip_eps = h->opts.clip_eps;
    zero1::plan_grids(count, false, h->num_sms, &s.grid_rs, &s.grid_update);
    if (max_ctas > 0 && s.grid_rs > max_ctas) s.grid_rs = max_ctas;
    s.phase = 1;
    s.bucket_sums = sums;
    s.bucket_index = index;
    cudaError_t e = zero1::launch_step(s, st, nullptr);
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e, "kernel launch");
}

// The clip + AdamW + bf16 cast + all-gather of parameters [offset,
// offset+count) (the update kernel, c formed from the first nsums norm
// partials in order): the replicas go to param_ptrs, whose entries point at
// that range.  capturable: the step scalars come from the device counter,
// which this launch advances only if advance_t.  alone: nothing else of the
// library's runs beside this launch, so the update kernel's load phasing
// (a period set for the whole device's bandwidth) may apply; the host path's
// pieces share the device with the next step's reduces and the copies, and
// a per-bucket update with the caller's backward.
int launch_update_piece(zero1_ctx *h, uint64_t offset, uint64_t count, void *const *param_ptrs, float *ghat,
                        double *sums, int nsums, bool capturable, bool advance_t, int max_ctas, bool alone,
                        cudaStream_t st)
{
    zero1::StepLaunch s;
    s.grads = nullptr;
    s.params = param_ptrs;
    s.world = h->world;
    s.n = count;
    s.master = h->master + offset;
    s.m = h->m + offset * h->msz;
    s.v = h->v + offset * h->msz;
    s.ghat = ghat + offset;
    s.partials = h->partials;
    s.status = h->status;
    s.sc = launch_scalars(h, h->t + 1);
    s.max_norm = h->hp.max_norm;
    zero1::plan_grids(count, false, h->num_sms, &s.grid_rs, &s.grid_update);
    if (max_ctas > 0 && s.grid_update > max_ctas) s.grid_update = max_ctas;
    s.moments_bf16 = h->opts.moments_bf16 != 0;
    if (alone)
        s.load_rate_gbs =
            zero1::load_rate_gbs(h->opts.load_phase_gbs, h->world, s.moments_bf16, false, s.grid_update, h->num_sms);
    s.decay_first = h->opts.decay_before_update != 0;
    s.clip_eps = h->opts.clip_eps;
    s.phase = 2;
    s.bucket_sums = sums;
    s.nbuckets = nsums;
    if (capturable) s.dev = dev_scalars(h);
    s.advance_t = advance_t;
    cudaError_t e = zero1::launch_step(s, st, nullptr);
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e, "kernel launch");
}

constexpr uint64_t kHostMaxChunks = 1ull << 16;

// Rings, streams and events of the host-buffer steps, on first use.
int host_path_ready(zero1_ctx *h)
{
    HostPath &P = h->host;
    if (P.ready) return ZERO1_OK;
    uint64_t chunk = h->opts.host_chunk;
    if (chunk == 0) chunk = kHostSlotBytes / (2ull * (uint64_t)h->world);
    chunk = std::max<uint64_t>(kHostChunkAlign, chunk / kHostChunkAlign * kHostChunkAlign);
    chunk = std::min<uint64_t>(chunk, round_up(h->n, kHostChunkAlign));
    const uint64_t nchunks = (h->n + chunk - 1) / chunk;
    if (nchunks > kHostMaxChunks)
        return fail(ZERO1_EINVAL, "host_chunk %llu cuts n into %llu chunks (at most %llu)",
                    (unsigned long long)chunk, (unsigned long long)nchunks, (unsigned long long)kHostMaxChunks);
    cudaError_t e;
    // W <= 2: the fp32 reduce-scatter scratch the plain step does without.
    if (!h->ghat && !h->ghat_bucket &&
        (e = cudaMalloc(&h->ghat_bucket, round_up(h->padded * sizeof(float), 256))) != cudaSuccess) {
        h->ghat_bucket = nullptr;
        return cuda_fail(e, "cudaMalloc of the reduce-scatter scratch");
    }
    HostPath Q;
    Q.chunk = chunk;
    Q.nchunks = (int)nchunks;
    Q.rank_stride = round_up(chunk * 2, 256);
    const uint64_t slot_bytes = Q.rank_stride * (uint64_t)h->world;
    auto undo = [&](cudaError_t err, const char *what) {
        if (Q.staging) cudaFree(Q.staging);
        release_host_path(Q);
        return cuda_fail(err, what);
    };
    if ((e = cudaMalloc(&Q.staging, 2 * kHostSlots * slot_bytes)) != cudaSuccess) {
        Q.staging = nullptr;
        return undo(e, "cudaMalloc of the host-path rings");
    }
    if ((e = cudaMalloc(&Q.sums, 4 * nchunks * sizeof(double))) != cudaSuccess) {
        Q.sums = nullptr;
        return undo(e, "cudaMalloc of the host-path norm partials");
    }
    std::vector<cudaStream_t *> sts = {&Q.rs, &Q.upd};
    for (int i = 0; i < kHostCopyStreams; ++i) {
        sts.push_back(&Q.up[i]);
        sts.push_back(&Q.down[i]);
    }
    for (cudaStream_t *x : sts)
        if ((e = cudaStreamCreateWithFlags(x, cudaStreamNonBlocking)) != cudaSuccess) return undo(e, "cudaStreamCreate");
    std::vector<cudaEvent_t *> evs = {&Q.fork, &Q.norm_done, &Q.last};
    for (int i = 0; i < kHostSlots; ++i)
        for (cudaEvent_t *x : {&Q.up_ready[i], &Q.up_free[i], &Q.down_ready[i], &Q.down_free[i]}) evs.push_back(x);
    Q.upd_done.assign(nchunks, nullptr);
    for (auto &x : Q.upd_done) evs.push_back(&x);
    for (cudaEvent_t *x : evs)
        if ((e = cudaEventCreateWithFlags(x, cudaEventDisableTiming)) != cudaSuccess) return undo(e, "cudaEventCreate");
    Q.upd_recorded.assign(nchunks, 0);
    Q.ready = true;
    P = std::move(Q);
    return ZERO1_OK;
}

#define HOST_CHECK(call, what)                              \
    do {                                                    \
        cudaError_t err_ = (call);                          \
        if (err_ != cudaSuccess) return cuda_fail(err_, what); \
    } while (0)

// One host-buffer step: enqueue every chunk's upload, reduce, update and
// download on the handle's internal streams (see HostPath).  blocking:
// wait for all of it before returning.
int host_step(zero1_ctx *h, const void *const *host_grads, void *const *host_params, cudaStream_t st, bool blocking)
{
    int rc = host_path_ready(h);
    if (rc) return rc;
    HostPath &P = h->host;
    const int W = h->world, M = P.nchunks;
    const bool capturable = h->bctab != nullptr;
    float *ghat = h->ghat ? h->ghat : h->ghat_bucket;
    double *sums = P.sums + (size_t)P.parity * 2 * (size_t)M;
    char *ring = static_cast<char *>(P.staging);
    const uint64_t slot_bytes = P.rank_stride * (uint64_t)W;
    const void *gslot[ZERO1_MAX_WORLD];
    void *pslot[ZERO1_MAX_WORLD];

    // The step follows the caller's earlier work on `st`.
    HOST_CHECK(cudaEventRecord(P.fork, st), "cudaEventRecord");
    HOST_CHECK(cudaStreamWaitEvent(P.rs, P.fork, 0), "cudaStreamWaitEvent");
    for (int i = 0; i < M; ++i) {                    // uploads and reduces
        const uint64_t lo = (uint64_t)i * P.chunk, cnt = std::min<uint64_t>(P.chunk, h->n - lo);
        const int sl = (int)(P.up_count % kHostSlots);
        cudaStream_t u = P.up[P.up_count % kHostCopyStreams];
        char *base = ring + (uint64_t)sl * slot_bytes;
        if (P.up_used[sl]) HOST_CHECK(cudaStreamWaitEvent(u, P.up_free[sl], 0), "cudaStreamWaitEvent");
        for (int r = 0; r < W; ++r) {
            void *dst = base + (uint64_t)r * P.rank_stride;
            gslot[r] = dst;
            HOST_CHECK(cudaMemcpyAsync(dst, static_cast<const char *>(host_grads[r]) + lo * 2, cnt * 2,
                                       cudaMemcpyHostToDevice, u),
                       "gradient upload");
        }
        HOST_CHECK(cudaEventRecord(P.up_ready[sl], u), "cudaEventRecord");
        HOST_CHECK(cudaStreamWaitEvent(P.rs, P.up_ready[sl], 0), "cudaStreamWaitEvent");
        // the previous step's update of this chunk has read the scratch it overwrites
        if (P.upd_recorded[i]) HOST_CHECK(cudaStreamWaitEvent(P.rs, P.upd_done[i], 0), "cudaStreamWaitEvent");
        if ((rc = launch_rs_piece(h, lo, cnt, gslot, ghat, sums, i, 0, P.rs))) return rc;
        HOST_CHECK(cudaEventRecord(P.up_free[sl], P.rs), "cudaEventRecord");
        P.up_used[sl] = true;
        ++P.up_count;
    }
    HOST_CHECK(cudaEventRecord(P.norm_done, P.rs), "cudaEventRecord");
    HOST_CHECK(cudaStreamWaitEvent(P.upd, P.norm_done, 0), "cudaStreamWaitEvent");
    for (int i = 0; i < M; ++i) {                    // updates and downloads
        const uint64_t lo = (uint64_t)i * P.chunk, cnt = std::min<uint64_t>(P.chunk, h->n - lo);
        const int sl = (int)(P.down_count % kHostSlots);
        cudaStream_t d = P.down[P.down_count % kHostCopyStreams];
        char *base = ring + (uint64_t)(kHostSlots + sl) * slot_bytes;
        if (P.down_used[sl]) HOST_CHECK(cudaStreamWaitEvent(P.upd, P.down_free[sl], 0), "cudaStreamWaitEvent");
        for (int r = 0; r < W; ++r) pslot[r] = base + (uint64_t)r * P.rank_stride;
        if ((rc = launch_update_piece(h, lo, cnt, pslot, ghat, sums, M, capturable, i == M - 1, 0, false, P.upd)))
            return rc;
        HOST_CHECK(cudaEventRecord(P.upd_done[i], P.upd), "cudaEventRecord");
        P.upd_recorded[i] = 1;
        HOST_CHECK(cudaEventRecord(P.down_ready[sl], P.upd), "cudaEventRecord");
        HOST_CHECK(cudaStreamWaitEvent(d, P.down_ready[sl], 0), "cudaStreamWaitEvent");
        for (int r = 0; r < W; ++r)
            HOST_CHECK(cudaMemcpyAsync(static_cast<char *>(host_params[r]) + lo * 2, pslot[r], cnt * 2,
                                       cudaMemcpyDeviceToHost, d),
                       "replica download");
        HOST_CHECK(cudaEventRecord(P.down_free[sl], d), "cudaEventRecord");
        P.down_used[sl] = true;
        ++P.down_count;
    }
    HOST_CHECK(cudaEventRecord(P.last, P.upd), "cudaEventRecord");
    P.parity ^= 1;
    P.pending = true;
    h->t += 1;
    if (blocking) {
        HOST_CHECK(cudaStreamWaitEvent(st, P.last, 0), "cudaStreamWaitEvent");
        HOST_CHECK(cudaStreamSynchronize(P.upd), "cudaStreamSynchronize");
        for (cudaStream_t x : P.down) HOST_CHECK(cudaStreamSynchronize(x), "cudaStreamSynchronize");
        P.pending = false;
    }
    return ZERO1_OK;
}

int check_host_call(zero1_ctx *h, const void *const *host_grads, void *const *host_params)
{
    if (h->bucket_open) return fail(ZERO1_EINVAL, "a bucketed step is open; finish it first");
    if (!host_grads || !host_params) return fail(ZERO1_EINVAL, "pointer array is NULL");
    for (int r = 0; r < h->world; ++r)
        if (!host_grads[r] || !host_params[r]) return fail(ZERO1_EINVAL, "rank %d host buffer is NULL", r);
    return ZERO1_OK;
}

}  // namespace

int zero1_step_host(zero1_handle h, const void *const *host_grads, void *const *host_params, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    int rc = check_host_call(h, host_grads, host_params);
    if (rc) return rc;
    DeviceGuard g(h->device);
    return host_step(h, host_grads, host_params, static_cast<cudaStream_t>(stream), true);
}

int zero1_step_host_async(zero1_handle h, const void *const *host_grads, void *const *host_params, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    int rc = check_host_call(h, host_grads, host_params);
    if (rc) return rc;
    DeviceGuard g(h->device);
    return host_step(h, host_grads, host_params, static_cast<cudaStream_t>(stream), false);
}

int zero1_host_sync(zero1_handle h)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    HostPath &P = h->host;
    if (!P.ready) return ZERO1_OK;
    DeviceGuard g(h->device);
    std::vector<cudaStream_t> all(P.up, P.up + kHostCopyStreams);
    all.push_back(P.rs);
    all.push_back(P.upd);
    all.insert(all.end(), P.down, P.down + kHostCopyStreams);
    for (cudaStream_t x : all) {
        cudaError_t e = cudaStreamSynchronize(x);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    }
    P.pending = false;
    return ZERO1_OK;
}

int zero1_set_state_range(zero1_handle h, uint64_t offset, uint64_t count, const float *master,
                          const void *m, const void *v, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (!master) return fail(ZERO1_EINVAL, "master is NULL");
    if (offset > h->n || count > h->n - offset) return fail(ZERO1_EINVAL, "range outside [0, n)");
    if (count == 0) return ZERO1_OK;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = join_host(h, st);
    if (rc) return rc;
    const uint64_t bytes = count * sizeof(float);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(h->master + offset, master, bytes, cudaMemcpyDefault, st)) != cudaSuccess)
        return cuda_fail(e, "master copy");
    const uint64_t mbytes = count * h->msz;
    e = m ? cudaMemcpyAsync(h->m + offset * h->msz, m, mbytes, cudaMemcpyDefault, st)
          : cudaMemsetAsync(h->m + offset * h->msz, 0, mbytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "m copy");
    e = v ? cudaMemcpyAsync(h->v + offset * h->msz, v, mbytes, cudaMemcpyDefault, st)
          : cudaMemsetAsync(h->v + offset * h->msz, 0, mbytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "v copy");
    return ZERO1_OK;
}

int zero1_get_state_range(zero1_handle h, uint64_t offset, uint64_t count, float *master,
                          void *m, void *v, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (offset > h->n || count > h->n - offset) return fail(ZERO1_EINVAL, "range outside [0, n)");
    if (count == 0) return ZERO1_OK;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = join_host(h, st);
    if (rc) return rc;
    const uint64_t bytes = count * sizeof(float);
    cudaError_t e;
    if (master && (e = cudaMemcpyAsync(master, h->master + offset, bytes, cudaMemcpyDefault, st)) != cudaSuccess)
        return cuda_fail(e, "master copy");
    const uint64_t mbytes = count * h->msz;
    if (m && (e = cudaMemcpyAsync(m, h->m + offset * h->msz, mbytes, cudaMemcpyDefault, st)) != cudaSuccess)
        return cuda_fail(e, "m copy");
    if (v && (e = cudaMemcpyAsync(v, h->v + offset * h->msz, mbytes, cudaMemcpyDefault, st)) != cudaSuccess)
        return cuda_fail(e, "v copy");
    return ZERO1_OK;
}

int zero1_set_state(zero1_handle h, const float *master, const void *m, const void *v, uint64_t t, void *stream)
{
    int rc = zero1_set_state_range(h, 0, h && live(h) ? h->n : 0, master, m, v, stream);
    if (rc) return rc;
    h->t = t;
    if (h->bctab) {   // capturable: the device counter is the step count
        DeviceGuard g(h->device);
        const unsigned long long tt = t;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemcpyAsync(&h->status->t, &tt, sizeof tt, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "step counter write");
    }
    return ZERO1_OK;
}

int zero1_get_state(zero1_handle h, float *master, void *m, void *v, uint64_t *t, void *stream)
{
    int rc = zero1_get_state_range(h, 0, h && live(h) ? h->n : 0, master, m, v, stream);
    if (rc) return rc;
    if (t && h->bctab) {   // capturable: read the device counter (replayed graphs advance it)
        DeviceGuard g(h->device);
        unsigned long long tt = 0;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemcpyAsync(&tt, &h->status->t, sizeof tt, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "step counter read");
        h->t = tt;
    }
    if (t) *t = h->t;
    return ZERO1_OK;
}

int zero1_set_lr(zero1_handle h, double lr)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (!finite_nonneg(lr)) return fail(ZERO1_EINVAL, "lr must be finite and >= 0");
    h->hp.lr = lr;
    if (h->bctab) {   // capturable: the handle's device lr slot, after all queued work
        DeviceGuard g(h->device);
        cudaError_t e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaMemcpy(&h->status->lr, &lr, sizeof lr, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "lr write");
    }
    return ZERO1_OK;
}

int zero1_set_lr_ptr(zero1_handle h, const double *device_lr)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (!h->bctab) return fail(ZERO1_EINVAL, "zero1_set_lr_ptr needs a capturable handle");
    if (device_lr && (reinterpret_cast<uintptr_t>(device_lr) & 7u))
        return fail(ZERO1_EALIGN, "device_lr is not 8-byte aligned");
    h->lr_ptr = device_lr ? device_lr : &h->status->lr;
    return ZERO1_OK;
}

int zero1_get_grad_norm(zero1_handle h, double *norm, float *clip_coef, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    DeviceGuard g(h->device);
    zero1::DevStatus st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = join_host(h, s);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(&st, h->status, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (st.errors & zero1::kErrWaitTimeout)
        return fail(ZERO1_ECUDA, "a step kernel's pipeline wait gave up after 1 s; the state is not valid");
    if (norm) *norm = st.norm;
    if (clip_coef) *clip_coef = st.clip;
    return ZERO1_OK;
}

int zero1_layout(zero1_handle h, uint64_t *shard_len, uint64_t *padded_len, uint64_t *device_bytes)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (shard_len) *shard_len = h->shard;
    if (padded_len) *padded_len = h->padded;
    if (device_bytes) *device_bytes = h->block_bytes;
    return ZERO1_OK;
}

int zero1_profile_start(zero1_handle h, int capacity)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (capacity < 1) return fail(ZERO1_EINVAL, "capacity must be >= 1");
    DeviceGuard g(h->device);
    for (cudaEvent_t ev : h->prof) cudaEventDestroy(ev);
    h->prof.assign(3 * (size_t)capacity, nullptr);
    h->prof_capacity = h->prof_used = 0;
    for (auto &ev : h->prof) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
            for (cudaEvent_t x : h->prof)
                if (x) cudaEventDestroy(x);
            h->prof.clear();
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    h->prof_capacity = capacity;
    return ZERO1_OK;
}

int zero1_profile_stop(zero1_handle h, double *rs_norm_ms, double *update_ms, uint64_t *steps)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (h->prof_capacity == 0) return fail(ZERO1_EINVAL, "profiling was not started");
    DeviceGuard g(h->device);
    double a = 0.0, b = 0.0;
    cudaError_t e = cudaSuccess;
    if (h->prof_used > 0) e = cudaEventSynchronize(h->prof[3 * (size_t)h->prof_used - 1]);
    for (int i = 0; e == cudaSuccess && i < h->prof_used; ++i) {
        float x = 0.f, y = 0.f;
        e = cudaEventElapsedTime(&x, h->prof[3 * (size_t)i], h->prof[3 * (size_t)i + 1]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&y, h->prof[3 * (size_t)i + 1], h->prof[3 * (size_t)i + 2]);
        a += x;
        b += y;
    }
    const uint64_t used = (uint64_t)h->prof_used;
    for (cudaEvent_t ev : h->prof) cudaEventDestroy(ev);
    h->prof.clear();
    h->prof_capacity = h->prof_used = 0;
    if (e != cudaSuccess) return cuda_fail(e, "event timing");
    if (rs_norm_ms) *rs_norm_ms = a;
    if (update_ms) *update_ms = b;
    if (steps) *steps = used;
    return ZERO1_OK;
}

int zero1_step_launches(zero1_handle h, int *launches)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (!launches) return fail(ZERO1_EINVAL, "launches is NULL");
    *launches = zero1::small_step_vpt(h->n, h->world, h->opts.small_step) > 0 ? 1 : 2;
    return ZERO1_OK;
}

int zero1_profile_read(zero1_handle h, float *rs_norm_ms, float *update_ms, uint64_t capacity, uint64_t *steps)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (h->prof_capacity == 0) return fail(ZERO1_EINVAL, "profiling was not started");
    DeviceGuard g(h->device);
    cudaError_t e = cudaSuccess;
    if (h->prof_used > 0) e = cudaEventSynchronize(h->prof[3 * (size_t)h->prof_used - 1]);
    const uint64_t used = (uint64_t)h->prof_used;
    const uint64_t k = used < capacity ? used : capacity;
    for (uint64_t i = 0; e == cudaSuccess && i < k; ++i) {
        float x = 0.f, y = 0.f;
        e = cudaEventElapsedTime(&x, h->prof[3 * i], h->prof[3 * i + 1]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&y, h->prof[3 * i + 1], h->prof[3 * i + 2]);
        if (rs_norm_ms) rs_norm_ms[i] = x;
        if (update_ms) update_ms[i] = y;
    }
    if (e != cudaSuccess) return cuda_fail(e, "event timing");
    if (steps) *steps = used;
    return ZERO1_OK;
}

int zero1_bucket_begin(zero1_handle h)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (h->bucket_open) return fail(ZERO1_EINVAL, "a bucketed step is already open");
    if (h->host.pending) return fail(ZERO1_EINVAL, "host-buffer steps are in flight; call zero1_host_sync first");
    DeviceGuard g(h->device);
    cudaError_t e;
    if (!h->bucket_sums &&
        (e = cudaMalloc(&h->bucket_sums, 2 * sizeof(double) * kMaxBuckets)) != cudaSuccess) {
        h->bucket_sums = nullptr;
        return cuda_fail(e, "cudaMalloc of bucket sums");
    }
    if (!h->ghat && !h->ghat_bucket &&
        (e = cudaMalloc(&h->ghat_bucket, round_up(h->padded * sizeof(float), 256))) != cudaSuccess) {
        h->ghat_bucket = nullptr;
        return cuda_fail(e, "cudaMalloc of the reduce-scatter scratch");
    }
    h->buckets.clear();
    h->bucket_mode = 0;
    h->bucket_open = true;
    return ZERO1_OK;
}

namespace {

// The checks every bucket of an open step passes: inside [0, n), an offset
// on a vector boundary, a count that keeps the next bucket on one (only the
// bucket that ends at n may be ragged), no overlap with an earlier bucket,
// room in the table, and aligned per-rank pointers.
int check_bucket(zero1_ctx *h, uint64_t offset, uint64_t count, const void *const *ptrs, int mode)
{
    if (!h->bucket_open) return fail(ZERO1_EINVAL, "no bucketed step is open (call zero1_bucket_begin)");
    if (h->host.pending) return fail(ZERO1_EINVAL, "host-buffer steps are in flight; call zero1_host_sync first");
    if (h->bucket_mode != 0 && h->bucket_mode != mode)
        return fail(ZERO1_EINVAL, "one bucketed step uses zero1_bucket_reduce or zero1_bucket_update, not both");
    if (count == 0 || offset > h->n || count > h->n - offset)
        return fail(ZERO1_EINVAL, "bucket [%llu, +%llu) is outside [0, n)", (unsigned long long)offset,
                    (unsigned long long)count);
    if (offset % zero1::kVec) return fail(ZERO1_EINVAL, "bucket offsets must be multiples of 8");
    if (count % zero1::kVec && offset + count != h->n)
        return fail(ZERO1_EINVAL, "only the bucket that ends at n may have a count that is not a multiple of 8");
    if ((int)h->buckets.size() >= kMaxBuckets) return fail(ZERO1_EINVAL, "more than %d buckets", kMaxBuckets);
    for (const auto &b : h->buckets)
        if (offset < b.first + b.second && b.first < offset + count)
            return fail(ZERO1_EINVAL, "bucket [%llu, +%llu) overlaps an earlier bucket", (unsigned long long)offset,
                        (unsigned long long)count);
    if (!ptrs) return fail(ZERO1_EINVAL, "pointer array is NULL");
    for (int r = 0; r < h->world; ++r) {
        if (!ptrs[r]) return fail(ZERO1_EINVAL, "rank %d buffer is NULL", r);
        if (!aligned16(ptrs[r])) return fail(ZERO1_EALIGN, "rank %d buffer is not 16-byte aligned", r);
    }
    return ZERO1_OK;
}

// Reduce-scatter + norm partial of one bucket (K1 in bucket mode).
int launch_bucket_rs(zero1_ctx *h, uint64_t offset, uint64_t count, const void *const *grad_ptrs, cudaStream_t st)
{
    return launch_rs_piece(h, offset, count, grad_ptrs, h->ghat ? h->ghat : h->ghat_bucket, h->bucket_sums,
                           (int)h->buckets.size(), h->opts.bucket_ctas, st);
}

}  // namespace

int zero1_bucket_reduce(zero1_handle h, uint64_t offset, uint64_t count, const void *const *grad_ptrs, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    int rc = check_bucket(h, offset, count, grad_ptrs, 1);
    if (rc) return rc;
    DeviceGuard g(h->device);
    if ((rc = launch_bucket_rs(h, offset, count, grad_ptrs, static_cast<cudaStream_t>(stream)))) return rc;
    h->buckets.emplace_back(offset, count);
    h->bucket_mode = 1;
    return ZERO1_OK;
}

int zero1_bucket_update(zero1_handle h, uint64_t offset, uint64_t count, const void *const *grad_ptrs,
                        void *const *param_ptrs, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (h->hp.max_norm > 0.0)
        return fail(ZERO1_EINVAL, "zero1_bucket_update needs clipping off (max_norm <= 0): a clipped update "
                                  "waits for the global norm (use zero1_bucket_reduce)");
    if (h->bctab) return fail(ZERO1_EINVAL, "zero1_bucket_update is not available on a capturable handle");
    int rc = check_bucket(h, offset, count, grad_ptrs, 2);
    if (rc) return rc;
    if ((rc = check_bucket(h, offset, count, param_ptrs, 2))) return rc;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = launch_bucket_rs(h, offset, count, grad_ptrs, st))) return rc;
    // The update of the bucket's parameters right away (c = 1 without
    // clipping); CTA 0 also records the norm of the buckets so far.
    if ((rc = launch_update_piece(h, offset, count, param_ptrs, h->ghat ? h->ghat : h->ghat_bucket, h->bucket_sums,
                                  (int)h->buckets.size() + 1, false, true, h->opts.bucket_ctas, false, st)))
        return rc;
    h->buckets.emplace_back(offset, count);
    h->bucket_mode = 2;
    return ZERO1_OK;
}

int zero1_bucket_finish(zero1_handle h, void *const *param_ptrs, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    if (!h->bucket_open) return fail(ZERO1_EINVAL, "no bucketed step is open");
    const bool updated = h->bucket_mode == 2;   // every bucket already updated its parameters
    if (!updated) {
        if (!param_ptrs) return fail(ZERO1_EINVAL, "pointer array is NULL");
        for (int r = 0; r < h->world; ++r) {
            if (!param_ptrs[r]) return fail(ZERO1_EINVAL, "rank %d buffer is NULL", r);
            if (!aligned16(param_ptrs[r])) return fail(ZERO1_EALIGN, "rank %d buffer is not 16-byte aligned", r);
        }
    }
    std::vector<std::pair<uint64_t, uint64_t>> sorted = h->buckets;
    std::sort(sorted.begin(), sorted.end());
    uint64_t next = 0;
    for (const auto &b : sorted) {
        if (b.first != next) break;
        next = b.first + b.second;
    }
    if (next != h->n) {
        h->bucket_open = false;
        return fail(ZERO1_EINVAL, "the buckets must cover [0, n) exactly once; the bucketed step is abandoned");
    }
    if (updated) {
        h->bucket_open = false;
        h->t += 1;
        return ZERO1_OK;
    }
    DeviceGuard g(h->device);
    int rc = launch_update_piece(h, 0, h->n, param_ptrs, h->ghat ? h->ghat : h->ghat_bucket, h->bucket_sums,
                                 (int)h->buckets.size(), true, true, 0, true, static_cast<cudaStream_t>(stream));
    if (rc) return rc;
    h->bucket_open = false;
    h->t += 1;
    return ZERO1_OK;
}

int zero1_allreduce_sum(zero1_handle h, const void *const *in_ptrs, void *const *out_ptrs, void *stream)
{
    if (!live(h)) return fail(ZERO1_EINVAL, "invalid handle");
    DeviceGuard g(h->device);
    return zero1_allreduce(h->n, h->world, ZERO1_DTYPE_BF16, ZERO1_OP_SUM, in_ptrs, out_ptrs, nullptr, stream);
}

int zero1_shard_plan(uint64_t n, int world, uint64_t *shard_len, uint64_t *padded_len)
{
    if (n == 0) return fail(ZERO1_EINVAL, "n must be > 0");
    if (world < 1 || world > ZERO1_MAX_WORLD)
        return fail(ZERO1_EINVAL, "world must be in [1, %d], got %d", ZERO1_MAX_WORLD, world);
    const uint64_t s = round_up((n + (uint64_t)world - 1) / (uint64_t)world, zero1::kShardAlign);
    if (shard_len) *shard_len = s;
    if (padded_len) *padded_len = s * (uint64_t)world;
    return ZERO1_OK;
}

int zero1_step_scalars(const zero1_hparams *hp, int world, uint64_t t, float out[8])
{
    if (!hp || !out) return fail(ZERO1_EINVAL, "NULL pointer");
    if (t == 0) return fail(ZERO1_EINVAL, "step numbers start at 1");
    if (world < 1 || world > ZERO1_MAX_WORLD) return fail(ZERO1_EINVAL, "bad world size %d", world);
    int rc = check_hparams(hp);
    if (rc) return rc;
    const zero1::StepScalars s = step_scalars(*hp, world, t);
    const float v[8] = {s.inv_w, s.beta1, s.omb1, s.beta2, s.omb2, s.step_size, s.decay, s.eps};
    std::memcpy(out, v, sizeof v);
    return ZERO1_OK;
}

}  // extern "C"
