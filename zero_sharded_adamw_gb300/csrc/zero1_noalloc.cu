// zero1_noalloc.cu -- zero1_step_noalloc: one ZeRO-1 step that allocates no
// device memory.
//
// Who needs it: callers that cannot call cudaMalloc.  A framework whose
// caching allocator has already reserved the device's memory (a library
// cudaMalloc would fail or break the framework's budget), a plug-in whose
// host fixes the device memory it may use up front, or a loop that cannot
// afford the implicit device synchronisation cudaMalloc/cudaFree bring.
// Such a caller owns every buffer the step reads or writes -- gradients,
// replicas and the fp32 master/m/v -- and passes them in; no handle (whose
// creation allocates) is involved.
//
// The step's scratch (the fp32 reduce-scatter result, the per-CTA norm
// partials and the 32-byte norm status) lives in one file-scope device
// array, g_noalloc_scratch, of fixed size: it is part of the library image,
// so every GPU that loads the library holds it (about 16.1 MiB) until the
// process exits.  It bounds n at kNoAllocMaxN = 4,194,304 parameters.
//
// Host code must not hand the array's name to a kernel: on the host the
// name is a stand-in, not a device address.  The first call on each device
// (with that device current) looks the address up with cudaGetSymbolAddress
// and caches it together with the identity of the CUDA context it was
// looked up in; that first call should therefore come before any stream
// capture.  Later calls compare the current context's identity with the
// cached one (two driver queries, no device work) and look the address up
// again when it changed, e.g. after cudaDeviceReset destroyed the context
// and a new one loaded the module, possibly at another address.  Every call
// shares the one array and its contents survive from call to call, so the
// parts that must start at zero are cleared on the stream at the start of
// each call; calls whose work overlaps on the GPU (different streams, or
// different host threads) race on the array.
//
// The status block in the scratch also carries the sticky error bit that a
// kernel pipeline wait sets when it gives up after its 1 s limit.  Each call
// clears it with the rest of the status, and nothing on this path reads it
// back, so such a timeout is not reported here (the handle-based step
// reports it through zero1_get_grad_norm).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "zero1.h"
#include "zero1_internal.h"
#include "zero1_policy.h"

namespace {

constexpr uint64_t kNoAllocMaxN = uint64_t(1) << 22;          // parameters
constexpr size_t kGhatBytes = kNoAllocMaxN * sizeof(float);    // 16 MiB
constexpr size_t kPartialDoubles = 8192;                       // 2 * 4096 CTAs
constexpr size_t kPartialBytes = kPartialDoubles * sizeof(double);
constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes = kGhatBytes + kPartialBytes + kStatusBytes;

// The step's scratch.  Zero-initialised at module load; see above.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
// Per device: the scratch address, the context it was looked up in
// (cuCtxGetId's identity, unique for the life of the process) and the SM count.
unsigned char *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// The two driver queries that identify the current context, fetched from the
// driver through the runtime (the library does not link libcuda itself).
// The handle types are opaque pointers; the return codes are CUresult,
// where 0 is success.
typedef int (*CtxGetCurrentFn)(void **ctx);
typedef int (*CtxGetIdFn)(void *ctx, unsigned long long *id);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_ctx_fns_tried = false;

// The identity of the calling thread's current context, or 0 if there is
// none yet or the driver queries are unavailable (then the address is
// looked up on every call).  Called with g_setup_mu held.
unsigned long long current_context_id()
{
    if (!g_ctx_fns_tried) {
        g_ctx_fns_tried = true;
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
        }
    }
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != 0 || ctx == nullptr || g_ctx_get_id(ctx, &id) != 0) return 0;
    return id;
}

// Record the message for zero1_last_error() and return the code.
int nfail(int code, const char *fmt, ...)
{
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    zero1::set_error_message(msg);
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device and context, with that device current: the scratch's
// device address and the SM count.
int setup_device(int dev, unsigned char **scratch, int *num_sms)
{
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (dev < 0 || dev >= kMaxDevices) return nfail(ZERO1_ENODEV, "device ordinal %d out of range", dev);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        int major = 0, minor = 0, sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return nfail(ZERO1_ECUDA, "device query: %s", cudaGetErrorString(e));
        if (major != 10 || minor != 3)
            return nfail(ZERO1_ENODEV, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess || addr == nullptr)
            return nfail(ZERO1_ECUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = static_cast<unsigned char *>(addr);
        g_num_sms[dev] = sms;
        // The lookup made the device's primary context current if no context
        // was; record the context the address belongs to.
        g_scratch_ctx[dev] = ctx != 0 ? ctx : current_context_id();
    }
    *scratch = g_scratch_addr[dev];
    *num_sms = g_num_sms[dev];
    return ZERO1_OK;
}

}  // namespace

extern "C" int zero1_step_noalloc(uint64_t n, int world, const zero1_hparams *hp, uint64_t t,
                                  const void *const *grad_ptrs, void *const *param_ptrs,
                                  float *master, float *m, float *v, void *stream)
{
    if (n == 0 || n > kNoAllocMaxN)
        return nfail(ZERO1_EINVAL, "zero1_step_noalloc: n = %llu is outside [1, %llu] (the fixed scratch "
                     "holds %llu parameters; use zero1_create/zero1_step for larger n)",
                     (unsigned long long)n, (unsigned long long)kNoAllocMaxN, (unsigned long long)kNoAllocMaxN);
    if (world < 1 || world > ZERO1_MAX_WORLD)
        return nfail(ZERO1_EINVAL, "world must be in [1, %d], got %d", ZERO1_MAX_WORLD, world);
    if (!hp || !grad_ptrs || !param_ptrs || !master || !m || !v)
        return nfail(ZERO1_EINVAL, "NULL pointer argument");
    if (t == 0) return nfail(ZERO1_EINVAL, "step numbers start at 1");
    if (!aligned16(master) || !aligned16(m) || !aligned16(v))
        return nfail(ZERO1_EALIGN, "master, m and v must be 16-byte aligned");
    for (int r = 0; r < world; ++r) {
        if (!grad_ptrs[r] || !param_ptrs[r]) return nfail(ZERO1_EINVAL, "rank %d buffer is NULL", r);
        if (!aligned16(grad_ptrs[r]) || !aligned16(param_ptrs[r]))
            return nfail(ZERO1_EALIGN, "rank %d buffer is not 16-byte aligned", r);
    }
    float sc[8];
    if (zero1_step_scalars(hp, world, t, sc) != ZERO1_OK)
        return ZERO1_EINVAL;                  // message already recorded

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return nfail(ZERO1_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    unsigned char *scratch = nullptr;
    int num_sms = 0;
    int rc = setup_device(dev, &scratch, &num_sms);
    if (rc) return rc;

    zero1::StepLaunch s;
    s.grads = grad_ptrs;
    s.params = param_ptrs;
    s.world = world;
    s.n = n;
    s.master = master;
    s.m = m;
    s.v = v;
    const bool reread = world <= 2;           // the same choice zero1_create makes
    s.ghat = reread ? nullptr : reinterpret_cast<float *>(scratch);
    s.partials = reinterpret_cast<double *>(scratch + kGhatBytes);
    s.status = reinterpret_cast<zero1::DevStatus *>(scratch + kGhatBytes + kPartialBytes);
    s.sc = zero1::StepScalars{sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};
    s.max_norm = hp->max_norm;
    s.small_vpt = zero1::small_step_vpt(n, world, 0);
    zero1::plan_grids(n, reread, num_sms, &s.grid_rs, &s.grid_update);
    s.load_rate_gbs = zero1::load_rate_gbs(0.0, world, false, reread, s.grid_update, num_sms);
    if ((size_t)s.grid_rs * 2 > kPartialDoubles)
        return nfail(ZERO1_EINVAL, "grid of %d CTAs exceeds the fixed partials scratch", s.grid_rs);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The norm status (and its last-CTA ticket) must start at zero.
    if ((e = cudaMemsetAsync(s.status, 0, sizeof(zero1::DevStatus), st)) != cudaSuccess)
        return nfail(ZERO1_ECUDA, "clearing the scratch status: %s", cudaGetErrorString(e));
    if ((e = zero1::launch_step(s, st, nullptr)) != cudaSuccess)
        return nfail(ZERO1_ECUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ZERO1_OK;
}
