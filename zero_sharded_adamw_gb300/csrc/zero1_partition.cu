// zero1_partition.cu -- two streams on disjoint sets of the device's SMs.
//
// The bucketed step ("Stanford CS336 Lecture 7 close reading: Parallelism
// (part 1)", 5.3: each layer's gradients are reduced as the backward
// produces them; "Parallel training", "Data parallel and ZeRO": buckets,
// communication hidden behind the backward) runs its reduce-scatters beside
// the caller's backward.  On Blackwell the library GEMMs of a backward are
// persistent kernels that hold every SM until they end, so a concurrent
// bucket reduce finds no SM to run on.  A green context owns a fixed group
// of SMs: work launched on a stream of that context runs only on those SMs.
// zero1_sm_partition_create splits the current device's SMs into two such
// groups and returns a stream on each; a caller runs its backward on one
// and the bucket reduces on the other.
//
// The driver functions are fetched through the runtime's entry-point query
// (the library does not link the driver library itself).  Every call
// returns an error code; nothing here changes a device setting that
// outlives the process (the green contexts are destroyed with the partition).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <new>

#include "zero1.h"
#include "zero1_internal.h"

namespace {

int pfail(int code, const char *fmt, ...)
{
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    zero1::set_error_message(msg);
    return code;
}

typedef CUresult (*DeviceGetFn)(CUdevice *, int);
typedef CUresult (*DevResourceFn)(CUdevice, CUdevResource *, CUdevResourceType);
typedef CUresult (*SplitFn)(CUdevResource *, unsigned int *, const CUdevResource *, CUdevResource *, unsigned int,
                            unsigned int);
typedef CUresult (*DescFn)(CUdevResourceDesc *, CUdevResource *, unsigned int);
typedef CUresult (*GreenCreateFn)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int);
typedef CUresult (*GreenDestroyFn)(CUgreenCtx);
typedef CUresult (*GreenStreamFn)(CUstream *, CUgreenCtx, unsigned int, int);
typedef CUresult (*StreamDestroyFn)(CUstream);

struct Driver {
    bool tried = false, ok = false;
    char missing[128] = "";        // the first entry point the driver did not provide
    DeviceGetFn device_get = nullptr;
    DevResourceFn dev_resource = nullptr;
    SplitFn split = nullptr;
    DescFn desc = nullptr;
    GreenCreateFn green_create = nullptr;
    GreenDestroyFn green_destroy = nullptr;
    GreenStreamFn green_stream = nullptr;
    StreamDestroyFn stream_destroy = nullptr;
};
std::mutex g_mu;
Driver g_drv;

// The driver's entry point `name` in the version this library is built
// against; on failure the name and the query's answer go to g_drv.missing.
template <typename F>
bool fetch(const char *name, F *out)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion(name, &p, CUDART_VERSION, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr) {
        snprintf(g_drv.missing, sizeof g_drv.missing, "%s (runtime %d, query %d)", name, (int)e, (int)q);
        return false;
    }
    *out = reinterpret_cast<F>(p);
    return true;
}

const Driver *driver()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_drv.tried) {
        g_drv.tried = true;
        g_drv.ok = fetch("cuDeviceGet", &g_drv.device_get) &&
                   fetch("cuDeviceGetDevResource", &g_drv.dev_resource) &&
                   fetch("cuDevSmResourceSplitByCount", &g_drv.split) &&
                   fetch("cuDevResourceGenerateDesc", &g_drv.desc) &&
                   fetch("cuGreenCtxCreate", &g_drv.green_create) &&
                   fetch("cuGreenCtxDestroy", &g_drv.green_destroy) &&
                   fetch("cuGreenCtxStreamCreate", &g_drv.green_stream) &&
                   fetch("cuStreamDestroy", &g_drv.stream_destroy);
    }
    return g_drv.ok ? &g_drv : nullptr;
}

struct Partition {
    CUgreenCtx ctx[2] = {nullptr, nullptr};
    CUstream stream[2] = {nullptr, nullptr};
};

void release(const Driver *d, Partition *p)
{
    for (int i = 0; i < 2; ++i) {
        if (p->stream[i]) d->stream_destroy(p->stream[i]);
        if (p->ctx[i]) d->green_destroy(p->ctx[i]);
    }
    delete p;
}

}  // namespace

extern "C" int zero1_sm_partition_create(int sms_a, zero1_sm_partition *out)
{
    if (!out) return pfail(ZERO1_EINVAL, "out is NULL");
    *out = zero1_sm_partition{};
    if (sms_a < 1) return pfail(ZERO1_EINVAL, "sms_a must be >= 1, got %d", sms_a);
    int ord = 0, total = 0;
    cudaError_t e = cudaGetDevice(&ord);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&total, cudaDevAttrMultiProcessorCount, ord);
    if (e != cudaSuccess) return pfail(ZERO1_ENODEV, "no CUDA device (%s)", cudaGetErrorString(e));
    if (sms_a >= total) return pfail(ZERO1_EINVAL, "sms_a = %d leaves none of the %d SMs for the second group", sms_a, total);
    const Driver *d = driver();
    if (!d) return pfail(ZERO1_ECUDA, "the driver does not provide green contexts: %s", g_drv.missing);
    CUdevice dev;
    CUdevResource all{}, group{}, rest{};
    unsigned int ngroups = 1;
    CUresult r = d->device_get(&dev, ord);
    if (r == CUDA_SUCCESS) r = d->dev_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM);
    if (r == CUDA_SUCCESS) r = d->split(&group, &ngroups, &all, &rest, 0, (unsigned)sms_a);
    if (r != CUDA_SUCCESS || ngroups != 1)
        return pfail(ZERO1_ECUDA, "splitting the device's SMs failed (driver error %d)", (int)r);
    if (rest.sm.smCount == 0)
        return pfail(ZERO1_EINVAL, "%d SMs rounded up to the partition granularity leave none for the second group",
                     sms_a);
    Partition *p = new (std::nothrow) Partition;
    if (!p) return pfail(ZERO1_ENOMEM, "host allocation failed");
    CUdevResource *res[2] = {&group, &rest};
    for (int i = 0; i < 2; ++i) {
        CUdevResourceDesc desc;
        r = d->desc(&desc, res[i], 1);
        if (r == CUDA_SUCCESS) r = d->green_create(&p->ctx[i], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM);
        if (r == CUDA_SUCCESS) r = d->green_stream(&p->stream[i], p->ctx[i], CU_STREAM_NON_BLOCKING, 0);
        if (r != CUDA_SUCCESS) {
            release(d, p);
            return pfail(ZERO1_ECUDA, "creating green context %d failed (driver error %d)", i, (int)r);
        }
    }
    out->stream_a = p->stream[0];
    out->stream_b = p->stream[1];
    out->sms_a = (int)group.sm.smCount;
    out->sms_b = (int)rest.sm.smCount;
    out->opaque = p;
    return ZERO1_OK;
}

extern "C" int zero1_sm_partition_destroy(zero1_sm_partition *part)
{
    if (!part || !part->opaque) return ZERO1_OK;
    const Driver *d = driver();
    if (!d) return pfail(ZERO1_ECUDA, "the driver does not provide green contexts");
    Partition *p = static_cast<Partition *>(part->opaque);
    // Work still queued on either stream finishes before its green context
    // goes away; a failed wait is reported, and the partition released all
    // the same.
    cudaError_t werr = cudaSuccess;
    for (int i = 0; i < 2; ++i) {
        const cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(p->stream[i]));
        if (e != cudaSuccess && werr == cudaSuccess) werr = e;
    }
    release(d, p);
    *part = zero1_sm_partition{};
    if (werr != cudaSuccess)
        return pfail(ZERO1_ECUDA, "waiting for the partition's streams failed: %s", cudaGetErrorString(werr));
    return ZERO1_OK;
}
