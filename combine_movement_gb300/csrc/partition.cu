// partition.cu -- SM partitions: streams whose kernels the hardware keeps on
// a fixed set of SMs (CUDA green contexts), for running the data movement
// on a few SMs next to other work on the rest.
//
// DeepEP's Buffer.set_num_sms ("How DeepEP Utilizes TMA Instructions for
// Minimal SM Usage on Hopper GPUs", Minimal SM Occupancy Configuration)
// limits the communication kernels to a few SMs by launching that many
// CTAs, so the remaining SMs stay free for computation. The SM budget of
// this library does the same (ep_set_num_sms). A budget alone does not say
// WHICH SMs a kernel uses, though: a kernel launched while others run goes
// to any SM with room. That is why kernel launches may not overlap the
// previous kernel's tail below the full budget by default: measured beside
// an ALU-bound kernel on the other SMs, the early-launched layout kernel (a
// small block that fits beside a foreign CTA) landed on a busy SM and the
// decode step took twice as long.
//
// A green context fixes the SMs: it is created from a split of the device's
// SMs, and every kernel launched into one of its streams runs on those SMs
// only. ep_sm_partition splits off at least num_sms SMs (rounded up to the
// device's partition granularity, 8 SMs on GB300) and makes one stream for
// them and one for the SMs that remain. Launches of this library into a
// partition stream use at most the partition's SMs and, under the default
// launch-overlap policy, those of decode-size calls may overlap the previous
// kernel's tail: nothing foreign can share those SMs. Other work goes into
// the rest stream.
//
// The driver functions are reached through the runtime's driver entry
// points, so the library links no driver library. Partitions are created
// once per (device, num_sms) and live until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/ep.h"
#include "kernels.cuh"

namespace {

using DeviceGetFn = CUresult (*)(CUdevice*, int);
using DeviceGetDevResourceFn = CUresult (*)(CUdevice, CUdevResource*, CUdevResourceType);
using SmResourceSplitByCountFn = CUresult (*)(CUdevResource*, unsigned int*, const CUdevResource*,
                                              CUdevResource*, unsigned int, unsigned int);
using DevResourceGenerateDescFn = CUresult (*)(CUdevResourceDesc*, CUdevResource*, unsigned int);
using GreenCtxCreateFn = CUresult (*)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned int);
using GreenCtxStreamCreateFn = CUresult (*)(CUstream*, CUgreenCtx, unsigned int, int);
using GreenCtxDestroyFn = CUresult (*)(CUgreenCtx);
using StreamDestroyFn = CUresult (*)(CUstream);

struct DriverApi {
    DeviceGetFn device_get = nullptr;
    DeviceGetDevResourceFn get_resource = nullptr;
    SmResourceSplitByCountFn split = nullptr;
    DevResourceGenerateDescFn gen_desc = nullptr;
    GreenCtxCreateFn green_create = nullptr;
    GreenCtxStreamCreateFn green_stream = nullptr;
    GreenCtxDestroyFn green_destroy = nullptr;
    StreamDestroyFn stream_destroy = nullptr;
    bool ok = false;
};

template <class F>
bool entry_point(const char* name, F* fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    // the functions as this runtime's version declares them (green contexts
    // came with CUDA 12.4, their streams with 12.5)
    if (cudaGetDriverEntryPointByVersion(name, &p, CUDART_VERSION, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const DriverApi& driver() {
    static const DriverApi api = [] {
        DriverApi a;
        a.ok = entry_point("cuDeviceGet", &a.device_get) &&
               entry_point("cuDeviceGetDevResource", &a.get_resource) &&
               entry_point("cuDevSmResourceSplitByCount", &a.split) &&
               entry_point("cuDevResourceGenerateDesc", &a.gen_desc) &&
               entry_point("cuGreenCtxCreate", &a.green_create) &&
               entry_point("cuGreenCtxStreamCreate", &a.green_stream) &&
               entry_point("cuGreenCtxDestroy", &a.green_destroy) &&
               entry_point("cuStreamDestroy", &a.stream_destroy);
        return a;
    }();
    return api;
}

struct Partition {
    int device;
    int requested;
    cudaStream_t stream;  // kernels run on `sms` SMs
    int sms;
    cudaStream_t rest;    // the device's other SMs (nullptr if none are left)
    int rest_sms;
};

std::mutex g_mu;
std::vector<Partition> g_parts;

// A green context on `res` and a non-blocking stream in it.
ep_status_t make_stream(const DriverApi& d, CUdevice dev, CUdevResource* res, CUgreenCtx* ctx,
                        cudaStream_t* out) {
    CUdevResourceDesc desc = nullptr;
    if (d.gen_desc(&desc, res, 1) != CUDA_SUCCESS) return EP_ERR_CUDA;
    CUgreenCtx g = nullptr;
    if (d.green_create(&g, desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) return EP_ERR_CUDA;
    CUstream s = nullptr;
    if (d.green_stream(&s, g, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
        d.green_destroy(g);
        return EP_ERR_CUDA;
    }
    *ctx = g;
    *out = reinterpret_cast<cudaStream_t>(s);
    return EP_OK;
}

}  // namespace

namespace ep {

int partition_sms(cudaStream_t stream) {
    if (stream == nullptr) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    for (const Partition& p : g_parts) {
        if (p.stream == stream) return p.sms;
        if (p.rest != nullptr && p.rest == stream) return p.rest_sms;
    }
    return 0;
}

}  // namespace ep

extern "C" ep_status_t ep_sm_partition(int num_sms, void** stream, void** rest_stream, int* sms,
                                       int* rest_sms) {
    if (num_sms < 1 || stream == nullptr) return EP_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    for (const Partition& p : g_parts) {
        if (p.device == dev && p.requested == num_sms) {
            *stream = p.stream;
            if (rest_stream != nullptr) *rest_stream = p.rest;
            if (sms != nullptr) *sms = p.sms;
            if (rest_sms != nullptr) *rest_sms = p.rest_sms;
            return EP_OK;
        }
    }
    const DriverApi& d = driver();
    if (!d.ok) return EP_ERR_UNSUPPORTED;
    int sm_count = 0;
    if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return EP_ERR_CUDA;
    if (num_sms > sm_count) return EP_ERR_UNSUPPORTED;
    CUdevice cu_dev = 0;
    if (d.device_get(&cu_dev, dev) != CUDA_SUCCESS) return EP_ERR_CUDA;
    CUdevResource all{};
    if (d.get_resource(cu_dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return EP_ERR_CUDA;
    CUdevResource group{}, remaining{};
    unsigned int groups = 1;
    if (d.split(&group, &groups, &all, &remaining, 0, static_cast<unsigned int>(num_sms)) !=
            CUDA_SUCCESS ||
        groups != 1)
        return EP_ERR_UNSUPPORTED;
    Partition p{};
    p.device = dev;
    p.requested = num_sms;
    p.sms = static_cast<int>(group.sm.smCount);
    p.rest_sms = static_cast<int>(remaining.sm.smCount);
    CUgreenCtx g_part = nullptr, g_rest = nullptr;
    ep_status_t st = make_stream(d, cu_dev, &group, &g_part, &p.stream);
    if (st != EP_OK) return st;
    if (p.rest_sms > 0) {
        st = make_stream(d, cu_dev, &remaining, &g_rest, &p.rest);
        if (st != EP_OK) {  // leave nothing half-made behind
            d.stream_destroy(reinterpret_cast<CUstream>(p.stream));
            d.green_destroy(g_part);
            return st;
        }
    }
    g_parts.push_back(p);
    *stream = p.stream;
    if (rest_stream != nullptr) *rest_stream = p.rest;
    if (sms != nullptr) *sms = p.sms;
    if (rest_sms != nullptr) *rest_sms = p.rest_sms;
    return EP_OK;
}
