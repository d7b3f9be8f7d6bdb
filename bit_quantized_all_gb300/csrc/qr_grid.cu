// qr_grid.cu -- launch-shape choice shared by every launcher: how many CTAs
// a grid-stride kernel gets (from the SM count and the kernel's occupancy,
// cached per device and kernel), and the per-context state every launcher
// relies on (kernel attributes, symbol addresses), cached per CUDA context.
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "qr_launch.h"

namespace qrk {

namespace {

// cuCtxGetCurrent / cuCtxGetId, looked up through the runtime (the library
// does not link the driver library itself).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct DriverCtxApi {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    cudaError_t err = cudaSuccess;
};

const DriverCtxApi &driver_ctx_api() {
    static const DriverCtxApi api = [] {
        DriverCtxApi a;
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1 = cudaDriverEntryPointSymbolNotFound, r2 = r1;
        a.err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1);
        if (a.err == cudaSuccess)
            a.err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2);
        if (a.err == cudaSuccess && (r1 != cudaDriverEntryPointSuccess || r2 != cudaDriverEntryPointSuccess))
            a.err = cudaErrorNotSupported;
        if (a.err == cudaSuccess) {
            a.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
            a.get_id = reinterpret_cast<CtxGetIdFn>(q);
        }
        return a;
    }();
    return api;
}

}  // namespace

unsigned long long context_id(cudaError_t *err) {
    const DriverCtxApi &api = driver_ctx_api();
    if ((*err = api.err) != cudaSuccess) return 0;
    CUcontext ctx = nullptr;
    if (api.get_current(&ctx) != CUDA_SUCCESS) {
        *err = cudaErrorInvalidResourceHandle;
        return 0;
    }
    if (!ctx) {  // the runtime has not made the current device's context current yet
        int dev = 0;
        if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
        if ((*err = cudaSetDevice(dev)) != cudaSuccess) return 0;  // initializes it
        if (api.get_current(&ctx) != CUDA_SUCCESS || !ctx) {
            *err = cudaErrorInvalidResourceHandle;
            return 0;
        }
    }
    unsigned long long id = 0;
    if (api.get_id(ctx, &id) != CUDA_SUCCESS) {
        *err = cudaErrorInvalidResourceHandle;
        return 0;
    }
    return id + 1;  // never 0
}

cudaError_t context_symbol_address(const void *symbol, void **ptr) {
    cudaError_t err = cudaSuccess;
    const unsigned long long ctx = context_id(&err);
    if (!ctx) return err;
    static std::mutex mu;
    static std::map<std::pair<unsigned long long, const void *>, void *> addr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find({ctx, symbol});
    if (it != addr.end()) {
        *ptr = it->second;
        return cudaSuccess;
    }
    void *p = nullptr;
    if ((err = cudaGetSymbolAddress(&p, symbol)) != cudaSuccess) return err;
    addr[{ctx, symbol}] = p;
    *ptr = p;
    return cudaSuccess;
}

int grid_for(const void *kernel, int threads, long long tiles, int ctas, int waves, cudaError_t *err) {
    *err = cudaSuccess;
    if (tiles <= 0) return 0;
    if (ctas > 0) return static_cast<int>(tiles < ctas ? tiles : ctas);
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> resident;  // (device, kernel) -> CTAs per wave
    int wave = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = resident.find({dev, kernel});
        if (it != resident.end()) wave = it->second;
    }
    if (wave == 0) {
        int sms = 0, per_sm = 0;
        if ((*err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return 0;
        if ((*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0)) != cudaSuccess)
            return 0;
        wave = sms * (per_sm > 0 ? per_sm : 1);
        std::lock_guard<std::mutex> lock(mu);
        resident[{dev, kernel}] = wave;
    }
    const long long want = static_cast<long long>(wave) * (waves > 0 ? waves : 1);
    return static_cast<int>(tiles < want ? tiles : want);
}

int sm_count(cudaError_t *err) {
    *err = cudaSuccess;
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
    static std::mutex mu;
    static std::map<int, int> sms;
    std::lock_guard<std::mutex> lock(mu);
    auto it = sms.find(dev);
    if (it != sms.end()) return it->second;
    int v = 0;
    if ((*err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return 0;
    sms[dev] = v;
    return v;
}

cudaError_t allow_dynamic_smem(const void *kernel, int bytes) {
    cudaError_t err = cudaSuccess;
    const unsigned long long ctx = context_id(&err);  // the attribute lives in the context
    if (!ctx) return err;
    static std::mutex mu;
    static std::map<std::pair<unsigned long long, const void *>, int> done;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({ctx, kernel});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) done[{ctx, kernel}] = bytes;
    return err;
}

}  // namespace qrk
