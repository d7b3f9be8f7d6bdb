// qr_grid.cu -- launch-shape choice shared by every launcher: how many CTAs
// a grid-stride kernel gets (from the SM count and the kernel's occupancy,
// cached per device and kernel).
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "qr_launch.h"

namespace qrk {

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
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({dev, kernel});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) done[{dev, kernel}] = bytes;
    return err;
}

}  // namespace qrk
