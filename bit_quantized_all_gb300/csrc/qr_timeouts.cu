// qr_timeouts.cu -- the library's count of bounded waits that ran out, and a
// self-test that makes one run out on purpose.
//
// Kernels that wait (the staged fused and Phase-1B kernels on their CTA's
// shared-memory barriers, the flag-joined two-shot on other CTAs' flags)
// give every wait a limit of one second; when a wait runs out the kernel
// adds one to this per-device counter, stops, and returns, so the context
// stays usable.  The host reads (and clears) the counter with
// qr_wait_timeouts.  In a correct launch it never moves.
#include <map>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_launch.h"
#include "qr_pipeline.cuh"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

__device__ unsigned g_wait_timeouts;

// One thread waits on a barrier that nothing will ever complete.
__global__ void bounded_wait_selftest_kernel(unsigned *timeouts) {
    __shared__ __align__(8) uint64_t bar;
    qrk::mbar_init(&bar, 1);
    qrk::mbar_init_fence();
    if (!qrk::mbar_wait(&bar, 0)) atomicAdd(timeouts, 1u);
}

}  // namespace

namespace qrk {

unsigned *wait_timeout_counter(cudaError_t *err) {
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return nullptr;
    static std::mutex mu;
    static std::map<int, unsigned *> addr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void *p = nullptr;
    if ((*err = cudaGetSymbolAddress(&p, g_wait_timeouts)) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned *>(p);
    return static_cast<unsigned *>(p);
}

}  // namespace qrk

QR_EXPORT qr_status_t qr_wait_timeouts(unsigned *count) {
    if (!count) return QR_ERR_INVALID_ARG;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof v) != cudaSuccess) return QR_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof zero) != cudaSuccess) return QR_ERR_CUDA;
    *count = v;
    return QR_OK;
}

QR_EXPORT qr_status_t qr_selftest_bounded_wait(qr_stream_t stream) {
    cudaError_t err = cudaSuccess;
    unsigned *counter = qrk::wait_timeout_counter(&err);
    if (!counter) return QR_ERR_CUDA;
    bounded_wait_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(counter);
    return cudaGetLastError() == cudaSuccess ? QR_OK : QR_ERR_CUDA;
}
