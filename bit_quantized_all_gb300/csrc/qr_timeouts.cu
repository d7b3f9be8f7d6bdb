// qr_timeouts.cu -- the library's count of bounded waits that ran out, and a
// self-test that makes one run out on purpose.
//
// Kernels that wait (the staged fused and Phase-1B kernels on their CTA's
// shared-memory barriers, the flag-joined two-shot on other CTAs' flags)
// give every wait a limit of one second; when a wait runs out the kernel
// adds one to this counter (one per device, held in each CUDA context that
// loads the library), stops, and returns, so the context stays usable.  The
// host reads and clears the counter in one atomic step with
// qr_wait_timeouts.  In a correct launch it never moves.
#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_launch.h"
#include "qr_pipeline.cuh"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

__device__ unsigned g_wait_timeouts;
__device__ unsigned g_wait_timeouts_taken;  // what the last read-and-clear found

// One thread waits on a barrier that nothing will ever complete.
__global__ void bounded_wait_selftest_kernel(unsigned *timeouts) {
    __shared__ __align__(8) uint64_t bar;
    qrk::mbar_init(&bar, 1);
    qrk::mbar_init_fence();
    if (!qrk::mbar_wait(&bar, 0)) atomicAdd(timeouts, 1u);
}

// Reads the counter and sets it to zero in one atomic step, so that an
// increment from a kernel still running elsewhere is either counted now or
// left for the next read, never lost.
__global__ void take_timeouts_kernel() { g_wait_timeouts_taken = atomicExch(&g_wait_timeouts, 0u); }

}  // namespace

namespace qrk {

unsigned *wait_timeout_counter(cudaError_t *err) {
    void *p = nullptr;
    if ((*err = context_symbol_address(reinterpret_cast<const void *>(&g_wait_timeouts), &p)) != cudaSuccess)
        return nullptr;
    return static_cast<unsigned *>(p);
}

}  // namespace qrk

QR_EXPORT qr_status_t qr_wait_timeouts(unsigned *count) {
    if (!count) return QR_ERR_INVALID_ARG;
    // every kernel this process has enqueued on the current device, on any
    // stream, finishes first, so its timeouts are in the count
    if (cudaDeviceSynchronize() != cudaSuccess) return QR_ERR_CUDA;
    take_timeouts_kernel<<<1, 1, 0, 0>>>();
    if (cudaGetLastError() != cudaSuccess) return QR_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeouts_taken, sizeof v) != cudaSuccess) return QR_ERR_CUDA;
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
