// qr_reduce.cu -- launcher of the Phase-1B reduction kernels (reduce32_kernel
// and reduce16_kernel), R dispatched to a compile-time constant.
#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B, int R>
static cudaError_t run_reduce_r(const ConstPtrs &w, long long n, void *out, cudaStream_t s) {
    constexpr int U = reduce_units_per_thread<R>();  // work units per thread in flight
    const long long T = (n + kTileValues - 1) / kTileValues;
    cudaError_t err = cudaSuccess;
    if constexpr (reduce_two_threads_per_block<B, R>()) {
        const long long NH = 128 * T;
        auto kern = reduce16_kernel<B, R, U>;
        const long long units = (NH + kThreads32 * U - 1) / (kThreads32 * U);
        const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
        if (grid <= 0) return err;
        kern<<<grid, kThreads32, 0, s>>>(w, static_cast<uint8_t *>(out), NH);
    } else {
        const long long NB = 64 * T;
        auto kern = reduce32_kernel<B, R, U>;
        const long long units = (NB + kThreads32 * U - 1) / (kThreads32 * U);
        const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
        if (grid <= 0) return err;
        kern<<<grid, kThreads32, 0, s>>>(w, static_cast<uint8_t *>(out), NB);
    }
    return cudaGetLastError();
}

template <int B>
static cudaError_t run_reduce(int R, const void *const *wires, long long n, void *out, cudaStream_t s) {
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    switch (R) {
        case 1: return run_reduce_r<B, 1>(w, n, out, s);
        case 2: return run_reduce_r<B, 2>(w, n, out, s);
        case 3: return run_reduce_r<B, 3>(w, n, out, s);
        case 4: return run_reduce_r<B, 4>(w, n, out, s);
        case 5: return run_reduce_r<B, 5>(w, n, out, s);
        case 6: return run_reduce_r<B, 6>(w, n, out, s);
        case 7: return run_reduce_r<B, 7>(w, n, out, s);
        case 8: return run_reduce_r<B, 8>(w, n, out, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(int bits, int R, const void *const *wires, long long n, void *out, cudaStream_t s) {
    switch (bits) {
        case 3: return run_reduce<3>(R, wires, n, out, s);
        case 4: return run_reduce<4>(R, wires, n, out, s);
        case 6: return run_reduce<6>(R, wires, n, out, s);
        case 8: return run_reduce<8>(R, wires, n, out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qrk
