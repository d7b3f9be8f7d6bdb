// qr_reduce.cu -- launcher of the Phase-1B reduction kernel (reduce_kernel).
#include "qr_kernels.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B>
static cudaError_t run_reduce(int R, const void *const *wires, long long n, void *out, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    auto kern = reduce_kernel<B>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads, T, 0, &err);
    if (grid <= 0) return err;
    kern<<<grid, kThreads, 0, s>>>(w, R, static_cast<uint8_t *>(out), T);
    return cudaGetLastError();
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
