// qr_allreduce16.cuh -- launchers of the 16-values-per-thread fused kernels:
// the register-fed allreduce16_kernel and the staged kernel with QrTile
// (qr_staged.cuh), and the choice between them; R dispatched to a
// compile-time constant.  Each qr_allreduce16_b<B>.cu instantiates them for
// one code width so that the widths compile in parallel.
#pragma once

#include "qr_kernels.cuh"
#include "qr_launch.h"
#include "qr_staged.cuh"

namespace qrk {

template <int B, int DT, int R>
static cudaError_t run_allreduce16_r(const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    if (ctas == 0) {  // the library's choice of kernel
        cudaError_t err = cudaSuccess;
        if (take_staged(R, n, false, &err)) return launch_staged<QrTile<B, DT>, R>(xp, n, y, 0, s);
        if (err != cudaSuccess) return err;
    }
    auto kern = allreduce16_kernel<B, DT, R>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads16, T, ctas, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads16, 0, s, xp, n, static_cast<uint16_t *>(y), T);
}

template <int B, int DT>
cudaError_t run_allreduce16_staged(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    return launch_staged<QrTile<B, DT>>(R, xp, n, y, ctas, s);
}

template <int B, int DT>
cudaError_t run_allreduce16(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    switch (R) {
        case 1: return run_allreduce16_r<B, DT, 1>(xp, n, y, ctas, s);
        case 2: return run_allreduce16_r<B, DT, 2>(xp, n, y, ctas, s);
        case 3: return run_allreduce16_r<B, DT, 3>(xp, n, y, ctas, s);
        case 4: return run_allreduce16_r<B, DT, 4>(xp, n, y, ctas, s);
        case 5: return run_allreduce16_r<B, DT, 5>(xp, n, y, ctas, s);
        case 6: return run_allreduce16_r<B, DT, 6>(xp, n, y, ctas, s);
        case 7: return run_allreduce16_r<B, DT, 7>(xp, n, y, ctas, s);
        case 8: return run_allreduce16_r<B, DT, 8>(xp, n, y, ctas, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qrk
