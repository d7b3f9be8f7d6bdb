// qr_fc_allreduce.cuh -- launchers of the fused Flash Communication all-reduce
// (fc_allreduce_kernel, and the staged kernel with FcTile), R dispatched to a
// compile-time constant.  Each qr_fc_allreduce_<rs><ag>.cu instantiates one
// width pair.
#pragma once

#include <cstdint>

#include "qr_kernels_fc.cuh"
#include "qr_launch.h"
#include "qr_staged.cuh"

namespace qrk {

template <int BRS, int BAG, int DT, int R, bool A32>
static cudaError_t run_fc_allreduce_r(const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    if constexpr (A32) {
        if (ctas == 0) {  // the library's choice of kernel
            cudaError_t err = cudaSuccess;
            if (take_staged(R, n, true, &err)) return launch_staged<FcTile<BRS, BAG, DT>, R>(xp, n, y, 0, s);
            if (err != cudaSuccess) return err;
        }
    }
    auto kern = fc_allreduce_kernel<BRS, BAG, DT, R, A32>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreadsFc, T, ctas, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreadsFc, 0, s, xp, n, static_cast<uint16_t *>(y), T);
}

template <int BRS, int BAG, int DT, bool A32>
static cudaError_t run_fc_allreduce_a(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    switch (R) {
        case 1: return run_fc_allreduce_r<BRS, BAG, DT, 1, A32>(xp, n, y, ctas, s);
        case 2: return run_fc_allreduce_r<BRS, BAG, DT, 2, A32>(xp, n, y, ctas, s);
        case 3: return run_fc_allreduce_r<BRS, BAG, DT, 3, A32>(xp, n, y, ctas, s);
        case 4: return run_fc_allreduce_r<BRS, BAG, DT, 4, A32>(xp, n, y, ctas, s);
        case 5: return run_fc_allreduce_r<BRS, BAG, DT, 5, A32>(xp, n, y, ctas, s);
        case 6: return run_fc_allreduce_r<BRS, BAG, DT, 6, A32>(xp, n, y, ctas, s);
        case 7: return run_fc_allreduce_r<BRS, BAG, DT, 7, A32>(xp, n, y, ctas, s);
        case 8: return run_fc_allreduce_r<BRS, BAG, DT, 8, A32>(xp, n, y, ctas, s);
    }
    return cudaErrorInvalidValue;
}

// The staged kernel at any size (every pointer 32-byte aligned).
template <int BRS, int BAG>
cudaError_t run_fc_allreduce_staged(int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                    cudaStream_t s) {
    ConstPtrs xp{};
    for (int r = 0; r < R; ++r) xp.p[r] = x[r];
    return dtype ? launch_staged<FcTile<BRS, BAG, 1>>(R, xp, n, y, ctas, s)
                 : launch_staged<FcTile<BRS, BAG, 0>>(R, xp, n, y, ctas, s);
}

template <int BRS, int BAG>
cudaError_t run_fc_allreduce(int dtype, int R, const void *const *x, long long n, void *y, int ctas, cudaStream_t s) {
    ConstPtrs xp{};
    bool a32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
    for (int r = 0; r < R; ++r) {
        xp.p[r] = x[r];
        a32 = a32 && (reinterpret_cast<uintptr_t>(x[r]) & 31u) == 0;
    }
    if (dtype)
        return a32 ? run_fc_allreduce_a<BRS, BAG, 1, true>(R, xp, n, y, ctas, s)
                   : run_fc_allreduce_a<BRS, BAG, 1, false>(R, xp, n, y, ctas, s);
    return a32 ? run_fc_allreduce_a<BRS, BAG, 0, true>(R, xp, n, y, ctas, s)
               : run_fc_allreduce_a<BRS, BAG, 0, false>(R, xp, n, y, ctas, s);
}

}  // namespace qrk
