// qr_allreduce16.cuh -- launcher of the 16-values-per-thread fused kernel
// (allreduce16_kernel), dispatching R to a compile-time constant.  Each
// qr_allreduce16_b<B>.cu instantiates it for one code width so that the
// widths compile in parallel.
#pragma once

#include "qr_kernels.cuh"
#include "qr_launch.h"

namespace qrk {

// Launch shape of the staged kernel for R ranks: five groups of 128 threads
// (20 warps: at 96 registers a thread, the most that five warps in each of
// the SM's four register quadrants allow), each with as many stages (at most
// 4) as fit in 224 KiB of shared memory at R * 4 KiB per stage; each group
// sums the first R/2 ranks straight from shared memory and copies the other
// R/2 into registers before it releases the stage.  Measured on GB300 at
// R=8 (2^27 bf16 values per rank, INT4 and INT3, back-to-back launches):
//   groups x early ranks:  5 x 0: 6.65 TB/s   5 x 2: 6.92   5 x 4: 6.99
//                          5 x 6: 6.84        6 x 4: 6.75   6 x 6: 6.98
//                          7 x 4: 6.50        7 x 6: 6.65   4 x 4: 6.75
// (one to three groups with deeper rings: 4.4-5.5 TB/s, too few warps to
// issue the arithmetic); the register-fed kernel 6.36 TB/s.
template <int R>
struct StagedShape {
    static constexpr int kGroups = 5;
    static constexpr int kFit = (224 * 1024) / (kGroups * R * kTileValues * 2);
    static constexpr int kStages = kFit >= 4 ? 4 : kFit;  // per group
    static constexpr int kSmemBytes = kGroups * kStages * R * kTileValues * 2;
    static constexpr int kEarlyRanks = R / 2;  // summed from shared memory before the stage is released
    static_assert(kStages >= 1, "at least one stage per group");
};

// Where qr_allreduce takes the staged kernel: full tiles per SM from which it
// was faster than the register-fed kernel in back-to-back launches on GB300
// (INT4, bf16, 2^20..2^27 values per rank).  With R <= 2 the register-fed
// kernel already has enough warps and stays ahead at every size; at R = 3
// the staged kernel wins from ~200 tiles per SM, at R >= 4 from ~50 (at
// 2^27 values per rank: +14% at R=4 and R=6, +7% at R=8).
template <int R>
constexpr long long staged_min_tiles_per_sm() {
    return R <= 2 ? -1 : (R == 3 ? 128 : 48);
}

template <int B, int DT, int R>
static cudaError_t run_allreduce16_staged_r(const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    using Shape = StagedShape<R>;
    auto kern = allreduce16_staged_kernel<B, DT, R, Shape::kGroups, Shape::kStages, Shape::kEarlyRanks>;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (sms <= 0) return err;
    if ((err = allow_dynamic_smem(reinterpret_cast<const void *>(kern), Shape::kSmemBytes)) != cudaSuccess)
        return err;
    unsigned *timeouts = wait_timeout_counter(&err);
    if (!timeouts) return err;
    const long long full_tiles = n / kTileValues;
    long long grid = ctas > 0 ? ctas : sms;  // persistent: at most one CTA per SM
    if (grid > sms) grid = sms;
    if (grid > full_tiles) grid = full_tiles;
    if (grid < 1) grid = 1;  // a message shorter than one tile: CTA 0 does the ragged tile
    kern<<<static_cast<int>(grid), 128 * Shape::kGroups, Shape::kSmemBytes, s>>>(
        xp, n, static_cast<uint16_t *>(y), full_tiles, timeouts);
    return cudaGetLastError();
}

template <int B, int DT, int R>
static cudaError_t run_allreduce16_r(const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    if (ctas == 0 && staged_min_tiles_per_sm<R>() > 0) {  // the library's choice of kernel
        cudaError_t err = cudaSuccess;
        const int sms = sm_count(&err);
        if (sms <= 0) return err;
        if (n / kTileValues >= staged_min_tiles_per_sm<R>() * sms)
            return run_allreduce16_staged_r<B, DT, R>(xp, n, y, 0, s);
    }
    auto kern = allreduce16_kernel<B, DT, R>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads16, T, ctas, 4, &err);
    if (grid <= 0) return err;
    kern<<<grid, kThreads16, 0, s>>>(xp, n, static_cast<uint16_t *>(y), T);
    return cudaGetLastError();
}

template <int B, int DT>
cudaError_t run_allreduce16_staged(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    switch (R) {
        case 1: return run_allreduce16_staged_r<B, DT, 1>(xp, n, y, ctas, s);
        case 2: return run_allreduce16_staged_r<B, DT, 2>(xp, n, y, ctas, s);
        case 3: return run_allreduce16_staged_r<B, DT, 3>(xp, n, y, ctas, s);
        case 4: return run_allreduce16_staged_r<B, DT, 4>(xp, n, y, ctas, s);
        case 5: return run_allreduce16_staged_r<B, DT, 5>(xp, n, y, ctas, s);
        case 6: return run_allreduce16_staged_r<B, DT, 6>(xp, n, y, ctas, s);
        case 7: return run_allreduce16_staged_r<B, DT, 7>(xp, n, y, ctas, s);
        case 8: return run_allreduce16_staged_r<B, DT, 8>(xp, n, y, ctas, s);
    }
    return cudaErrorInvalidValue;
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
