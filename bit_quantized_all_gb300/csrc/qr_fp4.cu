// qr_fp4.cu -- launchers of the FP4 codec's kernels (qr_kernels_fp4.cuh): the
// send path, the receive path, Phase-1B on the staged reduce kernel and the
// fused all-reduce on the staged fused kernel, R dispatched to a
// compile-time constant.
#include <cstdint>

#include "qr_kernels_fp4.cuh"
#include "qr_launch.h"
#include "qr_staged.cuh"

namespace qrk {

template <int DT>
static cudaError_t run_fp4_encode(const void *x, long long n, void *wire, cudaStream_t s) {
    const long long NB = 64 * ((n + kTileValues - 1) / kTileValues);
    auto kern = fp4_encode_kernel<DT>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, (NB + kThreads32 - 1) / kThreads32,
                              0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint16_t *>(x), n,
                          static_cast<uint8_t *>(wire), NB);
}

cudaError_t launch_fp4_encode(int dtype, const void *x, long long n, void *wire, cudaStream_t s) {
    return dtype ? run_fp4_encode<1>(x, n, wire, s) : run_fp4_encode<0>(x, n, wire, s);
}

template <int DT>
static cudaError_t run_fp4_decode(const void *wire, long long n, void *y, cudaStream_t s) {
    const long long NH = 128 * ((n + kTileValues - 1) / kTileValues);  // half-blocks
    const bool y32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
    auto kern = y32 ? fp4_decode_kernel<DT, true> : fp4_decode_kernel<DT, false>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, (NH + kThreads32 - 1) / kThreads32,
                              0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint8_t *>(wire), n,
                          static_cast<uint16_t *>(y), NH);
}

cudaError_t launch_fp4_decode(int dtype, const void *wire, long long n, void *y, cudaStream_t s) {
    return dtype ? run_fp4_decode<1>(wire, n, y, s) : run_fp4_decode<0>(wire, n, y, s);
}

// Phase-1B on the staged kernel with min(ctas or #SMs, #SMs, tiles) CTAs;
// with ctas = 0, from 48 tiles per SM at the rank counts that
// fp4_reduce_ahead_min_blocks names, the one-block-ahead kernel instead (two
// waves of resident CTAs).
template <int R>
static cudaError_t run_fp4_reduce_r(const ConstPtrs &w, long long n, void *out, int ctas, cudaStream_t s) {
    using Shape = StagedReduceShape<Fp4Reduce, R>;
    auto kern = staged_reduce_kernel<Fp4Reduce, R, Shape::kGroups, Shape::kStages>;
    const long long T = (n + kTileValues - 1) / kTileValues;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (sms <= 0) return err;
    constexpr int kAhead = fp4_reduce_ahead_min_blocks<R>();
    if constexpr (kAhead > 0) {
        if (ctas == 0 && T >= 48LL * sms) {
            const long long NB = 64 * T;
            auto ahead = reduce_ahead_kernel<Fp4BlockReducer, R, kAhead>;
            const int grid = grid_for(reinterpret_cast<const void *>(ahead), kThreads32, NB, 0, 2, &err);
            if (grid <= 0) return err;
            return launch_chained(ahead, grid, kThreads32, 0, s, w, static_cast<uint8_t *>(out), NB);
        }
    }
    if ((err = allow_dynamic_smem(reinterpret_cast<const void *>(kern), Shape::kSmemBytes)) != cudaSuccess)
        return err;
    unsigned *timeouts = wait_timeout_counter(&err);
    if (!timeouts) return err;
    long long grid = ctas > 0 ? ctas : sms;
    if (grid > sms) grid = sms;
    if (grid > T) grid = T;
    return launch_chained(kern, static_cast<int>(grid), Fp4Reduce::kThreads * Shape::kGroups, Shape::kSmemBytes,
                          s, w, static_cast<uint8_t *>(out), T, n, timeouts);
}

cudaError_t launch_fp4_reduce(int R, const void *const *wires, long long n, void *out, int ctas, cudaStream_t s) {
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    switch (R) {
        case 1: return run_fp4_reduce_r<1>(w, n, out, ctas, s);
        case 2: return run_fp4_reduce_r<2>(w, n, out, ctas, s);
        case 3: return run_fp4_reduce_r<3>(w, n, out, ctas, s);
        case 4: return run_fp4_reduce_r<4>(w, n, out, ctas, s);
        case 5: return run_fp4_reduce_r<5>(w, n, out, ctas, s);
        case 6: return run_fp4_reduce_r<6>(w, n, out, ctas, s);
        case 7: return run_fp4_reduce_r<7>(w, n, out, ctas, s);
        case 8: return run_fp4_reduce_r<8>(w, n, out, ctas, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fp4_allreduce(int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                 cudaStream_t s) {
    ConstPtrs xp{};
    for (int r = 0; r < R; ++r) xp.p[r] = x[r];
    return dtype ? launch_staged<Fp4Tile<1>>(R, xp, n, y, ctas, s) : launch_staged<Fp4Tile<0>>(R, xp, n, y, ctas, s);
}

}  // namespace qrk
