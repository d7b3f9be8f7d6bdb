// qr_reduce.cu -- launchers of the Phase-1B reduction kernels (reduce32_kernel,
// reduce_ahead_kernel and staged_reduce_kernel), R dispatched to a
// compile-time constant.
#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

// The staged kernel with min(ctas or #SMs, #SMs, tiles) persistent CTAs.
template <int B, int R>
static cudaError_t run_reduce_staged_r(const ConstPtrs &w, long long n, void *out, int ctas, cudaStream_t s) {
    using Shape = StagedReduceShape<QrReduce<B>, R>;
    auto kern = staged_reduce_kernel<QrReduce<B>, R, Shape::kGroups, Shape::kStages>;
    const long long T = (n + kTileValues - 1) / kTileValues;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (sms <= 0) return err;
    if ((err = allow_dynamic_smem(reinterpret_cast<const void *>(kern), Shape::kSmemBytes)) != cudaSuccess)
        return err;
    unsigned *timeouts = wait_timeout_counter(&err);
    if (!timeouts) return err;
    long long grid = ctas > 0 ? ctas : sms;
    if (grid > sms) grid = sms;
    if (grid > T) grid = T;
    return launch_chained(kern, static_cast<int>(grid), QrReduce<B>::kThreads * Shape::kGroups, Shape::kSmemBytes, s,
                          w, static_cast<uint8_t *>(out), T, n, timeouts);
}

// Where the default takes the staged kernel: INT4, INT6 and INT8 from 48
// tiles per SM (INT3 is bound by the integer pipe and stays register-fed),
// except where reduce_ahead_min_blocks names the one-block-ahead kernel.
constexpr long long kStagedReduceMinTilesPerSm = 48;

// The one-block-ahead kernel with two waves of resident CTAs.
template <int B, int R, int MINB>
static cudaError_t run_reduce_ahead_r(const ConstPtrs &w, long long T, void *out, cudaStream_t s) {
    const long long NB = 64 * T;
    auto kern = reduce_ahead_kernel<QrBlockReducer<B>, R, MINB>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, NB, 0, 2, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, w, static_cast<uint8_t *>(out), NB);
}

template <int B, int R>
static cudaError_t run_reduce_r(const ConstPtrs &w, long long n, void *out, cudaStream_t s) {
    constexpr int U = reduce_units_per_thread<R>();  // work units per thread in flight
    constexpr int kAhead = reduce_ahead_min_blocks<B, R>();
    const long long T = (n + kTileValues - 1) / kTileValues;
    cudaError_t err = cudaSuccess;
    if constexpr (B != 3 || kAhead > 0) {
        const int sms = sm_count(&err);
        if (sms <= 0) return err;
        if (T >= kStagedReduceMinTilesPerSm * sms) {
            if constexpr (kAhead > 0)
                return run_reduce_ahead_r<B, R, kAhead>(w, T, out, s);
            else
                return run_reduce_staged_r<B, R>(w, n, out, 0, s);
        }
    }
    const long long NB = 64 * T;
    auto kern = reduce32_kernel<B, R, U>;
    const long long units = (NB + kThreads32 * U - 1) / (kThreads32 * U);
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, w, static_cast<uint8_t *>(out), NB);
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

template <int B>
static cudaError_t run_reduce_staged(int R, const void *const *wires, long long n, void *out, int ctas,
                                     cudaStream_t s) {
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    switch (R) {
        case 1: return run_reduce_staged_r<B, 1>(w, n, out, ctas, s);
        case 2: return run_reduce_staged_r<B, 2>(w, n, out, ctas, s);
        case 3: return run_reduce_staged_r<B, 3>(w, n, out, ctas, s);
        case 4: return run_reduce_staged_r<B, 4>(w, n, out, ctas, s);
        case 5: return run_reduce_staged_r<B, 5>(w, n, out, ctas, s);
        case 6: return run_reduce_staged_r<B, 6>(w, n, out, ctas, s);
        case 7: return run_reduce_staged_r<B, 7>(w, n, out, ctas, s);
        case 8: return run_reduce_staged_r<B, 8>(w, n, out, ctas, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_staged(int bits, int R, const void *const *wires, long long n, void *out, int ctas,
                                 cudaStream_t s) {
    switch (bits) {
        case 3: return run_reduce_staged<3>(R, wires, n, out, ctas, s);
        case 4: return run_reduce_staged<4>(R, wires, n, out, ctas, s);
        case 6: return run_reduce_staged<6>(R, wires, n, out, ctas, s);
        case 8: return run_reduce_staged<8>(R, wires, n, out, ctas, s);
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
