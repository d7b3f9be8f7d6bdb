// qr_fc.cu -- launchers of the Flash Communication codec's encode, Phase-1B
// reduce (register-fed, and the staged kernel with FcReduce) and decode
// kernels, and the width-pair dispatch of its fused all-reduce.
#include <cstdint>

#include "qr_kernels_fc.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B, int DT, bool A32>
static cudaError_t run_fc_encode_t(const void *x, long long n, void *wire, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    auto kern = fc_encode_kernel<B, DT, A32>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreadsFc, T, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreadsFc, 0, s, static_cast<const uint16_t *>(x), n,
                          static_cast<uint8_t *>(wire), T);
}

template <int B, int DT, bool A32>
static cudaError_t run_fc_decode_t(const void *wire, long long n, void *y, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    auto kern = fc_decode_kernel<B, DT, A32>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreadsFc, T, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreadsFc, 0, s, static_cast<const uint8_t *>(wire), n,
                          static_cast<uint16_t *>(y), T);
}

// Phase-1B on the staged kernel (the R wire tiles brought into shared memory
// by bulk copies) with min(ctas or #SMs, #SMs, tiles) persistent CTAs.
template <int BIN, int BOUT, int R>
static cudaError_t run_fc_reduce_staged_t(const ConstPtrs &w, long long n, void *out, int ctas, cudaStream_t s) {
    using P = FcReduce<BIN, BOUT>;
    using Shape = StagedReduceShape<P, R>;
    auto kern = staged_reduce_kernel<P, R, Shape::kGroups, Shape::kStages>;
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
    return launch_chained(kern, static_cast<int>(grid), P::kThreads * Shape::kGroups, Shape::kSmemBytes,
                          s, w, static_cast<uint8_t *>(out), T, n, timeouts);
}

// Where the default takes the staged Phase-1B kernel (tiles per SM from which
// it does; 0 = never), else a register-fed kernel.  Measured on GB300 at 2^27
// bf16 values per rank, fraction of the measured HBM bandwidth, register-fed
// with one tile in flight / with two / staged (five groups):
//   4 -> 4: R=2 0.51 / 0.52 / 0.39, R=4 0.46 / 0.56 / 0.47, R=6 0.39 / 0.57 /
//     0.51, R=8 0.39 / 0.58 / 0.53;
//   4 -> 8: R=2 0.59 / 0.64 / 0.50, R=4 0.51 / 0.64 / 0.54, R=8 0.47 / 0.62 /
//     0.58;
//   8 -> 8: R=2 0.82 / 0.85 / 0.73, R=3 0.74 / 0.86 / 0.83, R=4 0.75 / 0.87 /
//     0.88, R=6 0.61 / 0.90 / 0.95, R=8 0.74 / 0.93 / 1.01;
// so the staged kernel only for 8-bit inputs from R = 4 (memory-bound there),
// from 48 tiles per SM (below that the register-fed grid has more warps).
template <int BIN, int BOUT, int R>
__host__ __device__ constexpr long long staged_fc_reduce_min_tiles_per_sm() {
    return (BIN == 8 && R >= 4) ? 48 : 0;
}

constexpr int kFcReduceUnroll = 2;  // tiles per thread in flight in the register-fed kernel

// Where the register-fed Phase-1B loads one tile ahead (fc_reduce_ahead_kernel)
// instead of two tiles at once, and with how many CTAs per SM (0 = not).  At
// 2^27 values per rank, two at once / one ahead: 4-bit inputs R=2 0.49 / 0.51
// (4 -> 4) and 0.63 / 0.63 (4 -> 8), R=3 0.52 / 0.54 and 0.62 / 0.63, R=4
// 0.56 / 0.58, R=6 0.57 / 0.59, R=8 0.58 / 0.62 (4 -> 4) and 0.62 / 0.67
// (4 -> 8), with five CTAs per SM and four waves; 8 -> 8 at R=3 0.86 / 0.93
// (0.89 / 0.96 at 2^28) with eight CTAs per SM and two waves (at R = 2
// within 1% at 2^28).
template <int BIN, int BOUT, int R>
__host__ __device__ constexpr int fc_reduce_ahead_min_blocks() {
    return (BIN == 4 && R >= 2) ? 5 : (BIN == 8 && R == 3) ? 8 : 0;
}

template <int BIN, int BOUT, int R>
static cudaError_t run_fc_reduce_t(const ConstPtrs &w, long long n, void *out, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    constexpr long long kMinTilesPerSm = staged_fc_reduce_min_tiles_per_sm<BIN, BOUT, R>();
    if constexpr (kMinTilesPerSm > 0) {
        cudaError_t e = cudaSuccess;
        const int sms = sm_count(&e);
        if (sms <= 0) return e;
        if (T >= kMinTilesPerSm * sms) return run_fc_reduce_staged_t<BIN, BOUT, R>(w, n, out, 0, s);
    }
    cudaError_t err = cudaSuccess;
    constexpr int kAhead = fc_reduce_ahead_min_blocks<BIN, BOUT, R>();
    if constexpr (kAhead > 0) {
        auto kern = fc_reduce_ahead_kernel<BIN, BOUT, R, kAhead>;
        const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreadsFc, T, 0, BIN == 4 ? 4 : 2, &err);
        if (grid <= 0) return err;
        return launch_chained(kern, grid, kThreadsFc, 0, s, w, n, static_cast<uint8_t *>(out), T);
    }
    auto kern = fc_reduce_kernel<BIN, BOUT, R, kFcReduceUnroll>;
    const long long units = (T + kFcReduceUnroll - 1) / kFcReduceUnroll;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreadsFc, units, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreadsFc, 0, s, w, n, static_cast<uint8_t *>(out), T);
}

template <int B, int DT>
static cudaError_t fc_encode_dt(const void *x, long long n, void *wire, cudaStream_t s) {
    return (reinterpret_cast<uintptr_t>(x) & 31u) == 0 ? run_fc_encode_t<B, DT, true>(x, n, wire, s)
                                                        : run_fc_encode_t<B, DT, false>(x, n, wire, s);
}

template <int B, int DT>
static cudaError_t fc_decode_dt(const void *wire, long long n, void *y, cudaStream_t s) {
    return (reinterpret_cast<uintptr_t>(y) & 31u) == 0 ? run_fc_decode_t<B, DT, true>(wire, n, y, s)
                                                        : run_fc_decode_t<B, DT, false>(wire, n, y, s);
}

cudaError_t launch_fc_encode(int bits, int dtype, const void *x, long long n, void *wire, cudaStream_t s) {
    if (bits == 4) return dtype ? fc_encode_dt<4, 1>(x, n, wire, s) : fc_encode_dt<4, 0>(x, n, wire, s);
    if (bits == 8) return dtype ? fc_encode_dt<8, 1>(x, n, wire, s) : fc_encode_dt<8, 0>(x, n, wire, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fc_decode(int bits, int dtype, const void *wire, long long n, void *y, cudaStream_t s) {
    if (bits == 4) return dtype ? fc_decode_dt<4, 1>(wire, n, y, s) : fc_decode_dt<4, 0>(wire, n, y, s);
    if (bits == 8) return dtype ? fc_decode_dt<8, 1>(wire, n, y, s) : fc_decode_dt<8, 0>(wire, n, y, s);
    return cudaErrorInvalidValue;
}

template <int BIN, int BOUT>
static cudaError_t fc_reduce_r(int R, const ConstPtrs &w, long long n, void *out, cudaStream_t s) {
    switch (R) {
        case 1: return run_fc_reduce_t<BIN, BOUT, 1>(w, n, out, s);
        case 2: return run_fc_reduce_t<BIN, BOUT, 2>(w, n, out, s);
        case 3: return run_fc_reduce_t<BIN, BOUT, 3>(w, n, out, s);
        case 4: return run_fc_reduce_t<BIN, BOUT, 4>(w, n, out, s);
        case 5: return run_fc_reduce_t<BIN, BOUT, 5>(w, n, out, s);
        case 6: return run_fc_reduce_t<BIN, BOUT, 6>(w, n, out, s);
        case 7: return run_fc_reduce_t<BIN, BOUT, 7>(w, n, out, s);
        case 8: return run_fc_reduce_t<BIN, BOUT, 8>(w, n, out, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fc_reduce(int bits_in, int bits_out, int R, const void *const *wires, long long n, void *out,
                             cudaStream_t s) {
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    if (bits_in == 4 && bits_out == 4) return fc_reduce_r<4, 4>(R, w, n, out, s);
    if (bits_in == 4 && bits_out == 8) return fc_reduce_r<4, 8>(R, w, n, out, s);
    if (bits_in == 8 && bits_out == 8) return fc_reduce_r<8, 8>(R, w, n, out, s);
    return cudaErrorInvalidValue;
}

template <int BIN, int BOUT>
static cudaError_t fc_reduce_staged_r(int R, const ConstPtrs &w, long long n, void *out, int ctas, cudaStream_t s) {
    switch (R) {
        case 1: return run_fc_reduce_staged_t<BIN, BOUT, 1>(w, n, out, ctas, s);
        case 2: return run_fc_reduce_staged_t<BIN, BOUT, 2>(w, n, out, ctas, s);
        case 3: return run_fc_reduce_staged_t<BIN, BOUT, 3>(w, n, out, ctas, s);
        case 4: return run_fc_reduce_staged_t<BIN, BOUT, 4>(w, n, out, ctas, s);
        case 5: return run_fc_reduce_staged_t<BIN, BOUT, 5>(w, n, out, ctas, s);
        case 6: return run_fc_reduce_staged_t<BIN, BOUT, 6>(w, n, out, ctas, s);
        case 7: return run_fc_reduce_staged_t<BIN, BOUT, 7>(w, n, out, ctas, s);
        case 8: return run_fc_reduce_staged_t<BIN, BOUT, 8>(w, n, out, ctas, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fc_reduce_staged(int bits_in, int bits_out, int R, const void *const *wires, long long n, void *out,
                                    int ctas, cudaStream_t s) {
    ConstPtrs w{};
    for (int r = 0; r < R; ++r) w.p[r] = wires[r];
    if (bits_in == 4 && bits_out == 4) return fc_reduce_staged_r<4, 4>(R, w, n, out, ctas, s);
    if (bits_in == 4 && bits_out == 8) return fc_reduce_staged_r<4, 8>(R, w, n, out, ctas, s);
    if (bits_in == 8 && bits_out == 8) return fc_reduce_staged_r<8, 8>(R, w, n, out, ctas, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fc_allreduce(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                                void *y, int ctas, cudaStream_t s) {
    if (bits_rs == 4 && bits_ag == 4) return run_fc_allreduce<4, 4>(dtype, R, x, n, y, ctas, s);
    if (bits_rs == 4 && bits_ag == 8) return run_fc_allreduce<4, 8>(dtype, R, x, n, y, ctas, s);
    if (bits_rs == 8 && bits_ag == 8) return run_fc_allreduce<8, 8>(dtype, R, x, n, y, ctas, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fc_allreduce_staged(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                                       void *y, int ctas, cudaStream_t s) {
    if (bits_rs == 4 && bits_ag == 4) return run_fc_allreduce_staged<4, 4>(dtype, R, x, n, y, ctas, s);
    if (bits_rs == 4 && bits_ag == 8) return run_fc_allreduce_staged<4, 8>(dtype, R, x, n, y, ctas, s);
    if (bits_rs == 8 && bits_ag == 8) return run_fc_allreduce_staged<8, 8>(dtype, R, x, n, y, ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace qrk
