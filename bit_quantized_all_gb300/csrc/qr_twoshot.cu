// qr_twoshot.cu -- the two-shot all-reduce with its exchange laid out as it
// would be across R GPUs ([QR] Design Highlights: Phase-1 sends each rank's
// quantized segment k to its owner, Phase-1B the owner reduces its segment,
// Phase-2 every rank gathers and decodes all segments; [FC] key machinery:
// one all-to-all, a local sum and re-quantization, one all-gather).
//
// The message's T tiles are cut into R segments of seg = ceil(T/R) tiles;
// owner k holds tiles [k*seg, min(T, (k+1)*seg)).  Workspace layout:
//   recv[k][j] at ((k*R + j) * seg) tiles: owner k's copy of sender j's
//              quantized segment (seg tiles each; R*R buffers);
//   red        at (R*R*seg) tiles: the gathered reduced wire, tile order.
// Each phase is one launch on the caller's stream whose grid has one row
// (blockIdx.y) per rank or owner, and each row does exactly what that rank
// would do on its own GPU, so the data each rank would move is moved:
// R*(2N + W) for the sends, R*W + W for the owners' reductions, R*(W + 2N)
// for the decodes (W = wire bytes).  The three launches run in order, which
// is the synchronisation a real exchange needs between its phases.
#include <cstdint>

#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

long long twoshot_segment_tiles(long long tiles, int R) { return (tiles + R - 1) / R; }

// Phase-1: sender j = blockIdx.y quantizes its whole message straight into
// the owners' receive buffers (segment k of the wire lands in recv[k][j]).
template <int B, int DT, int U>
__global__ void __launch_bounds__(kThreads32) twoshot_send_kernel(ConstPtrs x, long long n, uint8_t *ws,
                                                                  long long seg, long long NB) {
    chain_entry();
    const int j = static_cast<int>(blockIdx.y);
    encode32_run<B, DT, U>(static_cast<const uint16_t *>(row_pointer(x.p, j)), n,
                           OwnerTiles{ws, seg, static_cast<int>(gridDim.y), j, Codec<B>::kTileBytes}, NB);
}

// Phase-1B: owner k = blockIdx.y reduces the R received copies of its
// segment, in sender order, into its segment of the gathered wire.
template <int B, int R, int U>
__global__ void __launch_bounds__(kThreads32) twoshot_reduce_kernel(uint8_t *ws, long long T, long long seg) {
    chain_entry();
    const long long k = blockIdx.y;
    const long long t0 = k * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return;  // more owners than tiles: nothing to reduce
    constexpr long long tb = Codec<B>::kTileBytes;
    ConstPtrs w;
#pragma unroll
    for (int j = 0; j < R; ++j) w.p[j] = ws + (k * R + j) * seg * tb;
    uint8_t *red = ws + static_cast<long long>(R) * R * seg * tb + t0 * tb;
    reduce32_run<B, R, U>(w, red, 64 * tiles);
}

// Phase-2: rank j = blockIdx.y decodes the gathered wire into its output.
template <int B, int DT, int U, bool Y32>
__global__ void __launch_bounds__(kThreads32) twoshot_decode_kernel(const uint8_t *__restrict__ red, long long n,
                                                                    MutPtrs y, long long NH) {
    chain_entry();
    decode16_run<B, DT, U, Y32>(red, n, static_cast<uint16_t *>(row_pointer(y.p, static_cast<int>(blockIdx.y))), NH);
}

// CTAs per row: four waves of resident CTAs over all rows together, split
// evenly between the rows, at most one per work unit of a row.
static int row_ctas(const void *kern, long long units_per_row, int rows, cudaError_t *err) {
    const int g = grid_for(kern, kThreads32, units_per_row * rows, 0, 4, err);
    if (g <= 0) return 0;
    long long per_row = (g + rows - 1) / rows;
    if (per_row > units_per_row) per_row = units_per_row;
    return static_cast<int>(per_row < 1 ? 1 : per_row);
}

template <int B, int DT>
static cudaError_t send_all(int R, const void *const *x, long long n, uint8_t *ws, long long seg, cudaStream_t s) {
    constexpr int U = 2;
    const long long NB = 64 * ((n + kTileValues - 1) / kTileValues);
    ConstPtrs xp{};
    for (int j = 0; j < R; ++j) xp.p[j] = x[j];
    auto kern = twoshot_send_kernel<B, DT, U>;
    cudaError_t err = cudaSuccess;
    const int gx = row_ctas(reinterpret_cast<const void *>(kern), (NB + kThreads32 * U - 1) / (kThreads32 * U), R, &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreads32, 0, s, xp, n, ws, seg, NB);
}

template <int B, int R>
static cudaError_t reduce_all_r(uint8_t *ws, long long T, long long seg, cudaStream_t s) {
    constexpr int U = reduce_units_per_thread<R>();
    const long long per_row = 64 * seg;
    auto kern = twoshot_reduce_kernel<B, R, U>;
    cudaError_t err = cudaSuccess;
    const int gx = row_ctas(reinterpret_cast<const void *>(kern), (per_row + kThreads32 * U - 1) / (kThreads32 * U), R,
                            &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreads32, 0, s, ws, T, seg);
}

template <int B>
static cudaError_t reduce_all(int R, uint8_t *ws, long long T, long long seg, cudaStream_t s) {
    switch (R) {
        case 1: return reduce_all_r<B, 1>(ws, T, seg, s);
        case 2: return reduce_all_r<B, 2>(ws, T, seg, s);
        case 3: return reduce_all_r<B, 3>(ws, T, seg, s);
        case 4: return reduce_all_r<B, 4>(ws, T, seg, s);
        case 5: return reduce_all_r<B, 5>(ws, T, seg, s);
        case 6: return reduce_all_r<B, 6>(ws, T, seg, s);
        case 7: return reduce_all_r<B, 7>(ws, T, seg, s);
        case 8: return reduce_all_r<B, 8>(ws, T, seg, s);
    }
    return cudaErrorInvalidValue;
}

template <int B, int DT>
static cudaError_t decode_all(int R, const uint8_t *red, long long n, void *const *y, cudaStream_t s) {
    constexpr int U = 4;  // half-blocks per thread in flight, as in the standalone decode
    const long long NH = 128 * ((n + kTileValues - 1) / kTileValues);
    MutPtrs yp{};
    bool y32 = true;
    for (int j = 0; j < R; ++j) {
        yp.p[j] = y[j];
        y32 = y32 && (reinterpret_cast<uintptr_t>(y[j]) & 31u) == 0;
    }
    auto kern = y32 ? twoshot_decode_kernel<B, DT, U, true> : twoshot_decode_kernel<B, DT, U, false>;
    cudaError_t err = cudaSuccess;
    const int gx = row_ctas(reinterpret_cast<const void *>(kern), (NH + kThreads32 * U - 1) / (kThreads32 * U), R, &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreads32, 0, s, red, n, yp, NH);
}

template <int B, int DT>
static cudaError_t run_twoshot(int R, const void *const *x, long long n, void *const *y, uint8_t *ws,
                               cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    cudaError_t err;
    if ((err = send_all<B, DT>(R, x, n, ws, seg, s)) != cudaSuccess) return err;
    if ((err = reduce_all<B>(R, ws, T, seg, s)) != cudaSuccess) return err;
    const uint8_t *red = ws + static_cast<long long>(R) * R * seg * Codec<B>::kTileBytes;
    return decode_all<B, DT>(R, red, n, y, s);
}

cudaError_t launch_twoshot(int bits, int dtype, int R, const void *const *x, long long n, void *const *y, void *ws,
                           cudaStream_t s) {
    uint8_t *w = static_cast<uint8_t *>(ws);
#define QR_CASE(B)                                                                                  \
    case B:                                                                                         \
        return dtype ? run_twoshot<B, 1>(R, x, n, y, w, s) : run_twoshot<B, 0>(R, x, n, y, w, s);
    switch (bits) {
        QR_CASE(3)
        QR_CASE(4)
        QR_CASE(6)
        QR_CASE(8)
    }
#undef QR_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qrk
