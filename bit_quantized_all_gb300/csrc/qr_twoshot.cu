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
// Every rank's send, every owner's reduction and every rank's decode is its
// own launch, on the caller's stream in that order, so the data each rank
// would move is moved: R*(2N + W) for the sends, R*W + W for the owners'
// reductions, R*(W + 2N) for the decodes (W = wire bytes).
#include <cstdint>

#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

long long twoshot_segment_tiles(long long tiles, int R) { return (tiles + R - 1) / R; }

template <int B, int DT>
static cudaError_t send_rank(const void *x, long long n, uint8_t *ws, long long seg, int R, int j,
                             cudaStream_t s) {
    constexpr int U = 2;
    const long long NB = 64 * ((n + kTileValues - 1) / kTileValues);
    auto kern = encode32_kernel<B, DT, U, OwnerTiles>;
    cudaError_t err = cudaSuccess;
    const long long units = (NB + kThreads32 * U - 1) / (kThreads32 * U);
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
    if (grid <= 0) return err;
    kern<<<grid, kThreads32, 0, s>>>(static_cast<const uint16_t *>(x), n,
                                     OwnerTiles{ws, seg, R, j, Codec<B>::kTileBytes}, NB);
    return cudaGetLastError();
}

static cudaError_t send(int bits, int dtype, const void *x, long long n, uint8_t *ws, long long seg, int R, int j,
                        cudaStream_t s) {
#define QR_CASE(B)                                                                                  \
    case B:                                                                                         \
        return dtype ? send_rank<B, 1>(x, n, ws, seg, R, j, s) : send_rank<B, 0>(x, n, ws, seg, R, j, s);
    switch (bits) {
        QR_CASE(3)
        QR_CASE(4)
        QR_CASE(6)
        QR_CASE(8)
    }
#undef QR_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_twoshot(int bits, int dtype, int R, const void *const *x, long long n, void *const *y, void *ws,
                           cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    const long long tb = 256LL * bits + 128;
    uint8_t *w = static_cast<uint8_t *>(ws);
    cudaError_t err;
    // Phase-1: every rank sends segment k of its quantized message to owner k
    for (int j = 0; j < R; ++j)
        if ((err = send(bits, dtype, x[j], n, w, seg, R, j, s)) != cudaSuccess) return err;
    // Phase-1B: owner k reduces the R copies of its segment into the gathered wire
    uint8_t *red = w + static_cast<long long>(R) * R * seg * tb;
    for (int k = 0; k < R; ++k) {
        const long long t0 = k * seg;
        if (t0 >= T) break;
        const long long end = (k + 1) * seg * kTileValues;
        const long long nk = (end < n ? end : n) - t0 * kTileValues;
        const void *copies[kMaxRanks];
        for (int j = 0; j < R; ++j) copies[j] = w + (static_cast<long long>(k) * R + j) * seg * tb;
        if ((err = launch_reduce(bits, R, copies, nk, red + t0 * tb, s)) != cudaSuccess) return err;
    }
    // Phase-2: every rank decodes the gathered wire into its own output
    for (int j = 0; j < R; ++j)
        if ((err = launch_decode(bits, dtype, red, n, y[j], s)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace qrk
