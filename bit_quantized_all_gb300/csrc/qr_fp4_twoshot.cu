// qr_fp4_twoshot.cu -- the two-shot all-reduce of the FP4 codec (E2M1
// elements in the INT4 tile) with its exchange laid out per rank and per
// owner, as qr_twoshot.cu does for the integer codes ([QR] Design
// Highlights: Phase-1 sends each rank's quantized segment k to its owner,
// Phase-1B the owner reduces its segment, Phase-2 every rank gathers and
// decodes; [QR] introduction: the FP4 mode interchangeable with INT4).
//
// Workspace layout (seg = ceil(T/R) tiles per owner, 1152-byte tiles):
//   recv[k][j] at ((k*R + j) * seg) tiles: owner k's copy of sender j's segment;
//   gathered   at (R*R*seg) tiles: the reduced wire, T tiles in tile order
//              (byte-identical to qr_fp4_segment_reduce's output).
#include <cstdint>

#include "qr_kernels_fp4.cuh"
#include "qr_launch.h"

namespace qrk {

// Phase-1: sender j = blockIdx.y quantizes its whole message into the owners'
// receive buffers, one 32-value block per thread.
template <int DT>
__global__ void __launch_bounds__(kThreads32) fp4_twoshot_send_kernel(ConstPtrs x, long long n, uint8_t *ws,
                                                                      long long seg, long long NB) {
    chain_entry();
    const long long j = blockIdx.y, R = gridDim.y;
    const uint16_t *xj = static_cast<const uint16_t *>(row_pointer(x.p, static_cast<int>(j)));
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb < NB; gb += S) {
        const long long t = gb >> 6, k = t / seg;
        fp4_encode_block<DT>(xj, n, gb, ws + ((k * R + j) * seg + (t - k * seg)) * Codec<4>::kTileBytes);
    }
}

// Phase-1B: owner k = blockIdx.y sums the R received copies of its segment in
// sender order and re-quantizes them into its part of the gathered wire.
template <int R>
__global__ void __launch_bounds__(kThreads32) fp4_twoshot_reduce_kernel(uint8_t *ws, long long T, long long seg) {
    chain_entry();
    const long long k = blockIdx.y;
    const long long t0 = k * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return;  // more owners than tiles: nothing to reduce
    constexpr long long tb = Codec<4>::kTileBytes;
    uint8_t *gathered = ws + static_cast<long long>(R) * R * seg * tb;
    const long long NB = 64 * tiles, S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long lb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; lb < NB; lb += S) {
        const long long lt = lb >> 6;
        const int g = static_cast<int>(lb & 63);
        BlockWords<4> c[R];
        uint32_t sb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t *tile = ws + ((k * R + r) * seg + lt) * tb;
            load_block_codes<4>(tile, g, c[r]);
            sb[r] = load_block_scale_bits<4>(tile, g);
        }
        fp4_reduce_block<R>(c, sb, gathered + (t0 + lt) * tb, g);
    }
}

// Phase-2: rank j = blockIdx.y decodes the gathered wire into its output.
template <int DT, bool Y32>
__global__ void __launch_bounds__(kThreads32) fp4_twoshot_decode_kernel(const uint8_t *__restrict__ gathered,
                                                                        long long n, MutPtrs y, long long NH) {
    chain_entry();
    fp4_decode_run<DT, Y32>(gathered, n, static_cast<uint16_t *>(row_pointer(y.p, static_cast<int>(blockIdx.y))),
                            NH);
}

namespace {

// CTAs per row: four waves of resident CTAs over all rows together, split
// evenly between the rows, at most one per `units_per_row` thread-units.
int fp4_row_ctas(const void *kern, long long units_per_row, int rows, cudaError_t *err) {
    const int g = grid_for(kern, kThreads32, units_per_row * rows, 0, 4, err);
    if (g <= 0) return 0;
    long long per_row = (g + rows - 1) / rows;
    if (per_row > units_per_row) per_row = units_per_row;
    return static_cast<int>(per_row < 1 ? 1 : per_row);
}

template <int R>
cudaError_t fp4_reduce_all_r(uint8_t *ws, long long T, long long seg, cudaStream_t s) {
    auto kern = fp4_twoshot_reduce_kernel<R>;
    cudaError_t err = cudaSuccess;
    const int gx = fp4_row_ctas(reinterpret_cast<const void *>(kern), (64 * seg + kThreads32 - 1) / kThreads32, R,
                                &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreads32, 0, s, ws, T, seg);
}

cudaError_t fp4_reduce_all(int R, uint8_t *ws, long long T, long long seg, cudaStream_t s) {
    switch (R) {
        case 1: return fp4_reduce_all_r<1>(ws, T, seg, s);
        case 2: return fp4_reduce_all_r<2>(ws, T, seg, s);
        case 3: return fp4_reduce_all_r<3>(ws, T, seg, s);
        case 4: return fp4_reduce_all_r<4>(ws, T, seg, s);
        case 5: return fp4_reduce_all_r<5>(ws, T, seg, s);
        case 6: return fp4_reduce_all_r<6>(ws, T, seg, s);
        case 7: return fp4_reduce_all_r<7>(ws, T, seg, s);
        case 8: return fp4_reduce_all_r<8>(ws, T, seg, s);
    }
    return cudaErrorInvalidValue;
}

template <int DT>
cudaError_t run_fp4_twoshot(int R, const void *const *x, long long n, void *const *y, uint8_t *ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    ConstPtrs xp{};
    MutPtrs yp{};
    bool y32 = true;
    for (int j = 0; j < R; ++j) {
        xp.p[j] = x[j];
        yp.p[j] = y[j];
        y32 = y32 && (reinterpret_cast<uintptr_t>(y[j]) & 31u) == 0;
    }
    cudaError_t err = cudaSuccess;
    {
        const long long NB = 64 * T;
        auto kern = fp4_twoshot_send_kernel<DT>;
        const int gx = fp4_row_ctas(reinterpret_cast<const void *>(kern), (NB + kThreads32 - 1) / kThreads32, R, &err);
        if (gx <= 0) return err;
        if ((err = launch_chained(kern, dim3(gx, R), kThreads32, 0, s, xp, n, ws, seg, NB)) != cudaSuccess) return err;
    }
    if ((err = fp4_reduce_all(R, ws, T, seg, s)) != cudaSuccess) return err;
    const uint8_t *gathered = ws + static_cast<long long>(R) * R * seg * Codec<4>::kTileBytes;
    const long long NH = 128 * T;
    auto kern = y32 ? fp4_twoshot_decode_kernel<DT, true> : fp4_twoshot_decode_kernel<DT, false>;
    const int gx = fp4_row_ctas(reinterpret_cast<const void *>(kern), (NH + kThreads32 - 1) / kThreads32, R, &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreads32, 0, s, gathered, n, yp, NH);
}

}  // namespace

cudaError_t launch_fp4_twoshot(int dtype, int R, const void *const *x, long long n, void *const *y, void *ws,
                               cudaStream_t s) {
    uint8_t *w = static_cast<uint8_t *>(ws);
    return dtype ? run_fp4_twoshot<1>(R, x, n, y, w, s) : run_fp4_twoshot<0>(R, x, n, y, w, s);
}

}  // namespace qrk
