// qr_fc_twoshot.cu -- the two-shot all-reduce of the asymmetric group-128
// codec with its exchange laid out per rank and per owner ([FC] key
// machinery: each rank quantizes its activations at the reduce-scatter
// width, an all-to-all sends segment k to its owner, the owner sums the R
// copies locally and re-quantizes the partial sums at the all-gather width,
// an all-gather brings every segment to every rank, which dequantizes; the
// mixed "INT6" is INT4 reduce-scatter with INT8 all-gather).
//
// The message's T tiles are cut into R segments of seg = ceil(T/R) tiles;
// owner k holds tiles [k*seg, min(T, (k+1)*seg)).  Workspace layout:
//   recv[k][j] at ((k*R + j) * seg) reduce-scatter tiles: owner k's copy of
//              sender j's segment (R*R buffers of seg tiles);
//   gathered   at R*R*seg reduce-scatter tiles: the reduced wire at the
//              all-gather width, T tiles in tile order (byte-identical to
//              qr_fc_segment_reduce's output).
// Each phase is one launch on the caller's stream with one grid row
// (blockIdx.y) per rank or owner, doing what that rank would do on its own
// GPU: R*(2N + Wrs) bytes for the sends, R*Wrs + Wag for the owners'
// reductions, R*(Wag + 2N) for the decodes.
#include <cstdint>

#include "qr_kernels_fc.cuh"
#include "qr_launch.h"

namespace qrk {

// Phase-1: sender j = blockIdx.y quantizes its whole message at BRS bits
// straight into the owners' receive buffers.
template <int BRS, int DT, bool A32>
__global__ void __launch_bounds__(kThreadsFc) fc_twoshot_send_kernel(ConstPtrs x, long long n, uint8_t *ws,
                                                                     long long seg, long long T) {
    chain_entry();
    const int j = static_cast<int>(blockIdx.y);
    const long long R = gridDim.y;
    const uint16_t *xj = static_cast<const uint16_t *>(row_pointer(x.p, j));
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const long long k = t / seg;
        fc_encode_tile16<BRS, DT, A32>(xj, n, t, threadIdx.x,
                                       ws + ((k * R + j) * seg + (t - k * seg)) * FcCodec<BRS>::kTileBytes);
    }
}

// Phase-1B: owner k = blockIdx.y sums the R received copies of its segment
// in sender order and re-quantizes at BAG bits into the gathered wire.
template <int BRS, int BAG, int R>
__global__ void __launch_bounds__(kThreadsFc) fc_twoshot_reduce_kernel(uint8_t *ws, long long n, long long T,
                                                                       long long seg) {
    chain_entry();
    const long long k = blockIdx.y;
    const long long t0 = k * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return;  // more owners than tiles: nothing to reduce
    constexpr long long tbi = FcCodec<BRS>::kTileBytes, tbo = FcCodec<BAG>::kTileBytes;
    uint8_t *gathered = ws + static_cast<long long>(R) * R * seg * tbi;
    const int i = threadIdx.x;
    for (long long lt = blockIdx.x; lt < tiles; lt += gridDim.x) {
        HalfWords<BRS> c[R];
        float s[R], z[R];
#pragma unroll
        for (int r = 0; r < R; ++r) fc_load16<BRS>(ws + ((k * R + r) * seg + lt) * tbi, i, c[r], s[r], z[r]);
        const long long t = t0 + lt;
        fc_reduce_tile<BRS, BAG, R>(c, s, z, gathered + t * tbo, i, t * kTileValues + 16 * i, n);
    }
}

// Phase-2: rank j = blockIdx.y decodes the gathered wire into its output.
template <int BAG, int DT, bool A32>
__global__ void __launch_bounds__(kThreadsFc) fc_twoshot_decode_kernel(const uint8_t *__restrict__ gathered,
                                                                       long long n, MutPtrs y, long long T) {
    chain_entry();
    uint16_t *yj = static_cast<uint16_t *>(row_pointer(y.p, static_cast<int>(blockIdx.y)));
    const int i = threadIdx.x;
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        HalfWords<BAG> c;
        FcParams p;
        fc_load16<BAG>(gathered + t * FcCodec<BAG>::kTileBytes, i, c, p.s, p.z);
        float2 u[8], o[8];
        fc_unpack16<BAG>(c, u);
        const float2 s2 = make_float2(p.s, p.s), z2 = make_float2(p.z, p.z);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = __ffma2_rn(u[q], s2, z2);
        store16v<DT, A32>(yj, t * kTileValues + 16 * i, n, o);
    }
}

namespace {

// CTAs per row: four waves of resident CTAs over all rows together, split
// evenly between the rows, at most one per tile of a row.
int fc_row_ctas(const void *kern, long long tiles_per_row, int rows, cudaError_t *err) {
    const int g = grid_for(kern, kThreadsFc, tiles_per_row * rows, 0, 4, err);
    if (g <= 0) return 0;
    long long per_row = (g + rows - 1) / rows;
    if (per_row > tiles_per_row) per_row = tiles_per_row;
    return static_cast<int>(per_row < 1 ? 1 : per_row);
}

template <int BRS, int BAG, int R>
cudaError_t fc_reduce_all_r(uint8_t *ws, long long n, long long T, long long seg, cudaStream_t s) {
    auto kern = fc_twoshot_reduce_kernel<BRS, BAG, R>;
    cudaError_t err = cudaSuccess;
    const int gx = fc_row_ctas(reinterpret_cast<const void *>(kern), seg, R, &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreadsFc, 0, s, ws, n, T, seg);
}

template <int BRS, int BAG>
cudaError_t fc_reduce_all(int R, uint8_t *ws, long long n, long long T, long long seg, cudaStream_t s) {
    switch (R) {
        case 1: return fc_reduce_all_r<BRS, BAG, 1>(ws, n, T, seg, s);
        case 2: return fc_reduce_all_r<BRS, BAG, 2>(ws, n, T, seg, s);
        case 3: return fc_reduce_all_r<BRS, BAG, 3>(ws, n, T, seg, s);
        case 4: return fc_reduce_all_r<BRS, BAG, 4>(ws, n, T, seg, s);
        case 5: return fc_reduce_all_r<BRS, BAG, 5>(ws, n, T, seg, s);
        case 6: return fc_reduce_all_r<BRS, BAG, 6>(ws, n, T, seg, s);
        case 7: return fc_reduce_all_r<BRS, BAG, 7>(ws, n, T, seg, s);
        case 8: return fc_reduce_all_r<BRS, BAG, 8>(ws, n, T, seg, s);
    }
    return cudaErrorInvalidValue;
}

template <int BRS, int BAG, int DT>
cudaError_t run_fc_twoshot(int R, const void *const *x, long long n, void *const *y, uint8_t *ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    ConstPtrs xp{};
    MutPtrs yp{};
    bool x32 = true, y32 = true;
    for (int j = 0; j < R; ++j) {
        xp.p[j] = x[j];
        yp.p[j] = y[j];
        x32 = x32 && (reinterpret_cast<uintptr_t>(x[j]) & 31u) == 0;
        y32 = y32 && (reinterpret_cast<uintptr_t>(y[j]) & 31u) == 0;
    }
    cudaError_t err = cudaSuccess;
    {
        auto kern = x32 ? fc_twoshot_send_kernel<BRS, DT, true> : fc_twoshot_send_kernel<BRS, DT, false>;
        const int gx = fc_row_ctas(reinterpret_cast<const void *>(kern), T, R, &err);
        if (gx <= 0) return err;
        if ((err = launch_chained(kern, dim3(gx, R), kThreadsFc, 0, s, xp, n, ws, seg, T)) != cudaSuccess) return err;
    }
    if ((err = fc_reduce_all<BRS, BAG>(R, ws, n, T, seg, s)) != cudaSuccess) return err;
    const uint8_t *gathered = ws + static_cast<long long>(R) * R * seg * FcCodec<BRS>::kTileBytes;
    auto kern = y32 ? fc_twoshot_decode_kernel<BAG, DT, true> : fc_twoshot_decode_kernel<BAG, DT, false>;
    const int gx = fc_row_ctas(reinterpret_cast<const void *>(kern), T, R, &err);
    if (gx <= 0) return err;
    return launch_chained(kern, dim3(gx, R), kThreadsFc, 0, s, gathered, n, yp, T);
}

template <int BRS, int BAG>
cudaError_t run_fc_twoshot_dt(int dtype, int R, const void *const *x, long long n, void *const *y, uint8_t *ws,
                              cudaStream_t s) {
    return dtype ? run_fc_twoshot<BRS, BAG, 1>(R, x, n, y, ws, s) : run_fc_twoshot<BRS, BAG, 0>(R, x, n, y, ws, s);
}

}  // namespace

cudaError_t launch_fc_twoshot(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                              void *const *y, void *ws, cudaStream_t s) {
    uint8_t *w = static_cast<uint8_t *>(ws);
    if (bits_rs == 4 && bits_ag == 4) return run_fc_twoshot_dt<4, 4>(dtype, R, x, n, y, w, s);
    if (bits_rs == 4 && bits_ag == 8) return run_fc_twoshot_dt<4, 8>(dtype, R, x, n, y, w, s);
    if (bits_rs == 8 && bits_ag == 8) return run_fc_twoshot_dt<8, 8>(dtype, R, x, n, y, w, s);
    return cudaErrorInvalidValue;
}

}  // namespace qrk
