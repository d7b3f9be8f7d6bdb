// qr_codec_peer.cu -- the per-rank two-shot all-reduce (R ranks, every rank
// storing straight into the others' workspaces, as qr_twoshot_peer.cu does
// for the symmetric codec) with the two other codecs:
//   the asymmetric group-128 codec ([FC] key machinery: quantize at the
//   reduce-scatter width, all-to-all, the owner's local sum re-quantized at
//   the all-gather width, all-gather, dequantize; the mixed "INT6" pair
//   reduce-scatters at INT4 and gathers at INT8), and
//   the FP4 codec ([QR] introduction: the FP4 mode interchangeable with INT4;
//   E2M1 elements in the INT4 tile).
// The workspace layout and the host checks are those of qr_peer.cuh; the
// phases and their joins are those of the symmetric per-rank calls: send,
// join, reduce, join, decode, no kernel waiting on another rank, plain loads
// and stores into peer memory (no bulk copy, no multicast).
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_kernels_fc.cuh"
#include "qr_kernels_fp4.cuh"
#include "qr_launch.h"
#include "qr_peer.cuh"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace qrk {

namespace {

// ---------------------------------------------------------------------------
// asymmetric codec: one 2048-value tile per CTA of kThreadsFc threads
// ---------------------------------------------------------------------------

// Phase-1 of one rank: its message quantized at BRS bits, tile t stored into
// recv[rank] of the tile's owner.
template <int BRS, int DT, bool A32>
__global__ void __launch_bounds__(kThreadsFc) fc_peer_send_kernel(const uint16_t *__restrict__ x, long long n,
                                                                  PeerOwnerTiles dst, long long T) {
    chain_entry();
    for (long long t = blockIdx.x; t < T; t += gridDim.x) fc_encode_tile16<BRS, DT, A32>(x, n, t, threadIdx.x, dst(t));
}

// Phase-1B of owner `rank` (its segment: tiles tile0 .. tile0 + tiles - 1):
// the R received copies summed in sender order and re-quantized at BAG bits;
// each tile stored into the gathered wire of every workspace (the
// all-gather, as peer stores).
template <int BRS, int BAG, int R>
__global__ void __launch_bounds__(kThreadsFc) fc_peer_reduce_kernel(const uint8_t *__restrict__ own, MutPtrs ws,
                                                                    long long n, long long seg, long long tile0,
                                                                    long long tiles) {
    chain_entry();
    constexpr long long tbi = FcCodec<BRS>::kTileBytes, tbo = FcCodec<BAG>::kTileBytes;
    const long long gathered = static_cast<long long>(R) * seg * tbi;
    const int i = threadIdx.x;
    for (long long lt = blockIdx.x; lt < tiles; lt += gridDim.x) {
        HalfWords<BRS> c[R];
        float s[R], z[R];
#pragma unroll
        for (int r = 0; r < R; ++r) fc_load16<BRS>(own + (r * seg + lt) * tbi, i, c[r], s[r], z[r]);
        const long long t = tile0 + lt;
        float2 f[8];
        FcParams p;
        fc_reduce_values<BRS, BAG, R>(c, s, z, t * kTileValues + 16 * i, n, f, p);
        HalfWords<BAG> cw;
        pack_half<BAG>(f, cw);
#pragma unroll
        for (int j = 0; j < R; ++j) fc_store_packed16<BAG>(static_cast<uint8_t *>(ws.p[j]) + gathered + t * tbo, i, cw, p);
    }
}

template <int BRS, int DT>
cudaError_t run_fc_peer_send(int R, int rank, const void *x, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    auto kern = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 ? fc_peer_send_kernel<BRS, DT, true>
                                                             : fc_peer_send_kernel<BRS, DT, false>;
    cudaError_t err = cudaSuccess;
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreadsFc, T, &err);
    if (grid <= 0) return err;
    PeerOwnerTiles dst{ws, twoshot_segment_tiles(T, R), rank, FcCodec<BRS>::kTileBytes};
    return launch_chained(kern, grid, kThreadsFc, 0, s, static_cast<const uint16_t *>(x), n, dst, T);
}

template <int BRS, int BAG, int R>
cudaError_t run_fc_peer_reduce_r(int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    const long long t0 = static_cast<long long>(rank) * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return cudaSuccess;  // more ranks than tiles: this owner has nothing
    auto kern = fc_peer_reduce_kernel<BRS, BAG, R>;
    cudaError_t err = cudaSuccess;
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreadsFc, tiles, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreadsFc, 0, s, static_cast<const uint8_t *>(ws.p[rank]), ws, n, seg, t0,
                          tiles);
}

template <int BRS, int BAG>
cudaError_t run_fc_peer_reduce(int R, int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    switch (R) {
        case 1: return run_fc_peer_reduce_r<BRS, BAG, 1>(rank, n, ws, s);
        case 2: return run_fc_peer_reduce_r<BRS, BAG, 2>(rank, n, ws, s);
        case 3: return run_fc_peer_reduce_r<BRS, BAG, 3>(rank, n, ws, s);
        case 4: return run_fc_peer_reduce_r<BRS, BAG, 4>(rank, n, ws, s);
        case 5: return run_fc_peer_reduce_r<BRS, BAG, 5>(rank, n, ws, s);
        case 6: return run_fc_peer_reduce_r<BRS, BAG, 6>(rank, n, ws, s);
        case 7: return run_fc_peer_reduce_r<BRS, BAG, 7>(rank, n, ws, s);
        case 8: return run_fc_peer_reduce_r<BRS, BAG, 8>(rank, n, ws, s);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// FP4 codec: one 32-value block per thread
// ---------------------------------------------------------------------------

template <int DT>
__global__ void __launch_bounds__(kThreads32) fp4_peer_send_kernel(const uint16_t *__restrict__ x, long long n,
                                                                   PeerOwnerTiles dst, long long NB) {
    chain_entry();
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb < NB; gb += S)
        fp4_encode_block<DT>(x, n, gb, dst(gb >> 6));
}

template <int R>
__global__ void __launch_bounds__(kThreads32) fp4_peer_reduce_kernel(const uint8_t *__restrict__ own, MutPtrs ws,
                                                                     long long seg, long long tile0, long long NB) {
    chain_entry();
    constexpr long long tb = Codec<4>::kTileBytes;
    const long long gathered = static_cast<long long>(R) * seg * tb;
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long lb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; lb < NB; lb += S) {
        const long long lt = lb >> 6;
        const int g = static_cast<int>(lb & 63);
        BlockWords<4> c[R];
        uint32_t sb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t *tile = own + (r * seg + lt) * tb;
            load_block_codes<4>(tile, g, c[r]);
            sb[r] = load_block_scale_bits<4>(tile, g);
        }
        BlockWords<4> cw;
        uint32_t bits;
        fp4_reduce_block_words<R>(c, sb, cw, bits);
        const long long off = gathered + (tile0 + lt) * tb;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            uint8_t *tile = static_cast<uint8_t *>(ws.p[j]) + off;
            store_block_codes<4>(tile, g, cw);
            store_block_scale<4>(tile, g, bits);
        }
    }
}

template <int DT>
cudaError_t run_fp4_peer_send(int R, int rank, const void *x, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long NB = 64 * T;
    auto kern = fp4_peer_send_kernel<DT>;
    cudaError_t err = cudaSuccess;
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreads32, (NB + kThreads32 - 1) / kThreads32,
                               &err);
    if (grid <= 0) return err;
    PeerOwnerTiles dst{ws, twoshot_segment_tiles(T, R), rank, Codec<4>::kTileBytes};
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint16_t *>(x), n, dst, NB);
}

template <int R>
cudaError_t run_fp4_peer_reduce_r(int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    const long long t0 = static_cast<long long>(rank) * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return cudaSuccess;  // more ranks than tiles: this owner has nothing
    const long long NB = 64 * tiles;
    auto kern = fp4_peer_reduce_kernel<R>;
    cudaError_t err = cudaSuccess;
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreads32, (NB + kThreads32 - 1) / kThreads32,
                               &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint8_t *>(ws.p[rank]), ws, seg, t0, NB);
}

cudaError_t run_fp4_peer_reduce(int R, int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    switch (R) {
        case 1: return run_fp4_peer_reduce_r<1>(rank, n, ws, s);
        case 2: return run_fp4_peer_reduce_r<2>(rank, n, ws, s);
        case 3: return run_fp4_peer_reduce_r<3>(rank, n, ws, s);
        case 4: return run_fp4_peer_reduce_r<4>(rank, n, ws, s);
        case 5: return run_fp4_peer_reduce_r<5>(rank, n, ws, s);
        case 6: return run_fp4_peer_reduce_r<6>(rank, n, ws, s);
        case 7: return run_fp4_peer_reduce_r<7>(rank, n, ws, s);
        case 8: return run_fp4_peer_reduce_r<8>(rank, n, ws, s);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

bool fc_pair(int bits_rs, int bits_ag) {
    return bits_rs == 4 ? (bits_ag == 4 || bits_ag == 8) : (bits_rs == 8 && bits_ag == 8);
}

bool dtype16(qr_dtype_t d) { return d == QR_FP16 || d == QR_BF16; }

// 2 * R * seg tiles of `tb` bytes each (R * seg of tb_in and R * seg of tb_out
// when the widths differ), 0 on overflow or bad arguments.
size_t peer_ws_bytes(size_t tb_in, size_t tb_out, int R, size_t n) {
    if (R < 1 || R > QR_MAX_RANKS || n == 0) return 0;
    const size_t T = n / QR_TILE_VALUES + (n % QR_TILE_VALUES != 0);
    const size_t tiles = static_cast<size_t>(R) * ((T + R - 1) / R);
    if (tiles > SIZE_MAX / (tb_in + tb_out)) return 0;
    return tiles * (tb_in + tb_out);
}

MutPtrs peer_ptrs(int R, void *const *workspaces) {
    MutPtrs ws{};
    for (int r = 0; r < R; ++r) ws.p[r] = workspaces[r];
    return ws;
}

// The input's own checks (after the shared ones): the dtype, its alignment,
// no overlap with any workspace.
qr_status_t check_send_input(qr_dtype_t dtype, int R, const void *x, size_t n, void *const *ws, size_t need) {
    if (!dtype16(dtype)) return QR_ERR_UNSUPPORTED;
    if (!peer_aligned16(x)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (peer_overlaps(x, 2 * n, ws[r], need)) return QR_ERR_INVALID_ARG;
    return QR_OK;
}

}  // namespace

}  // namespace qrk

QR_EXPORT size_t qr_fc_twoshot_peer_workspace_bytes(int bits_rs, int bits_ag, int R, size_t n) {
    if (!qrk::fc_pair(bits_rs, bits_ag)) return 0;
    return qrk::peer_ws_bytes(qr_fc_tile_bytes(bits_rs), qr_fc_tile_bytes(bits_ag), R, n);
}

QR_EXPORT qr_status_t qr_fc_twoshot_peer_send(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, int rank,
                                              const void *x, size_t n, void *const *workspaces,
                                              qr_stream_t stream) {
    if (!x || !workspaces || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (!qrk::fc_pair(bits_rs, bits_ag) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fc_twoshot_peer_workspace_bytes(bits_rs, bits_ag, R, n);
    qr_status_t st = qrk::check_peer_set(R, rank, n, workspaces, need);
    if (st == QR_OK) st = qrk::check_send_input(dtype, R, x, n, workspaces, need);
    if (st != QR_OK) return st;
    const qrk::MutPtrs ws = qrk::peer_ptrs(R, workspaces);
    const long long nn = static_cast<long long>(n);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf = dtype == QR_BF16;
    cudaError_t e;
    if (bits_rs == 4)
        e = bf ? qrk::run_fc_peer_send<4, 1>(R, rank, x, nn, ws, s) : qrk::run_fc_peer_send<4, 0>(R, rank, x, nn, ws, s);
    else
        e = bf ? qrk::run_fc_peer_send<8, 1>(R, rank, x, nn, ws, s) : qrk::run_fc_peer_send<8, 0>(R, rank, x, nn, ws, s);
    return qrk::peer_from_cuda(e);
}

QR_EXPORT qr_status_t qr_fc_twoshot_peer_reduce(int bits_rs, int bits_ag, int R, int rank, size_t n,
                                                void *const *workspaces, qr_stream_t stream) {
    if (!workspaces || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (!qrk::fc_pair(bits_rs, bits_ag) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fc_twoshot_peer_workspace_bytes(bits_rs, bits_ag, R, n);
    const qr_status_t st = qrk::check_peer_set(R, rank, n, workspaces, need);
    if (st != QR_OK) return st;
    const qrk::MutPtrs ws = qrk::peer_ptrs(R, workspaces);
    const long long nn = static_cast<long long>(n);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (bits_rs == 8)
        e = qrk::run_fc_peer_reduce<8, 8>(R, rank, nn, ws, s);
    else if (bits_ag == 8)
        e = qrk::run_fc_peer_reduce<4, 8>(R, rank, nn, ws, s);
    else
        e = qrk::run_fc_peer_reduce<4, 4>(R, rank, nn, ws, s);
    return qrk::peer_from_cuda(e);
}

QR_EXPORT qr_status_t qr_fc_twoshot_peer_decode(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, size_t n,
                                                const void *workspace, void *y, qr_stream_t stream) {
    if (!workspace || !y || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (!qrk::fc_pair(bits_rs, bits_ag) || R > QR_MAX_RANKS || !qrk::dtype16(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fc_twoshot_peer_workspace_bytes(bits_rs, bits_ag, R, n);
    const qr_status_t st = qrk::check_peer_decode(n, workspace, y, need);
    if (st != QR_OK) return st;
    const size_t T = n / QR_TILE_VALUES + (n % QR_TILE_VALUES != 0);
    const size_t seg = (T + R - 1) / R;
    const uint8_t *gathered =
        static_cast<const uint8_t *>(workspace) + static_cast<size_t>(R) * seg * qr_fc_tile_bytes(bits_rs);
    return qrk::peer_from_cuda(qrk::launch_fc_decode(bits_ag, static_cast<int>(dtype), gathered,
                                                     static_cast<long long>(n), y,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT size_t qr_fp4_twoshot_peer_workspace_bytes(int R, size_t n) {
    return qrk::peer_ws_bytes(qr_tile_bytes(4), qr_tile_bytes(4), R, n);
}

QR_EXPORT qr_status_t qr_fp4_twoshot_peer_send(qr_dtype_t dtype, int R, int rank, const void *x, size_t n,
                                               void *const *workspaces, qr_stream_t stream) {
    if (!x || !workspaces || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fp4_twoshot_peer_workspace_bytes(R, n);
    qr_status_t st = qrk::check_peer_set(R, rank, n, workspaces, need);
    if (st == QR_OK) st = qrk::check_send_input(dtype, R, x, n, workspaces, need);
    if (st != QR_OK) return st;
    const qrk::MutPtrs ws = qrk::peer_ptrs(R, workspaces);
    const long long nn = static_cast<long long>(n);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return qrk::peer_from_cuda(dtype == QR_BF16 ? qrk::run_fp4_peer_send<1>(R, rank, x, nn, ws, s)
                                                : qrk::run_fp4_peer_send<0>(R, rank, x, nn, ws, s));
}

QR_EXPORT qr_status_t qr_fp4_twoshot_peer_reduce(int R, int rank, size_t n, void *const *workspaces,
                                                 qr_stream_t stream) {
    if (!workspaces || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fp4_twoshot_peer_workspace_bytes(R, n);
    const qr_status_t st = qrk::check_peer_set(R, rank, n, workspaces, need);
    if (st != QR_OK) return st;
    return qrk::peer_from_cuda(qrk::run_fp4_peer_reduce(R, rank, static_cast<long long>(n),
                                                        qrk::peer_ptrs(R, workspaces),
                                                        reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_fp4_twoshot_peer_decode(qr_dtype_t dtype, int R, size_t n, const void *workspace, void *y,
                                                 qr_stream_t stream) {
    if (!workspace || !y || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (R > QR_MAX_RANKS || !qrk::dtype16(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_fp4_twoshot_peer_workspace_bytes(R, n);
    const qr_status_t st = qrk::check_peer_decode(n, workspace, y, need);
    if (st != QR_OK) return st;
    const size_t T = n / QR_TILE_VALUES + (n % QR_TILE_VALUES != 0);
    const size_t seg = (T + R - 1) / R;
    const uint8_t *gathered = static_cast<const uint8_t *>(workspace) + static_cast<size_t>(R) * seg * qr_tile_bytes(4);
    return qrk::peer_from_cuda(qrk::launch_fp4_decode(static_cast<int>(dtype), gathered, static_cast<long long>(n), y,
                                                      reinterpret_cast<cudaStream_t>(stream)));
}
