// qr_peer.cuh -- what the per-rank two-shot calls of every codec share: where
// a sender's tile lands in its owner's workspace, and the host checks of a
// set of peer workspaces.
//
// Rank j's workspace, for a wire of T tiles cut into R segments of
// seg = ceil(T/R) tiles (segment k: tiles [k*seg, min(T, (k+1)*seg))):
//   recv[s]   at input tile s*seg (s = 0..R-1): sender s's quantized copy of
//             the segment this rank owns;
//   gathered  at input tile R*seg: the reduced wire in tile order (output
//             tile t at R*seg input tiles + t output tiles), written by the
//             owners.
// (Input and output tiles differ in size only for the asymmetric codec's
// mixed widths.)
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_device.cuh"

namespace qrk {

// Where the send path stores tile t of sender `sender`: recv[sender] of the
// owner k = t / seg, at the tile's place in the owner's segment.
struct PeerOwnerTiles {
    MutPtrs ws;  // rank k's workspace at ws.p[k]
    long long seg;
    int sender, tile_bytes;
    __device__ __forceinline__ uint8_t *operator()(long long t) const {
        const int k = static_cast<int>(static_cast<unsigned long long>(t) / static_cast<unsigned long long>(seg));
        uint8_t *base = static_cast<uint8_t *>(row_pointer(ws.p, k));
        return base + (static_cast<long long>(sender) * seg + (t - k * seg)) * tile_bytes;
    }
};

inline bool peer_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) share a byte
inline bool peer_overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline qr_status_t peer_from_cuda(cudaError_t e) { return e == cudaSuccess ? QR_OK : QR_ERR_CUDA; }

// The checks of a send or reduce call that follow the codec's own (the
// caller has returned QR_ERR_INVALID_ARG for a null `ws`, n == 0 or R < 1,
// and QR_ERR_UNSUPPORTED for a codec or R it does not take): a rank outside
// [0, R) or a null workspace -> QR_ERR_INVALID_ARG; n too large, or `need`
// (the workspace bytes of one rank) 0 -> QR_ERR_SIZE; a workspace not 16-byte
// aligned -> QR_ERR_MISALIGNED; two workspaces sharing a byte ->
// QR_ERR_INVALID_ARG.
inline qr_status_t check_peer_set(int R, int rank, size_t n, void *const *ws, size_t need) {
    if (rank < 0 || rank >= R) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r)
        if (!ws[r]) return QR_ERR_INVALID_ARG;
    if (n > SIZE_MAX / 4 || need == 0) return QR_ERR_SIZE;
    for (int r = 0; r < R; ++r)
        if (!peer_aligned16(ws[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < r; ++i)
            if (peer_overlaps(ws[r], need, ws[i], need)) return QR_ERR_INVALID_ARG;
    return QR_OK;
}

// The checks of a decode call after the codec's: n too large or `need` 0 ->
// QR_ERR_SIZE; workspace or y not 16-byte aligned -> QR_ERR_MISALIGNED; y
// sharing a byte with the workspace -> QR_ERR_INVALID_ARG.
inline qr_status_t check_peer_decode(size_t n, const void *workspace, const void *y, size_t need) {
    if (n > SIZE_MAX / 4 || need == 0) return QR_ERR_SIZE;
    if (!peer_aligned16(workspace) || !peer_aligned16(y)) return QR_ERR_MISALIGNED;
    if (peer_overlaps(y, 2 * n, workspace, need)) return QR_ERR_INVALID_ARG;
    return QR_OK;
}

// Grid-stride CTAs for a per-rank launch: four waves of resident CTAs,
// at most one per work unit.
int peer_grid(const void *kern, int threads, long long units, cudaError_t *err);

}  // namespace qrk
