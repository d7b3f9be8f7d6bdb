// qr_twoshot_peer.cu -- the two-shot all-reduce run by R separate ranks
// (one process, or one GPU, each), every rank storing straight into the
// other ranks' workspaces: [QR] Design Highlights (Phase-1 sends each rank's
// quantized segment k to its owner k, Phase-1B the owner reduces its
// segment, Phase-2 every rank gathers and decodes all segments); [FC] key
// machinery (all-to-all, local sum and re-quantization, all-gather over
// peer-to-peer GPU memory access).
//
// Rank j's workspace is laid out as qr_peer.cuh states (recv[s] at tile
// s*seg, the gathered wire at tile R*seg).
// A step is three calls per rank, in order, each one launch on the rank's
// stream: send (rank j quantizes its message and stores segment k of it into
// recv[j] of rank k's workspace), reduce (owner j sums the R copies of its
// segment and stores the re-quantized tiles into the gathered wire of every
// rank), decode (rank j decodes its own gathered wire).  Between the calls
// every rank's previous call must have finished on the GPU (the caller joins
// the ranks, e.g. with a host barrier after a stream synchronize); no kernel
// here waits on another rank.  The peers' workspaces are reached through
// pointers the caller maps into this process (CUDA IPC handles, or peer
// access between GPUs of one process).  Plain loads and stores only: no bulk
// copy and no multicast touches another rank's memory.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_kernels32.cuh"
#include "qr_launch.h"
#include "qr_peer.cuh"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace qrk {

namespace {

// Three CTAs per SM, as the contiguous encode has (INT6 took 86 registers a
// thread without the bound, and two CTAs per SM).
template <int B, int DT, int U>
__global__ void __launch_bounds__(kThreads32, 3) peer_send_kernel(const uint16_t *__restrict__ x, long long n,
                                                                  PeerOwnerTiles dst, long long NB) {
    chain_entry();
    encode32_run<B, DT, U>(x, n, dst, NB);
}

// Phase-1B of owner `rank`: the R copies of its `tiles` tiles come from its
// own recv buffers; every re-quantized block is stored into the gathered
// wire of each of the R workspaces (the all-gather, as peer stores).
template <int B, int R, int U>
__global__ void __launch_bounds__(kThreads32) peer_reduce_kernel(const uint8_t *__restrict__ own, MutPtrs ws,
                                                                 long long seg, long long tile0, long long NB) {
    chain_entry();
    constexpr long long tb = Codec<B>::kTileBytes;
    const long long gathered = static_cast<long long>(R) * seg * tb;
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb0 = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb0 < NB; gb0 += U * S) {
        BlockWords<B> c[U][R];
        uint32_t sb[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB) {
                const long long lt = gb >> 6;
#pragma unroll
                for (int s = 0; s < R; ++s) {
                    const uint8_t *tile = own + (s * seg + lt) * tb;
                    load_block_codes<B>(tile, static_cast<int>(gb & 63), c[u][s]);
                    sb[u][s] = load_block_scale_bits<B>(tile, static_cast<int>(gb & 63));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB) {
                BlockWords<B> cw;
                uint32_t bits;
                reduce_block_words<B, R>(c[u], sb[u], cw, bits);
                const long long off = gathered + (tile0 + (gb >> 6)) * tb;
                const int g = static_cast<int>(gb & 63);
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    uint8_t *tile = static_cast<uint8_t *>(ws.p[j]) + off;
                    store_block_codes<B>(tile, g, cw);
                    store_block_scale<B>(tile, g, bits);
                }
            }
        }
    }
}

constexpr int kPeerSendUnroll = 2;  // blocks per thread in flight, as the standalone encode

template <int B, int DT>
cudaError_t run_peer_send(int R, int rank, const void *x, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long NB = 64 * T;
    auto kern = peer_send_kernel<B, DT, kPeerSendUnroll>;
    cudaError_t err = cudaSuccess;
    const long long units = (NB + kThreads32 * kPeerSendUnroll - 1) / (kThreads32 * kPeerSendUnroll);
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreads32, units, &err);
    if (grid <= 0) return err;
    PeerOwnerTiles dst{ws, twoshot_segment_tiles(T, R), rank, Codec<B>::kTileBytes};
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint16_t *>(x), n, dst, NB);
}

template <int B, int R>
cudaError_t run_peer_reduce_r(int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    const long long seg = twoshot_segment_tiles(T, R);
    const long long t0 = static_cast<long long>(rank) * seg;
    const long long tiles = (T < t0 + seg ? T : t0 + seg) - t0;
    if (tiles <= 0) return cudaSuccess;  // more ranks than tiles: this owner has nothing
    constexpr int U = reduce_units_per_thread<R>();
    const long long NB = 64 * tiles;
    auto kern = peer_reduce_kernel<B, R, U>;
    cudaError_t err = cudaSuccess;
    const long long units = (NB + kThreads32 * U - 1) / (kThreads32 * U);
    const int grid = peer_grid(reinterpret_cast<const void *>(kern), kThreads32, units, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint8_t *>(ws.p[rank]), ws, seg, t0, NB);
}

template <int B>
cudaError_t run_peer_reduce(int R, int rank, long long n, const MutPtrs &ws, cudaStream_t s) {
    switch (R) {
        case 1: return run_peer_reduce_r<B, 1>(rank, n, ws, s);
        case 2: return run_peer_reduce_r<B, 2>(rank, n, ws, s);
        case 3: return run_peer_reduce_r<B, 3>(rank, n, ws, s);
        case 4: return run_peer_reduce_r<B, 4>(rank, n, ws, s);
        case 5: return run_peer_reduce_r<B, 5>(rank, n, ws, s);
        case 6: return run_peer_reduce_r<B, 6>(rank, n, ws, s);
        case 7: return run_peer_reduce_r<B, 7>(rank, n, ws, s);
        case 8: return run_peer_reduce_r<B, 8>(rank, n, ws, s);
    }
    return cudaErrorInvalidValue;
}

// cuMemGetAddressRange through the runtime (the library does not link the
// driver library itself): the base of the allocation holding a pointer.
using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr *, size_t *, CUdeviceptr);

MemGetAddressRangeFn address_range_fn() {
    static const MemGetAddressRangeFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<MemGetAddressRangeFn>(nullptr);
        return reinterpret_cast<MemGetAddressRangeFn>(p);
    }();
    return fn;
}

// Mappings opened by qr_ipc_open_handle: returned pointer -> mapped base.
std::mutex g_ipc_mu;
std::multimap<uintptr_t, void *> g_ipc_open;

// The checks shared by the send and reduce calls.
qr_status_t check_peers(int bits, int R, int rank, size_t n, void *const *ws) {
    if (!ws || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (qr_tile_bytes(bits) == 0 || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    return check_peer_set(R, rank, n, ws, n > SIZE_MAX / 4 ? 0 : qr_twoshot_peer_workspace_bytes(bits, R, n));
}

}  // namespace

int peer_grid(const void *kern, int threads, long long units, cudaError_t *err) {
    return grid_for(kern, threads, units, 0, 4, err);
}

}  // namespace qrk

QR_EXPORT size_t qr_twoshot_peer_workspace_bytes(int bits, int R, size_t n) {
    const size_t tb = qr_tile_bytes(bits);
    if (tb == 0 || R < 1 || R > QR_MAX_RANKS || n == 0) return 0;
    const size_t T = n / QR_TILE_VALUES + (n % QR_TILE_VALUES != 0);
    const size_t seg = (T + R - 1) / R;
    const size_t tiles = 2 * static_cast<size_t>(R) * seg;
    if (tiles > SIZE_MAX / tb) return 0;
    return tiles * tb;
}

QR_EXPORT qr_status_t qr_twoshot_peer_send(int bits, qr_dtype_t dtype, int R, int rank, const void *x, size_t n,
                                           void *const *workspaces, qr_stream_t stream) {
    if (!x) return QR_ERR_INVALID_ARG;
    qr_status_t st = qrk::check_peers(bits, R, rank, n, workspaces);
    if (st != QR_OK) return st;
    if (dtype != QR_FP16 && dtype != QR_BF16) return QR_ERR_UNSUPPORTED;
    if (!qrk::peer_aligned16(x)) return QR_ERR_MISALIGNED;
    const size_t need = qr_twoshot_peer_workspace_bytes(bits, R, n);
    for (int r = 0; r < R; ++r)
        if (qrk::peer_overlaps(x, 2 * n, workspaces[r], need)) return QR_ERR_INVALID_ARG;
    qrk::MutPtrs ws{};
    for (int r = 0; r < R; ++r) ws.p[r] = workspaces[r];
    const long long nn = static_cast<long long>(n);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
#define QR_CASE(B)                                                                                           \
    case B:                                                                                                  \
        e = dtype == QR_BF16 ? qrk::run_peer_send<B, 1>(R, rank, x, nn, ws, s)                              \
                             : qrk::run_peer_send<B, 0>(R, rank, x, nn, ws, s);                             \
        break;
    switch (bits) {
        QR_CASE(3)
        QR_CASE(4)
        QR_CASE(6)
        QR_CASE(8)
    }
#undef QR_CASE
    return qrk::peer_from_cuda(e);
}

QR_EXPORT qr_status_t qr_twoshot_peer_reduce(int bits, int R, int rank, size_t n, void *const *workspaces,
                                             qr_stream_t stream) {
    qr_status_t st = qrk::check_peers(bits, R, rank, n, workspaces);
    if (st != QR_OK) return st;
    qrk::MutPtrs ws{};
    for (int r = 0; r < R; ++r) ws.p[r] = workspaces[r];
    const long long nn = static_cast<long long>(n);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorInvalidValue;
    switch (bits) {
        case 3: e = qrk::run_peer_reduce<3>(R, rank, nn, ws, s); break;
        case 4: e = qrk::run_peer_reduce<4>(R, rank, nn, ws, s); break;
        case 6: e = qrk::run_peer_reduce<6>(R, rank, nn, ws, s); break;
        case 8: e = qrk::run_peer_reduce<8>(R, rank, nn, ws, s); break;
    }
    return qrk::peer_from_cuda(e);
}

QR_EXPORT qr_status_t qr_twoshot_peer_decode(int bits, qr_dtype_t dtype, int R, size_t n, const void *workspace,
                                             void *y, qr_stream_t stream) {
    if (!workspace || !y || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    if (qr_tile_bytes(bits) == 0 || R > QR_MAX_RANKS || (dtype != QR_FP16 && dtype != QR_BF16))
        return QR_ERR_UNSUPPORTED;
    const size_t need = n > SIZE_MAX / 4 ? 0 : qr_twoshot_peer_workspace_bytes(bits, R, n);
    const qr_status_t st = qrk::check_peer_decode(n, workspace, y, need);
    if (st != QR_OK) return st;
    const size_t T = n / QR_TILE_VALUES + (n % QR_TILE_VALUES != 0);
    const size_t seg = (T + R - 1) / R;
    const uint8_t *gathered = static_cast<const uint8_t *>(workspace) + static_cast<size_t>(R) * seg * qr_tile_bytes(bits);
    return qrk::peer_from_cuda(qrk::launch_decode(bits, static_cast<int>(dtype), gathered, static_cast<long long>(n),
                                                  y, reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT size_t qr_ipc_handle_bytes(void) { return QR_IPC_HANDLE_BYTES; }

QR_EXPORT qr_status_t qr_ipc_get_handle(const void *dev_ptr, void *handle) {
    if (!dev_ptr || !handle) return QR_ERR_INVALID_ARG;
    const qrk::MemGetAddressRangeFn range = qrk::address_range_fn();
    if (!range) return QR_ERR_CUDA;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, reinterpret_cast<CUdeviceptr>(dev_ptr)) != CUDA_SUCCESS) return QR_ERR_CUDA;
    cudaIpcMemHandle_t h;
    if (cudaIpcGetMemHandle(&h, reinterpret_cast<void *>(base)) != cudaSuccess) return QR_ERR_CUDA;
    const uint64_t offset = reinterpret_cast<uintptr_t>(dev_ptr) - static_cast<uintptr_t>(base);
    static_assert(sizeof(h) + sizeof(offset) == QR_IPC_HANDLE_BYTES, "handle layout");
    std::memcpy(handle, &h, sizeof h);
    std::memcpy(static_cast<unsigned char *>(handle) + sizeof h, &offset, sizeof offset);
    return QR_OK;
}

QR_EXPORT qr_status_t qr_ipc_open_handle(const void *handle, void **dev_ptr) {
    if (!handle || !dev_ptr) return QR_ERR_INVALID_ARG;
    cudaIpcMemHandle_t h;
    uint64_t offset = 0;
    std::memcpy(&h, handle, sizeof h);
    std::memcpy(&offset, static_cast<const unsigned char *>(handle) + sizeof h, sizeof offset);
    void *base = nullptr;
    if (cudaIpcOpenMemHandle(&base, h, cudaIpcMemLazyEnablePeerAccess) != cudaSuccess) return QR_ERR_CUDA;
    void *p = static_cast<unsigned char *>(base) + offset;
    {
        std::lock_guard<std::mutex> lock(qrk::g_ipc_mu);
        qrk::g_ipc_open.emplace(reinterpret_cast<uintptr_t>(p), base);
    }
    *dev_ptr = p;
    return QR_OK;
}

QR_EXPORT qr_status_t qr_ipc_close_handle(void *dev_ptr) {
    if (!dev_ptr) return QR_ERR_INVALID_ARG;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(qrk::g_ipc_mu);
        auto it = qrk::g_ipc_open.find(reinterpret_cast<uintptr_t>(dev_ptr));
        if (it == qrk::g_ipc_open.end()) return QR_ERR_INVALID_ARG;
        base = it->second;
        qrk::g_ipc_open.erase(it);
    }
    return cudaIpcCloseMemHandle(base) == cudaSuccess ? QR_OK : QR_ERR_CUDA;
}
