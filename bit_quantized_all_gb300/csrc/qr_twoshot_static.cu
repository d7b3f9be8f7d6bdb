// qr_twoshot_static.cu -- qr_allreduce_twoshot_static: the two-shot
// all-reduce for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs where the process's
// device memory is managed by someone else (a framework's caching allocator
// or a fixed memory budget that must not grow), code inside a phase where
// allocation is not allowed or would synchronize the device, and plain C
// callers without an allocator of their own.  qr_allreduce_twoshot needs a
// workspace from its caller; this entry point instead uses one buffer that
// the library keeps in a file-scope device array of
// QR_TWOSHOT_STATIC_WORKSPACE_BYTES bytes.  Every GPU that loads the library
// holds that array until the process exits.
//
// In host code `g_twoshot_workspace` names a host-side stand-in, not a device
// address; a kernel given it would fault (or, where the GPU can reach host
// memory, silently use the wrong memory).  The device address is obtained
// with cudaGetSymbolAddress once per CUDA context, with that context's
// device current, on the first call made in it, and cached per context.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_launch.h"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_twoshot_workspace[QR_TWOSHOT_STATIC_WORKSPACE_BYTES];

// The workspace's device address in the current context.  It is looked up
// with cudaGetSymbolAddress once per CUDA context (with that context's
// device current) and cached under the context's id, so that after a
// cudaDeviceReset the address from the torn-down context is never reused.
cudaError_t workspace_address(void **ptr) {
    return qrk::context_symbol_address(reinterpret_cast<const void *>(&g_twoshot_workspace), ptr);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

QR_EXPORT qr_status_t qr_allreduce_twoshot_static(int bits, qr_dtype_t dtype, int R, const void *const *x,
                                                  size_t n, void *const *y, qr_stream_t stream) {
    // the checks of qr_allreduce_twoshot that do not involve a workspace, so
    // that a rejected call makes no CUDA call at all
    if (!x || !y || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r] || !y[r]) return QR_ERR_INVALID_ARG;
    if (qr_tile_bytes(bits) == 0 || (dtype != QR_FP16 && dtype != QR_BF16) || R > QR_MAX_RANKS)
        return QR_ERR_UNSUPPORTED;
    const size_t need = qr_twoshot_workspace_bytes(bits, R, n);
    if (n > SIZE_MAX / 4 || need == 0) return QR_ERR_SIZE;
    // a message whose exchange does not fit the library's buffer is refused
    if (need > QR_TWOSHOT_STATIC_WORKSPACE_BYTES) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || !aligned16(y[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        for (int i = 0; i < R; ++i) {
            if (y[r] != x[i] && overlaps(y[r], V, x[i], V)) return QR_ERR_INVALID_ARG;
            if (i < r && overlaps(y[r], V, y[i], V)) return QR_ERR_INVALID_ARG;
        }
    void *ws = nullptr;
    if (workspace_address(&ws) != cudaSuccess) return QR_ERR_CUDA;
    // Nothing needs clearing: every workspace byte the call reads is written
    // by the same call first (the senders fill every owner's buffers before
    // the owners read them, the owners fill the gathered wire before it is
    // decoded).
    return qr_allreduce_twoshot(bits, dtype, R, x, n, y, ws, QR_TWOSHOT_STATIC_WORKSPACE_BYTES, stream);
}
