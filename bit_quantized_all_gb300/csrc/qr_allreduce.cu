// qr_allreduce.cu -- launchers of the fused two-shot kernels: the choice between
// allreduce_kernel and the 16-values-per-thread kernels, and the staged entry.
#include <cstdint>

#include "qr_kernels.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B, int DT>
static cudaError_t run_allreduce(int R, const void *const *x, long long n, void *y,
                                 void *const *wire_out, void *red_out, int ctas, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    ConstPtrs xp{};
    MutPtrs wp{};
    for (int r = 0; r < R; ++r) {
        xp.p[r] = x[r];
        wp.p[r] = wire_out ? wire_out[r] : nullptr;
    }
    const bool emit = (wire_out != nullptr) || (red_out != nullptr);
    bool aligned32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
    for (int r = 0; r < R; ++r) aligned32 = aligned32 && (reinterpret_cast<uintptr_t>(x[r]) & 31u) == 0;
    if (!emit && aligned32) return run_allreduce16<B, DT>(R, xp, n, y, ctas, s);
    auto kern = emit ? allreduce_kernel<B, DT, true> : allreduce_kernel<B, DT, false>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads, T, ctas, 1, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads, 0, s, xp, R, n, static_cast<uint16_t *>(y), wp,
                          static_cast<uint8_t *>(red_out), T);
}

cudaError_t launch_allreduce_staged(int bits, int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                    cudaStream_t s) {
    ConstPtrs xp{};
    for (int r = 0; r < R; ++r) xp.p[r] = x[r];
#define QR_CASE(B)                                                                                  \
    case B:                                                                                         \
        return dtype ? run_allreduce16_staged<B, 1>(R, xp, n, y, ctas, s)                          \
                     : run_allreduce16_staged<B, 0>(R, xp, n, y, ctas, s);
    switch (bits) {
        QR_CASE(3)
        QR_CASE(4)
        QR_CASE(6)
        QR_CASE(8)
    }
#undef QR_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_allreduce(int bits, int dtype, int R, const void *const *x, long long n, void *y,
                             void *const *wire_out, void *red_out, int ctas, cudaStream_t s) {
#define QR_CASE(B)                                                                                  \
    case B:                                                                                         \
        return dtype ? run_allreduce<B, 1>(R, x, n, y, wire_out, red_out, ctas, s)                 \
                     : run_allreduce<B, 0>(R, x, n, y, wire_out, red_out, ctas, s);
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
