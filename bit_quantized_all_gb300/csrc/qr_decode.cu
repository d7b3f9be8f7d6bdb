// qr_decode.cu -- launcher of the receive-path kernel (decode16_kernel).
#include <cstdint>

#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

constexpr int kDecodeUnroll = 4;  // half-blocks per thread in flight (7-17 wire bytes each)

template <int B, int DT>
static cudaError_t run_decode(const void *wire, long long n, void *y, cudaStream_t s) {
    const long long NH = 128 * ((n + kTileValues - 1) / kTileValues);  // half-blocks
    const bool y32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
    auto kern = y32 ? decode16_kernel<B, DT, kDecodeUnroll, true> : decode16_kernel<B, DT, kDecodeUnroll, false>;
    cudaError_t err = cudaSuccess;
    const long long units = (NH + kThreads32 * kDecodeUnroll - 1) / (kThreads32 * kDecodeUnroll);
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint8_t *>(wire), n,
                          static_cast<uint16_t *>(y), NH);
}

cudaError_t launch_decode(int bits, int dtype, const void *wire, long long n, void *y, cudaStream_t s) {
#define QR_CASE(B)                                                                    \
    case B:                                                                           \
        return dtype ? run_decode<B, 1>(wire, n, y, s) : run_decode<B, 0>(wire, n, y, s);
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
