// qr_encode.cu -- launcher of the send-path kernel (encode32_kernel).
#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

constexpr int kEncodeUnroll = 2;  // blocks per thread in flight (2 x 64 bytes of input)

template <int B, int DT>
static cudaError_t run_encode(const void *x, long long n, void *wire, cudaStream_t s) {
    const long long NB = 64 * ((n + kTileValues - 1) / kTileValues);
    auto kern = encode32_kernel<B, DT, kEncodeUnroll>;
    cudaError_t err = cudaSuccess;
    const long long units = (NB + kThreads32 * kEncodeUnroll - 1) / (kThreads32 * kEncodeUnroll);
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads32, units, 0, 4, &err);
    if (grid <= 0) return err;
    return launch_chained(kern, grid, kThreads32, 0, s, static_cast<const uint16_t *>(x), n,
                                     ContigTiles{static_cast<uint8_t *>(wire), Codec<B>::kTileBytes}, NB);
}

cudaError_t launch_encode(int bits, int dtype, const void *x, long long n, void *wire, cudaStream_t s) {
#define QR_CASE(B)                                                                    \
    case B:                                                                           \
        return dtype ? run_encode<B, 1>(x, n, wire, s) : run_encode<B, 0>(x, n, wire, s);
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
