// qr_decode.cu -- launcher of the receive-path kernel (decode_kernel).
#include "qr_kernels.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B, int DT>
static cudaError_t run_decode(const void *wire, long long n, void *y, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    auto kern = decode_kernel<B, DT>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads, T, 0, &err);
    if (grid <= 0) return err;
    kern<<<grid, kThreads, 0, s>>>(static_cast<const uint8_t *>(wire), n, static_cast<uint16_t *>(y), T);
    return cudaGetLastError();
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
