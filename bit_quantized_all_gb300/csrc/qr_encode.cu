// qr_encode.cu -- launcher of the send-path kernel (encode_kernel).
#include "qr_kernels.cuh"
#include "qr_launch.h"

namespace qrk {

template <int B, int DT>
static cudaError_t run_encode(const void *x, long long n, void *wire, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    auto kern = encode_kernel<B, DT>;
    cudaError_t err = cudaSuccess;
    const int grid = grid_for(reinterpret_cast<const void *>(kern), kThreads, T, 0, &err);
    if (grid <= 0) return err;
    kern<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t *>(x), n, static_cast<uint8_t *>(wire), T);
    return cudaGetLastError();
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
