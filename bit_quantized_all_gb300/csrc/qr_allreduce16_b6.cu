// qr_allreduce16_b6.cu -- INT6 instances of the 16-values-per-thread fused kernels
// (register-fed and staged).
#include "qr_allreduce16.cuh"

namespace qrk {
template cudaError_t run_allreduce16<6, 0>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16<6, 1>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16_staged<6, 0>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16_staged<6, 1>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
}  // namespace qrk
