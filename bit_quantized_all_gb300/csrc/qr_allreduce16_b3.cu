// qr_allreduce16_b3.cu -- INT3 instances of the 16-values-per-thread fused kernels
// (register-fed and staged).
#include "qr_allreduce16.cuh"

namespace qrk {
template cudaError_t run_allreduce16<3, 0>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16<3, 1>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16_staged<3, 0>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
template cudaError_t run_allreduce16_staged<3, 1>(int, const ConstPtrs &, long long, void *, int, cudaStream_t);
}  // namespace qrk
