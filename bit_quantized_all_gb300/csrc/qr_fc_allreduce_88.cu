// qr_fc_allreduce_88.cu -- the INT8 reduce-scatter / INT8 all-gather instances of
// the fused Flash Communication all-reduce.
#include "qr_fc_allreduce.cuh"

namespace qrk {
template cudaError_t run_fc_allreduce<8, 8>(int, int, const void *const *, long long, void *, int, cudaStream_t);
template cudaError_t run_fc_allreduce_staged<8, 8>(int, int, const void *const *, long long, void *, int,
                                                              cudaStream_t);
}  // namespace qrk
