// qr_fc_allreduce_44.cu -- the INT4 reduce-scatter / INT4 all-gather instances of
// the fused Flash Communication all-reduce.
#include "qr_fc_allreduce.cuh"

namespace qrk {
template cudaError_t run_fc_allreduce<4, 4>(int, int, const void *const *, long long, void *, int, cudaStream_t);
template cudaError_t run_fc_allreduce_staged<4, 4>(int, int, const void *const *, long long, void *, int,
                                                              cudaStream_t);
}  // namespace qrk
