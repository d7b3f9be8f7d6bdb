// qr_launch.h -- internal host interface between the C ABI (qr_capi.cu) and
// the per-kernel translation units.  Arguments arrive already validated.
#pragma once

#include <cuda_runtime.h>

namespace qrk {

// Launches `kernel` on `s` with programmatic stream serialization: the grid
// may begin while the previous kernel on the stream is finishing; the kernel
// must call chain_entry() (qr_device.cuh) before it touches global memory,
// which makes it wait for that kernel's completion.  Returns the launch's
// error, else any error already pending.
template <class... Params, class... Args>
cudaError_t launch_chained(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// CTAs for a grid-stride launch over `tiles` work units: `ctas` if positive,
// else `waves` full waves of resident CTAs of `kernel` (launched with
// `threads` threads per CTA) on the current device; capped at `tiles`.
// Returns 0 (with *err set) if the device cannot be queried.
int grid_for(const void *kernel, int threads, long long tiles, int ctas, int waves, cudaError_t *err);

// Streaming multiprocessors of the current device (cached); 0 on error.
int sm_count(cudaError_t *err);

// A number that identifies the calling thread's current CUDA context for the
// life of the process (cuCtxGetId + 1; never reused, unlike a device ordinal
// or a context handle after cudaDeviceReset); 0 with *err set on failure.
// If no context is current yet, the current device's primary context is
// initialized first.
unsigned long long context_id(cudaError_t *err);

// The device address of a __device__ symbol of this library in the current
// context (cudaGetSymbolAddress, cached per context and symbol, so that an
// address from a context that was torn down is never reused).
cudaError_t context_symbol_address(const void *symbol, void **ptr);

// Raises the dynamic shared-memory limit of `kernel` to `bytes` in the
// current context (once per context and kernel).
cudaError_t allow_dynamic_smem(const void *kernel, int bytes);

// Device address of the library's wait-timeout counter in the current
// context (qr_timeouts.cu); nullptr with *err set on failure.
unsigned *wait_timeout_counter(cudaError_t *err);

cudaError_t launch_encode(int bits, int dtype, const void *x, long long n, void *wire,
                          cudaStream_t s);
cudaError_t launch_decode(int bits, int dtype, const void *wire, long long n, void *y,
                          cudaStream_t s);
cudaError_t launch_reduce(int bits, int R, const void *const *wires, long long n, void *out,
                          cudaStream_t s);
// Phase-1B on the staged kernel (bulk copies of the R wire tiles into shared
// memory; min(ctas or #SMs, #SMs, tiles) persistent CTAs).
cudaError_t launch_reduce_staged(int bits, int R, const void *const *wires, long long n, void *out, int ctas,
                                 cudaStream_t s);
cudaError_t launch_allreduce(int bits, int dtype, int R, const void *const *x, long long n,
                             void *y, void *const *wire_out, void *red_out, int ctas,
                             cudaStream_t s);

// The FP4 codec (qr_fp4.cu): encode, decode, Phase-1B on the staged reduce
// kernel and the fused all-reduce on the staged fused kernel (every x[r]
// and y 32-byte aligned), each staged launch with min(ctas or #SMs, #SMs,
// tiles) persistent CTAs.
cudaError_t launch_fp4_encode(int dtype, const void *x, long long n, void *wire, cudaStream_t s);
cudaError_t launch_fp4_decode(int dtype, const void *wire, long long n, void *y, cudaStream_t s);
cudaError_t launch_fp4_reduce(int R, const void *const *wires, long long n, void *out, int ctas, cudaStream_t s);
cudaError_t launch_fp4_allreduce(int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                 cudaStream_t s);

struct ConstPtrs;

// The 16-values-per-thread fused kernel (every pointer 32-byte aligned, no
// wire emission), instantiated per width in qr_allreduce16_b<B>.cu.
template <int B, int DT>
cudaError_t run_allreduce16(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s);

// The staged fused kernel (bulk copies into shared memory, one persistent
// CTA per SM; every pointer 32-byte aligned) with min(ctas or #SMs, #SMs,
// full tiles) CTAs, at least one.
template <int B, int DT>
cudaError_t run_allreduce16_staged(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s);
cudaError_t launch_allreduce_staged(int bits, int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                    cudaStream_t s);

// The two-shot all-reduce with its exchange laid out per rank and per owner in
// a workspace of R*(R+1)*seg tiles, seg = twoshot_segment_tiles(T, R)
// (qr_twoshot.cu): one launch each for the R sends, the R owner reductions
// and the R decodes into y[0..R-1].
long long twoshot_segment_tiles(long long tiles, int R);
cudaError_t launch_twoshot(int bits, int dtype, int R, const void *const *x, long long n, void *const *y, void *ws,
                           cudaStream_t s);

// The same exchange in one cooperative launch, its phases joined by per-chunk
// ready flags (qr_twoshot_flags.cu); `flags` holds 2T + 1 words that the call
// zeroes before the launch.  `drop_sender` is -1, or (self-test only) a rank
// whose sends are written but never announced, so that the owners' waits
// run out.
cudaError_t launch_twoshot_flags(int bits, int dtype, int R, const void *const *x, long long n, void *const *y,
                                 void *ws, void *flags, int drop_sender, cudaStream_t s);

// The Flash Communication codec (asymmetric groups of 128): widths 4 and 8;
// the (reduce-scatter, all-gather) width pairs (4,4), (4,8) and (8,8).
cudaError_t launch_fc_encode(int bits, int dtype, const void *x, long long n, void *wire, cudaStream_t s);
cudaError_t launch_fc_decode(int bits, int dtype, const void *wire, long long n, void *y, cudaStream_t s);
cudaError_t launch_fc_reduce(int bits_in, int bits_out, int R, const void *const *wires, long long n, void *out,
                             cudaStream_t s);
cudaError_t launch_fc_reduce_staged(int bits_in, int bits_out, int R, const void *const *wires, long long n, void *out,
                                    int ctas, cudaStream_t s);
// The FP4 codec's two-shot exchange (qr_fp4_twoshot.cu): the workspace of
// qr_twoshot_workspace_bytes(4, R, n).
cudaError_t launch_fp4_twoshot(int dtype, int R, const void *const *x, long long n, void *const *y, void *ws,
                               cudaStream_t s);
// The asymmetric codec's two-shot exchange (qr_fc_twoshot.cu): the workspace
// holds R*R*seg reduce-scatter tiles, then T all-gather tiles.
cudaError_t launch_fc_twoshot(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                              void *const *y, void *ws, cudaStream_t s);
cudaError_t launch_fc_allreduce(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                                void *y, int ctas, cudaStream_t s);
template <int BRS, int BAG>
cudaError_t run_fc_allreduce(int dtype, int R, const void *const *x, long long n, void *y, int ctas, cudaStream_t s);
// The staged kernel with the Flash Communication codec at any size (every
// pointer 32-byte aligned).
cudaError_t launch_fc_allreduce_staged(int bits_rs, int bits_ag, int dtype, int R, const void *const *x, long long n,
                                       void *y, int ctas, cudaStream_t s);
template <int BRS, int BAG>
cudaError_t run_fc_allreduce_staged(int dtype, int R, const void *const *x, long long n, void *y, int ctas,
                                    cudaStream_t s);

}  // namespace qrk
