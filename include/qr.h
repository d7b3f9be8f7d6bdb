/*
 * qr.h -- C ABI of libqr.so: the block-quantized two-shot all-reduce codec
 * (QuickReduce / Flash Communication) on one GB300 GPU (sm_103a).
 *
 * R "ranks" are R buffers in the one GPU's memory.  Each rank's fp16/bf16
 * message is cut into 2048-value tiles; every 32 values share one fp16 decode
 * scale.  The send path quantizes a tile into a packed wire tile; Phase-1B
 * decodes the R rank copies of a tile, sums them in fp32 and re-quantizes;
 * Phase-2 decodes the reduced tile.  Sources:
 *   [QR] "QuickReduce INT3 quantization and benchmarking on MI355" (AMD blog),
 *        sections Design Highlights; Quantization and Dequantization Paths.
 *   [FC] "Flash Communication" review record, arXiv 2412.04964, key
 *        machinery (two quantization round trips: quantize, all-to-all, local
 *        sum, re-quantize, all-gather, dequantize; one fused kernel).
 *
 * ---------------------------------------------------------------------------
 * Arithmetic (fixed; GPU results are bit-exact against it):
 *   per 32-value block: A = max|x|;  s = fp16_RNE(A / |qmin|), saturated at
 *   65504, and if s == 0 every code is the bias and the stored scale is +0;
 *   r = fp32_RN(1/s);  q = round_half_even(clip(fp32_RN(x*r), qmin, qmax));
 *   code u = q + bias;  decode = (u - bias) * s (exact in fp32).
 *   qmin = -2^(bits-1), qmax = 2^(bits-1) - 1, bias = 2^(bits-1).
 *   Phase-1B: acc = sum over r = 0..R-1 (in that order, each add rounded to
 *   fp32) of the decoded rank values; the reduced tile is the encode of acc.
 *   Phase-2: out = fp16/bf16 round-half-even of the decoded reduced value
 *   (an fp16 output that overflows becomes +-inf, as a native fp16 sum would).
 *   Inputs must be finite; non-finite inputs give unspecified results.
 *
 * Wire format (part of the ABI): tile t of a wire starts at byte
 * t * qr_tile_bytes(bits).  Slot k (0..255) = values 8k..8k+7 of the tile,
 * lane j = value 8k+j; block g (0..63) = values 32g..32g+31.  Little-endian:
 *   INT8 (2176 B): byte 8k+j = u;                              scales at 2048
 *   INT6 (1664 B): u32 at 4k bits 4j..4j+3 = u & 15;
 *                  u16 at 1024+2k bits 2j..2j+1 = u >> 4;      scales at 1536
 *   INT4 (1152 B): u32 at 4k bits 4j..4j+3 = u;                scales at 1024
 *   INT3  (896 B): u16 "q2w" at 2k bits 2j..2j+1 = u & 3;
 *                  u8 "q1w" at 512+k bit j = u >> 2;           scales at 768
 *   the fp16 decode scale of block g is at (scale offset) + 2g.
 * A message of n values that is not a multiple of 2048 is zero-padded to
 * whole tiles on the wire; decoded outputs are written for the first n values
 * only (bytes of y past n are never touched).
 *
 * ---------------------------------------------------------------------------
 * Conventions of every compute entry point:
 *   - All pointers are DEVICE pointers on the current CUDA device, except the
 *     arrays of R pointers (`x`, `wires`, `wire_out`), which are HOST arrays
 *     holding R device pointers.  Every device pointer must be 16-byte aligned.
 *   - fp16/bf16 values are raw 16-bit patterns, n values contiguous.
 *   - The caller owns and allocates every buffer; the library allocates no
 *     memory.  Work is enqueued asynchronously on `stream` (NULL = the legacy
 *     default stream); buffers must stay alive until the stream has run it.
 *   - Arguments are validated on the host before anything is enqueued; on any
 *     error nothing is launched and no memory is read or written.
 *   - An output may alias an input of the same call exactly (same pointer,
 *     in-place) where noted; partial overlap is rejected.
 *   - Calls are thread-safe.  The library keeps only a per-device cache of
 *     launch limits (SM count, occupancy), a per-context cache of what lives
 *     in a CUDA context (the staged kernels' shared-memory limits, the
 *     device addresses of the library's own device variables), filled on
 *     first use, and a counter of device-side waits that ran out
 *     (qr_wait_timeouts).  The first launch of each staged kernel in a
 *     context does this setup (a function attribute and a symbol address);
 *     make it before any stream capture.  The per-context entries are keyed
 *     by the context's id, so after cudaDeviceReset (or any other teardown
 *     and re-creation of the context) the first call in the new context
 *     repeats the setup instead of reusing addresses of the old one.
 *   - Stream order is kept, with the launches chained: every kernel is
 *     launched with programmatic stream serialization and, before it reads
 *     or writes global memory, waits until the previous kernel on the stream
 *     has completed (griddepcontrol.wait), so it sees everything that kernel
 *     wrote, as with an ordinary launch.  Its CTAs may take SMs, and run up
 *     to that wait, while the previous kernel's last CTAs finish, which
 *     removes the gap between back-to-back calls.  Each kernel also lets
 *     the next kernel on the stream start launching early
 *     (griddepcontrol.launch_dependents); a caller's own kernel launched
 *     after it with programmatic serialization must wait likewise before
 *     it reads this call's outputs.  (The flag-joined two-shot and the
 *     self-tests are launched plainly.)
 *   - Failure of a device-side wait: the staged kernels and the flag-joined
 *     two-shot bound every wait (one second).  A wait that runs out (which
 *     a correct launch never does) makes the kernel stop early and count
 *     one timeout; the call has already returned QR_OK, because it returns
 *     when the work is enqueued, and its outputs are then incomplete.  To
 *     detect this, call qr_wait_timeouts after the work has been enqueued:
 *     it waits for the device and returns the number of such timeouts since
 *     the last call (0 when every launch completed).
 */
#ifndef QR_H
#define QR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same pointer type), declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *qr_stream_t;

typedef enum {
    QR_OK = 0,
    QR_ERR_INVALID_ARG = 1, /* null pointer, n == 0, R < 1, partial aliasing */
    QR_ERR_UNSUPPORTED = 2, /* bits not in {3,4,6,8}, unknown dtype, R > 8   */
    QR_ERR_MISALIGNED = 3,  /* a device pointer not 16-byte aligned           */
    QR_ERR_SIZE = 4,        /* a byte count overflows size_t, or a workspace
                               is smaller than the call needs                */
    QR_ERR_CUDA = 5         /* the CUDA runtime reported an error at launch   */
} qr_status_t;

typedef enum { QR_FP16 = 0, QR_BF16 = 1 } qr_dtype_t;

#define QR_MAX_RANKS 8
#define QR_TILE_VALUES 2048

/* Values per tile: 2048 (the unit of [QR] Design Highlights' per-rank tile). */
size_t qr_tile_values(void);

/* Bytes of one wire tile: 256*bits + 128 (codes, then 64 fp16 scales);
 * 1152 for INT4 and 896 for INT3 as printed in [QR] Design Highlights.
 * 0 if bits is not one of 3, 4, 6, 8. */
size_t qr_tile_bytes(int bits);

/* Bytes of the wire of an n-value message: ceil(n/2048) * qr_tile_bytes(bits);
 * 0 if bits is unsupported or the product overflows size_t. */
size_t qr_wire_bytes(int bits, size_t n);

/* Send path ([QR] Quantization and Dequantization Paths, CodecQ3::send and
 * its INT4/INT6/INT8 counterparts): quantize n fp16/bf16 values `x` into
 * `wire` (qr_wire_bytes(bits, n) bytes).  `wire` must not overlap `x`. */
qr_status_t qr_encode(int bits, qr_dtype_t dtype, const void *x, size_t n,
                      void *wire, qr_stream_t stream);

/* Phase-1B in-segment reduction ([QR] Quantization and Dequantization Paths;
 * [FC] key machinery "sums locally, re-quantizes the partial sums"): decode
 * the R wires (host array of R device pointers, each qr_wire_bytes(bits, n)
 * bytes), add them in fp32 in rank order, re-quantize into `out_wire`.
 * 1 <= R <= 8.  `out_wire` may equal one of `wires` exactly.  At INT3, INT4
 * and INT6 with R >= 2, a block whose nonzero scales are all integer
 * multiples below 2^16 of the smallest one's unit (2^(floor(log2 smin) -
 * 10); about five binades; INT6 with at most four ranks also needs the
 * multiples to sum below 2^17) is summed exactly in integers (two-way
 * 16x8-bit dot products): then no partial sum of the rank order rounds, so
 * the result is the fp32 rank-order sum's, bit for bit; other blocks are
 * summed in fp32.  Which way a block went never shows in the bytes. */
qr_status_t qr_segment_reduce(int bits, int R, const void *const *wires,
                              size_t n, void *out_wire, qr_stream_t stream);

/* qr_segment_reduce on the staged kernel, whatever the size: a persistent
 * kernel (one CTA per SM of groups of 64 threads, ten for INT4 and INT6,
 * else eight) whose groups bring the R ranks' wire tiles into shared memory
 * with bulk asynchronous copies, one to four tiles ahead, and reduce from there.
 * `ctas` = 0 for one CTA per SM,
 * else min(ctas, #SMs) (at most one per tile); the result does not depend on
 * it; ctas < 0 is QR_ERR_INVALID_ARG.  qr_segment_reduce itself takes this
 * kernel for INT4, INT6 and INT8 from 48 tiles per SM, except INT8 at R = 4,
 * INT6 at R = 2..5 and INT4 at every R >= 2, where (as for INT3 at R = 2, 7
 * and 8) it runs a kernel from registers that loads each thread's next
 * block before reducing the current one; below 48 tiles per SM, and for
 * INT3 otherwise, a kernel from registers with one block per thread.  Its waits on its
 * shared-memory barriers are bounded (see qr_wait_timeouts).  Same other
 * arguments and errors as qr_segment_reduce. */
qr_status_t qr_segment_reduce_staged(int bits, int R, const void *const *wires,
                                     size_t n, void *out_wire, int ctas,
                                     qr_stream_t stream);

/* Receive path / Phase-2 ([QR] Quantization and Dequantization Paths,
 * CodecQ3::recv): decode the first n values of `wire` into fp16/bf16 `y`.
 * The wire does not record its dtype; that is the caller's contract.
 * `y` must not overlap `wire`. */
qr_status_t qr_decode(int bits, qr_dtype_t dtype, const void *wire, size_t n,
                      void *y, qr_stream_t stream);

/* The fused two-shot all-reduce ([FC] key machinery, a single fused kernel
 * with two quantization round trips): y = decode(segment_reduce(encode(x[0]),
 * ..., encode(x[R-1]))), in one pass over HBM with every intermediate on
 * chip.  `x` is a host array of R device pointers to n values each; 1 <= R
 * <= 8.  `y` (n values) may equal one of the x[r] exactly (in-place).
 * Kernel choice (the result is the same bytes either way): with every
 * pointer 32-byte aligned, R >= 4 and at least 48 full tiles per SM (R = 3:
 * 128), the staged kernel of qr_allreduce_staged; otherwise a grid-stride
 * kernel that loads the inputs straight into registers. */
qr_status_t qr_allreduce(int bits, qr_dtype_t dtype, int R,
                         const void *const *x, size_t n, void *y,
                         qr_stream_t stream);

/* qr_allreduce that also writes what a real two-shot exchange would send:
 * `wire_out` (NULL, or a host array of R device pointers) receives each
 * rank's Phase-1 wire, byte-identical to qr_encode; `red_out` (NULL or a
 * device pointer) receives the reduced wire, byte-identical to
 * qr_segment_reduce.  Each is qr_wire_bytes(bits, n) bytes and must not
 * overlap any other buffer of the call. */
qr_status_t qr_allreduce_emit(int bits, qr_dtype_t dtype, int R,
                              const void *const *x, size_t n, void *y,
                              void *const *wire_out, void *red_out,
                              qr_stream_t stream);

/* qr_allreduce on the staged kernel, whatever the size: a persistent kernel
 * (one CTA per SM) whose CTAs bring every rank's slice of a tile into shared
 * memory with bulk asynchronous copies, one to four tiles ahead, and run the
 * arithmetic from there.  `ctas` = 0 for one CTA per SM, else min(ctas,
 * #SMs) CTAs (at least one, at most one per full tile); the result does not
 * depend on it.  Every x[r] and y must be 32-byte aligned
 * (QR_ERR_MISALIGNED otherwise); ctas < 0 is QR_ERR_INVALID_ARG.  The
 * kernel's waits on its shared-memory barriers are bounded (see
 * qr_wait_timeouts).  Same other arguments and errors as qr_allreduce. */
qr_status_t qr_allreduce_staged(int bits, qr_dtype_t dtype, int R,
                                const void *const *x, size_t n, void *y,
                                int ctas, qr_stream_t stream);

/* qr_allreduce with an explicit grid size: `ctas` > 0 runs the grid-stride
 * kernel with `ctas` CTAs over the tiles; 0 = the library's choice (what
 * qr_allreduce does).  The result does not depend on `ctas`; it is the
 * SM-count knob of [FC] key machinery ("tuning the number of streaming
 * multiprocessors"). */
qr_status_t qr_allreduce_ctas(int bits, qr_dtype_t dtype, int R,
                              const void *const *x, size_t n, void *y,
                              int ctas, qr_stream_t stream);

/* The two-shot all-reduce with its exchange laid out as across R GPUs
 * ([QR] Design Highlights and Quantization and Dequantization Paths: Phase-1
 * sends, Phase-1B in-segment reduction by the segment's owner, Phase-2
 * gather; [FC] key machinery: one all-to-all, local sum and re-quantization,
 * one all-gather).  The T tiles are cut into R segments of seg = ceil(T/R)
 * tiles, owner k holding tiles [k*seg, (k+1)*seg).  Rank j quantizes its
 * message and writes segment k into owner k's receive buffer; owner k
 * reduces the R copies of its segment into the gathered wire; every rank
 * decodes the whole gathered wire into its own output y[j].  Each phase is
 * one launch on `stream` (the sends, then the owners' reductions, then the
 * decodes), with one grid row per rank or owner doing that rank's or owner's
 * work alone.  Every y[j] equals qr_allreduce's output.
 * `workspace` (device, 16-byte aligned, at least
 * qr_twoshot_workspace_bytes(bits, R, n) bytes, owned by the caller) holds
 *   recv[k][j] at byte ((k*R + j) * seg) * qr_tile_bytes(bits): owner k's
 *              copy of sender j's segment, seg tiles each;
 *   the gathered reduced wire at byte (R*R*seg) * qr_tile_bytes(bits), in
 *              tile order (byte-identical to qr_segment_reduce's output).
 * Every byte the call reads from the workspace is written by the same call
 * first.  `y` is a host array of R device pointers; outputs must not overlap
 * each other or the workspace; y[j] may equal an input exactly (every input
 * is read before any output is written).  A workspace smaller than needed
 * returns QR_ERR_SIZE. */
size_t qr_twoshot_workspace_bytes(int bits, int R, size_t n); /* R*(R+1)*seg tiles; 0 if invalid */

qr_status_t qr_allreduce_twoshot(int bits, qr_dtype_t dtype, int R,
                                 const void *const *x, size_t n, void *const *y,
                                 void *workspace, size_t workspace_bytes,
                                 qr_stream_t stream);

/* The same two-shot exchange in one cooperative launch, its phases joined
 * by ready flags instead of launch boundaries -- the protocol a multi-GPU
 * version runs between ranks (a sender stores its quantized tiles into the
 * owner's buffer and raises the owner's flag; the owner waits for R
 * raises, reduces, and raises the "reduced" flag that the decoders wait
 * for), here between the CTAs of one GPU.  The flags are per chunk of two
 * consecutive tiles, and chunks flow through the three phases as soon as
 * their inputs are ready.  Every y[j] equals
 * qr_allreduce's output and the workspace's exchange buffers hold the same
 * bytes as qr_allreduce_twoshot's.
 * `workspace` (device, 16-byte aligned, at least
 * qr_twoshot_flags_workspace_bytes(bits, R, n) bytes) = the two-shot
 * workspace, then, 16-byte aligned, 2T + 1 32-bit flag words (T tiles:
 * "sent" flags from word 0 and "reduced" flags from word T, one word per
 * chunk used; word 2T is the abort word) that the call zeroes (on
 * `stream`) before its launch.  Every wait on a flag is bounded
 * (one second); if one runs out the launch counts a timeout (see
 * qr_wait_timeouts), every other wait returns at once, and the outputs are
 * incomplete.  Same arguments, aliasing rules and errors as
 * qr_allreduce_twoshot; QR_ERR_CUDA if the cooperative launch is refused. */
size_t qr_twoshot_flags_workspace_bytes(int bits, int R, size_t n); /* 0 if invalid */

qr_status_t qr_allreduce_twoshot_flags(int bits, qr_dtype_t dtype, int R,
                                       const void *const *x, size_t n, void *const *y,
                                       void *workspace, size_t workspace_bytes,
                                       qr_stream_t stream);

/* qr_allreduce_twoshot for callers that cannot allocate device memory (no
 * counterpart on the source pages; a convenience of this library).  Some
 * callers cannot call cudaMalloc: code running inside someone else's memory
 * budget or caching allocator, code in a phase where allocating is not
 * allowed or would synchronize the device, plain C callers without an
 * allocator.  This entry point computes exactly what qr_allreduce_twoshot
 * computes, with its workspace taken from one buffer of
 * QR_TWOSHOT_STATIC_WORKSPACE_BYTES that the library itself holds in device
 * memory: every GPU that loads the library keeps that buffer until the
 * process exits.  The caller still passes the inputs `x` and the outputs `y`.
 *   - Sizes: a call whose qr_twoshot_workspace_bytes(bits, R, n) exceeds
 *     QR_TWOSHOT_STATIC_WORKSPACE_BYTES returns QR_ERR_SIZE and does nothing
 *     (32 MiB holds, for example, R=8 at INT4 up to 6.6 M values per rank, at
 *     INT8 up to 3.5 M).
 *   - The first call made in a CUDA context looks up the buffer's device
 *     address in that context (cudaGetSymbolAddress, with the context's
 *     device current); make that first call before any stream capture.  The
 *     address is cached per context, so a context re-created after
 *     cudaDeviceReset gets its own lookup.  It allocates nothing, and neither
 *     does any later call.
 *   - All calls share the one buffer, and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (every byte a call reads is
 *     written by that call first), but calls that overlap on the GPU (on two
 *     streams, or from two threads without ordering) race on it.
 * Arguments and errors are those of qr_allreduce_twoshot without the
 * workspace. */
#define QR_TWOSHOT_STATIC_WORKSPACE_BYTES (32u << 20)

qr_status_t qr_allreduce_twoshot_static(int bits, qr_dtype_t dtype, int R,
                                        const void *const *x, size_t n,
                                        void *const *y, qr_stream_t stream);

/* ---------------------------------------------------------------------------
 * The two-shot all-reduce run by R separate ranks, each in its own process
 * (or on its own GPU), storing into the other ranks' workspaces ([QR]
 * Design Highlights: Phase-1 sends segment k of every rank's quantized
 * message to owner k, Phase-1B the owner reduces its segment, Phase-2 every
 * rank gathers all segments; [FC] key machinery: all-to-all, local sum and
 * re-quantization, all-gather, over peer-to-peer GPU memory access).
 * Every rank owns a workspace of qr_twoshot_peer_workspace_bytes(bits, R, n)
 * bytes (device, 16-byte aligned) in its own memory; with seg = ceil(T/R)
 * tiles of the T-tile wire it holds
 *   recv[s]  at byte (s*seg) * qr_tile_bytes(bits), s = 0..R-1: sender s's
 *            quantized copy of the segment this rank owns (segment j of rank
 *            j: tiles [j*seg, (j+1)*seg));
 *   gathered at byte (R*seg) * qr_tile_bytes(bits): the reduced wire in tile
 *            order, byte-identical to qr_segment_reduce's output.
 * One step is three calls on every rank, in this order: qr_twoshot_peer_send,
 * qr_twoshot_peer_reduce, qr_twoshot_peer_decode.  Before a rank starts a
 * call, the previous call of EVERY rank must have finished on the GPU (the
 * caller joins the ranks, for example by synchronizing its stream and
 * meeting the others at a host barrier): no kernel of these calls waits on
 * another rank, and a call of one rank reads what the previous call of the
 * other ranks wrote.  `workspaces` is a host array of R device pointers, as
 * mapped in the calling process: entry r is rank r's workspace (the caller's
 * own at entry `rank`; the others opened with qr_ipc_open_handle, or
 * reached by peer access between GPUs of one process); workspaces must not
 * overlap.  Every rank's decoded output equals qr_allreduce's output over
 * the R messages.  Loads and stores only: no bulk copy or multicast touches
 * another rank's memory.  Errors as for qr_allreduce_twoshot; `rank` outside
 * [0, R) is QR_ERR_INVALID_ARG.  0 from the size call means unsupported
 * bits or R, n == 0, or overflow. */
size_t qr_twoshot_peer_workspace_bytes(int bits, int R, size_t n); /* 2*R*seg tiles */

/* Phase-1 of rank `rank`: quantize its n values `x` and store segment k of
 * the wire into recv[rank] of workspaces[k], for every k. */
qr_status_t qr_twoshot_peer_send(int bits, qr_dtype_t dtype, int R, int rank,
                                 const void *x, size_t n, void *const *workspaces,
                                 qr_stream_t stream);

/* Phase-1B of owner `rank`: decode the R copies recv[0..R-1] of its segment
 * from workspaces[rank], sum them in fp32 in sender order, re-quantize, and
 * store the reduced tiles into the gathered wire of every workspace (the
 * all-gather).  An owner past the last tile (R > T) does nothing. */
qr_status_t qr_twoshot_peer_reduce(int bits, int R, int rank, size_t n,
                                   void *const *workspaces, qr_stream_t stream);

/* Phase-2 of a rank: decode the gathered wire of its own `workspace` into
 * its n-value output `y` (which must not overlap the workspace). */
qr_status_t qr_twoshot_peer_decode(int bits, qr_dtype_t dtype, int R, size_t n,
                                   const void *workspace, void *y, qr_stream_t stream);

/* Sharing a device buffer with another process (no counterpart on the source
 * pages; the plumbing of the per-rank two-shot).  A handle is
 * QR_IPC_HANDLE_BYTES bytes of host memory: the CUDA IPC handle of the
 * allocation that holds `dev_ptr`, followed by the offset of `dev_ptr` in
 * it (so buffers carved out of a larger allocation can be shared).
 * qr_ipc_get_handle fills `handle`; qr_ipc_open_handle, in another process
 * on the same node, maps it and stores the buffer's address in *dev_ptr;
 * qr_ipc_close_handle unmaps a pointer qr_ipc_open_handle returned.  A
 * process cannot open its own handles.  QR_ERR_INVALID_ARG for null
 * arguments or an unknown pointer, QR_ERR_CUDA if CUDA refuses. */
#define QR_IPC_HANDLE_BYTES 72
size_t qr_ipc_handle_bytes(void); /* QR_IPC_HANDLE_BYTES */
qr_status_t qr_ipc_get_handle(const void *dev_ptr, void *handle);
qr_status_t qr_ipc_open_handle(const void *handle, void **dev_ptr);
qr_status_t qr_ipc_close_handle(void *dev_ptr);

/* Device-side waits that ran out (no counterpart on the source pages; a
 * safety property of this library).  A kernel that waits on a shared-memory
 * barrier or on another CTA's flag gives each wait one second; if a wait
 * runs out (which a correct launch never does) the kernel adds one to a
 * counter (one per device in the current context), stops issuing work,
 * waits (again bounded) for its own copies in flight and returns, leaving
 * the context usable; its outputs are then incomplete, although the call
 * that enqueued it returned QR_OK.  A flag-joined two-shot launch that
 * fails counts exactly one timeout, however many of its waits give up.
 * qr_wait_timeouts first waits for all work this process has enqueued on
 * the current device (cudaDeviceSynchronize), then reads the counter and
 * resets it to zero in one atomic step (an increment is never lost between
 * the read and the reset), and stores the count in *count.  Call it between
 * steps, never inside a stream capture.  QR_ERR_INVALID_ARG for a null
 * `count`, QR_ERR_CUDA if a CUDA call fails. */
qr_status_t qr_wait_timeouts(unsigned *count);

/* Self-test of the bounded wait: enqueues one single-thread kernel on
 * `stream` that waits on a barrier nothing completes; after one second it
 * gives up and adds one to the qr_wait_timeouts counter.  Only for tests. */
qr_status_t qr_selftest_bounded_wait(qr_stream_t stream);

/* Self-test of the flag-joined two-shot's failure path (no counterpart on
 * the source pages; only for tests): qr_allreduce_twoshot_flags with the
 * same arguments, except that sender `drop_sender` (0 <= drop_sender < R,
 * else QR_ERR_INVALID_ARG) writes its quantized tiles into the owners'
 * buffers but never raises their "sent" flags, as a peer that stopped
 * would.  Every owner's wait then runs out after one second, the launch
 * raises the workspace's abort word (flag word 2T), counts exactly one
 * timeout (qr_wait_timeouts) and returns; the outputs are incomplete.  The
 * next normal call over the same workspace is unaffected (each call clears
 * the flag words before its launch). */
qr_status_t qr_selftest_twoshot_flags_drop(int bits, qr_dtype_t dtype, int R,
                                           const void *const *x, size_t n, void *const *y,
                                           void *workspace, size_t workspace_bytes,
                                           int drop_sender, qr_stream_t stream);

/* ---------------------------------------------------------------------------
 * The Flash Communication codec ([FC] key machinery "asymmetric group-128
 * scaling"; pith summary "group size 128", "INT4 for the reduce stage and
 * INT8 for the gather stage"; minor comments: "INT6" is that mixed scheme;
 * Algorithm 1 dequantizes from codes, a zero point z and a scale s).
 * Per group of 128 values: lo = min x, hi = max x; s = fp32_RN(fp32_RN(hi -
 * lo) / (2^b - 1)), stored as 0 below 2^-126; z = lo (a zero minimum stored
 * as +0); r = fp32_RN(1/s) (0 when s = 0); u = RNE(fp32_RN(fp32_RN(x - z) *
 * r)) (never above 2^b - 1); decode = fp32_RN(u*s + z) (one rounding).
 * Phase-1B: fp32 rank-order sum of the decoded ranks, values at or past n
 * reset to 0 (a padded zero does not decode to exactly 0), re-quantized at
 * the all-gather width.  bits is 4 or 8.
 * Wire tile (2048 values = 16 groups, 256*bits + 128 bytes, little-endian):
 * codes as INT4 / INT8 above, then 16 fp32 scales at 256*bits, then 16 fp32
 * zero points at 256*bits + 64.  Same conventions as the entry points above.
 * ------------------------------------------------------------------------ */

/* 256*bits + 128 for bits 4 and 8, else 0. */
size_t qr_fc_tile_bytes(int bits);

/* ceil(n/2048) * qr_fc_tile_bytes(bits); 0 if unsupported or on overflow. */
size_t qr_fc_wire_bytes(int bits, size_t n);

/* Send path: quantize n fp16/bf16 values into a bits-wide wire. */
qr_status_t qr_fc_encode(int bits, qr_dtype_t dtype, const void *x, size_t n,
                         void *wire, qr_stream_t stream);

/* Phase-1B: decode R bits_in-wide wires (host array of R device pointers),
 * sum in fp32 in rank order, re-quantize into a bits_out-wide wire.
 * (bits_in, bits_out) is (4,4), (4,8) or (8,8). */
qr_status_t qr_fc_segment_reduce(int bits_in, int bits_out, int R,
                                 const void *const *wires, size_t n,
                                 void *out_wire, qr_stream_t stream);

/* qr_fc_segment_reduce on the staged Phase-1B kernel at any size, as
 * qr_segment_reduce_staged (`ctas` = 0 for one CTA per SM, else min(ctas,
 * #SMs); ctas < 0 is QR_ERR_INVALID_ARG).  qr_fc_segment_reduce itself
 * takes it from 48 tiles per SM when bits_in = 8 and R >= 4, and otherwise
 * runs a grid-stride kernel from registers: one that issues the loads of a
 * thread's next tile before reducing the current one when bits_in = 4 and
 * R >= 2, or bits_in = 8 and R = 3, else one that loads two tiles at a
 * time. */
qr_status_t qr_fc_segment_reduce_staged(int bits_in, int bits_out, int R,
                                        const void *const *wires, size_t n,
                                        void *out_wire, int ctas, qr_stream_t stream);

/* Receive path / Phase-2: decode the first n values into fp16/bf16. */
qr_status_t qr_fc_decode(int bits, qr_dtype_t dtype, const void *wire, size_t n,
                         void *y, qr_stream_t stream);

/* The fused two-shot all-reduce with this codec: reduce-scatter wires at
 * bits_rs, all-gather at bits_ag -- (4,4) INT4, (8,8) INT8, (4,8) the mixed
 * "INT6".  y may equal one of the x[r] exactly (in-place).  Kernel choice as
 * for qr_allreduce, with this codec's thresholds: the staged kernel for
 * R >= 3 and at least 48 full tiles per SM (R = 2: 128), with every pointer
 * 32-byte aligned. */
qr_status_t qr_fc_allreduce(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                            const void *const *x, size_t n, void *y,
                            qr_stream_t stream);

/* qr_fc_allreduce with an explicit grid size, as qr_allreduce_ctas: `ctas` >
 * 0 runs the grid-stride (register-fed) kernel with `ctas` CTAs; 0 = the
 * library's choice.  The result does not depend on it. */
qr_status_t qr_fc_allreduce_ctas(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                                 const void *const *x, size_t n, void *y,
                                 int ctas, qr_stream_t stream);

/* qr_fc_allreduce on the staged kernel at any size, as qr_allreduce_staged:
 * `ctas` = 0 for one CTA per SM, else min(ctas, #SMs); every x[r] and y
 * 32-byte aligned (QR_ERR_MISALIGNED otherwise); ctas < 0 is
 * QR_ERR_INVALID_ARG. */
qr_status_t qr_fc_allreduce_staged(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                                   const void *const *x, size_t n, void *y,
                                   int ctas, qr_stream_t stream);

/* The asymmetric codec's two-shot exchange laid out per rank and per owner
 * ([FC] key machinery: quantize at the reduce-scatter width, all-to-all,
 * local sum and re-quantization at the all-gather width, all-gather,
 * dequantize), as qr_allreduce_twoshot for the symmetric codec: with
 * seg = ceil(T/R) tiles per owner, owner k's copy of sender j's segment at
 * reduce-scatter tile (k*R + j)*seg of `workspace`, then the gathered wire
 * (T all-gather tiles, byte-identical to qr_fc_segment_reduce's output) at
 * byte R*R*seg*qr_fc_tile_bytes(bits_rs).  Three launches on `stream`, one
 * per phase, each with one grid row per rank or owner; every y[j] receives
 * qr_fc_allreduce's output.  workspace_bytes >= qr_fc_twoshot_workspace_bytes
 * (QR_ERR_SIZE otherwise); the workspace must not overlap any x or y; a y[j]
 * may equal an x[i] exactly (in place), never partly; outputs must not
 * overlap one another.  Widths and other errors as qr_fc_allreduce. */
size_t qr_fc_twoshot_workspace_bytes(int bits_rs, int bits_ag, int R, size_t n); /* 0 if unsupported */
qr_status_t qr_fc_allreduce_twoshot(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                                    const void *const *x, size_t n, void *const *y,
                                    void *workspace, size_t workspace_bytes, qr_stream_t stream);

/* The asymmetric codec's two-shot run by R separate ranks, as
 * qr_twoshot_peer_send / _reduce / _decode for the symmetric codec (the same
 * three calls per step, the same joins between them, the same `workspaces`
 * array and aliasing rules; loads and stores only into peer memory).  With
 * seg = ceil(T/R) tiles, rank j's workspace of
 * qr_fc_twoshot_peer_workspace_bytes(bits_rs, bits_ag, R, n) bytes holds
 *   recv[s]  at byte (s*seg) * qr_fc_tile_bytes(bits_rs): sender s's copy of
 *            segment j at the reduce-scatter width;
 *   gathered at byte (R*seg) * qr_fc_tile_bytes(bits_rs): the reduced wire
 *            at the all-gather width, byte-identical to
 *            qr_fc_segment_reduce's output.
 * send quantizes rank `rank`'s message at bits_rs and stores segment k into
 * recv[rank] of workspaces[k]; reduce sums owner `rank`'s R copies in
 * sender order, re-quantizes at bits_ag and stores the tiles into the
 * gathered wire of every workspace; decode dequantizes the caller's own
 * gathered wire into y.  Every rank's output equals qr_fc_allreduce's.
 * Width pairs as qr_fc_allreduce (QR_ERR_UNSUPPORTED otherwise); `rank`
 * outside [0, R) is QR_ERR_INVALID_ARG; other errors as the symmetric
 * per-rank calls.  0 from the size call means an unsupported pair or R,
 * n == 0, or overflow. */
size_t qr_fc_twoshot_peer_workspace_bytes(int bits_rs, int bits_ag, int R, size_t n);
qr_status_t qr_fc_twoshot_peer_send(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, int rank,
                                    const void *x, size_t n, void *const *workspaces,
                                    qr_stream_t stream);
qr_status_t qr_fc_twoshot_peer_reduce(int bits_rs, int bits_ag, int R, int rank, size_t n,
                                      void *const *workspaces, qr_stream_t stream);
qr_status_t qr_fc_twoshot_peer_decode(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                                      size_t n, const void *workspace, void *y,
                                      qr_stream_t stream);

/* ---- the FP4 codec -------------------------------------------------------
 * "QuickReduce INT3 quantization and benchmarking on MI355", introduction: a
 * hardware-accelerated FP4 quantization path on MI355, "essentially
 * interchangeable" with INT4.  The page gives no format; this library reads
 * it as the INT4 block framework and tile with E2M1 elements (sign, two
 * exponent bits with bias 1, one mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6) in place of the biased integers:
 *   per block of 32 values: A = max|x|; d = fp32_RN(A / 6);
 *   s = fp16_RNE(d), saturated at 65504; s == 0 stores +0 and every code is
 *   0; r = fp32_RN(1/s); code = the E2M1 value nearest to fp32_RN(x * r),
 *   ties to the even code, saturating at +-6, the sign kept (-0 is code 8);
 *   decode = value(code) * s (exact in fp32);
 *   Phase-1B sums the R decoded copies in fp32 in rank order and
 *   re-quantizes; Phase-2 decodes and rounds to fp16/bf16 (half to even).
 * Wire: the INT4 layout -- tile t at byte t*1152; the code of value 8k+j of
 * the tile in bits 4j..4j+3 of the little-endian uint32 at byte 4k; the fp16
 * scale of block g (values 32g..32g+31) at byte 1024 + 2g.  Conversions to
 * and from E2M1 run on the native instructions.  Arguments, aliasing and
 * errors as for the symmetric codec's calls of the same name, except where
 * stated. */
size_t qr_fp4_tile_bytes(void);          /* 1152 */
size_t qr_fp4_wire_bytes(size_t n);      /* ceil(n/2048) * 1152, 0 on overflow */

qr_status_t qr_fp4_encode(qr_dtype_t dtype, const void *x, size_t n, void *wire,
                          qr_stream_t stream);

qr_status_t qr_fp4_decode(qr_dtype_t dtype, const void *wire, size_t n, void *y,
                          qr_stream_t stream);

/* Phase-1B of the FP4 codec on the staged kernel (the R wire tiles brought
 * into shared memory by bulk copies), `ctas` = 0 for one CTA per SM, else
 * min(ctas, #SMs); the result does not depend on it; ctas < 0 is
 * QR_ERR_INVALID_ARG.  With ctas = 0 and R = 2, 3 or 8, from 48 tiles per
 * SM, a kernel from registers that loads each thread's next block before
 * reducing the current one runs instead (the same bytes).  out_wire may
 * equal one of the wires exactly. */
qr_status_t qr_fp4_segment_reduce(int R, const void *const *wires, size_t n,
                                  void *out_wire, int ctas, qr_stream_t stream);

/* The FP4 codec's two-shot exchange laid out per rank and per owner, as
 * qr_allreduce_twoshot for the integer codes: the workspace of
 * qr_fp4_twoshot_workspace_bytes(R, n) (= qr_twoshot_workspace_bytes(4, R, n):
 * owner k's copy of sender j's segment at tile (k*R + j)*seg, then the
 * gathered wire, byte-identical to qr_fp4_segment_reduce's output, at tile
 * R*R*seg); three launches, one per phase, with one grid row per rank or
 * owner; every y[j] receives qr_fp4_allreduce's output.  Aliasing rules and
 * errors as qr_allreduce_twoshot. */
size_t qr_fp4_twoshot_workspace_bytes(int R, size_t n);      /* 0 if unsupported */
qr_status_t qr_fp4_allreduce_twoshot(qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                     void *const *y, void *workspace, size_t workspace_bytes,
                                     qr_stream_t stream);

/* The FP4 codec's two-shot run by R separate ranks: qr_twoshot_peer_send /
 * _reduce / _decode with FP4 in place of the integer codes -- the same
 * calls, joins, workspace layout at the 1152-byte tile
 * (qr_fp4_twoshot_peer_workspace_bytes(R, n) =
 * qr_twoshot_peer_workspace_bytes(4, R, n)), aliasing rules and errors.
 * The gathered wire is byte-identical to qr_fp4_segment_reduce's output;
 * every rank's output equals qr_fp4_allreduce's. */
size_t qr_fp4_twoshot_peer_workspace_bytes(int R, size_t n);
qr_status_t qr_fp4_twoshot_peer_send(qr_dtype_t dtype, int R, int rank, const void *x, size_t n,
                                     void *const *workspaces, qr_stream_t stream);
qr_status_t qr_fp4_twoshot_peer_reduce(int R, int rank, size_t n, void *const *workspaces,
                                       qr_stream_t stream);
qr_status_t qr_fp4_twoshot_peer_decode(qr_dtype_t dtype, int R, size_t n, const void *workspace,
                                       void *y, qr_stream_t stream);

/* The fused FP4 all-reduce D(E(sum_r D(E(x_r)))) on the staged kernel;
 * every x[r] and y 32-byte aligned (QR_ERR_MISALIGNED otherwise); `ctas` as
 * above; y may equal one of the x[r] exactly (in place). */
qr_status_t qr_fp4_allreduce(qr_dtype_t dtype, int R, const void *const *x,
                             size_t n, void *y, int ctas, qr_stream_t stream);

/* A static string naming a status code (never NULL). */
const char *qr_status_string(qr_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* QR_H */
