// qr_kernels.cuh -- the register-fed fused two-shot kernels, templated on the
// code width B and the storage type DT (0 = fp16, 1 = bf16), and their
// per-tile steps as the policy QrTile of the staged kernel (qr_staged.cuh).
// (The standalone encode, reduce and decode kernels are in qr_kernels32.cuh.)
//
// Every kernel here is a grid-stride loop over 2048-value tiles; tiles are
// independent, so any grid size gives the same bytes.  No kernel here waits
// on another CTA, allocates, or uses global scratch memory.
#pragma once

#include "qr_device.cuh"

namespace qrk {

// The fused two-shot all-reduce [FC key machinery: one fused kernel, two
// quantization round trips]: for each tile, quantize every rank's slot
// (send), dequantize and add in rank order (Phase-1B), re-quantize, and
// dequantize into y (Phase-2).  The codes never leave registers unless EMIT,
// in which case the Phase-1 rank wires and the reduced wire are written too.
template <int B, int DT, bool EMIT>
__global__ void __launch_bounds__(kThreads) allreduce_kernel(ConstPtrs x, int R, long long n, uint16_t *y,
                                                             MutPtrs wire_out, uint8_t *red_out,
                                                             long long T) {
    chain_entry();
    const int k = threadIdx.x;
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const long long base = t * kTileValues + 8 * k;
        const bool full = (t + 1) * kTileValues <= n;
        // issue every rank's 16-byte load before any arithmetic
        uint4 raw[kMaxRanks];
        if (full) {
#pragma unroll
            for (int r = 0; r < kMaxRanks; ++r)
                if (r < R) raw[r] = ld_stream16(static_cast<const uint16_t *>(x.p[r]) + base);
        }
        float acc[8];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r < R) {
                float v[8];
                if (full)
                    widen8<DT>(raw[r], v);
                else
                    load_slot<DT>(static_cast<const uint16_t *>(x.p[r]), base, n, v);
                const BlockScale sc = block_scale<B>(quad_absmax(v));
                float f[8];
                quantize8<B>(v, sc.r, f);
                if constexpr (EMIT) {
                    if (wire_out.p[r] != nullptr) {
                        uint8_t *tile = static_cast<uint8_t *>(wire_out.p[r]) + t * Codec<B>::kTileBytes;
                        store_codes<B>(tile, k, f);
                        store_scale<B>(tile, k, sc.bits);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float q = magic_to_q<B>(f[j]);
                    acc[j] = (r == 0) ? __fmul_rn(q, sc.s) : __fmaf_rn(q, sc.s, acc[j]);
                }
            }
        }
        const BlockScale sc = block_scale<B>(quad_absmax(acc));
        float f[8];
        quantize8<B>(acc, sc.r, f);
        if constexpr (EMIT) {
            if (red_out != nullptr) {
                uint8_t *tile = red_out + t * Codec<B>::kTileBytes;
                store_codes<B>(tile, k, f);
                store_scale<B>(tile, k, sc.bits);
            }
        }
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(magic_to_q<B>(f[j]), sc.s);
        store_slot<DT>(y, base, n, o);
    }
}

// The fused kernel with 16 values per thread (2 threads per block, 128
// threads per tile) and R fixed at compile time; every x[r] and y must be
// 32-byte aligned.  Same arithmetic as allreduce_kernel, fewer instructions
// per value: 256-bit loads and stores, packed f32x2 multiply / add / fma, the
// per-block scale work shared by 16 values per thread instead of 8, and the
// clip at qmin only when some block of the warp has a subnormal or
// saturated scale (block_scale2).
constexpr int kThreads16 = 128;

// Phase-1 and Phase-1B of one rank for one thread: quantize the thread's 16
// values of rank r (w; values base..base+15, or with their two 8-value
// halves exchanged -- the same way for every rank, since every step here is
// per value or over the whole block) and add their dequantized values into
// acc in rank order (acc = q*s for the first rank).  Called by whole warps
// (the absmax of a block is shared by a lane pair).
template <int B, int DT>
__device__ __forceinline__ void accumulate_rank(const uint32_t (&w)[8], float2 (&acc)[8], bool first) {
    float2 v[8], q[8];
    widen16<DT>(w, v);
    const BlockScale2 sc = block_scale2<B>(pair_absmax(v));
    quantize16<B>(v, sc.r, __any_sync(0xFFFFFFFFu, sc.low_clip), q);
    const float2 s2 = make_float2(sc.s, sc.s);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = first ? __fmul2_rn(q[i], s2) : __ffma2_rn(q[i], s2, acc[i]);
}

// Requantize the sums and write the dequantized result (Phase-2) to y[base..].
template <int B, int DT>
__device__ __forceinline__ void finish_tile(const float2 (&acc)[8], uint16_t *y, long long base, long long n,
                                            bool full, bool swapped = false) {
    const BlockScale2 sc = block_scale2<B>(pair_absmax(acc));
    float2 q[8], o[8];
    quantize16<B>(acc, sc.r, __any_sync(0xFFFFFFFFu, sc.low_clip), q);
    const float2 s2 = make_float2(sc.s, sc.s);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __fmul2_rn(q[i], s2);
    store16<DT>(y, base, n, full, o, swapped);
}

// One tile for one thread: raw[r] holds this thread's 16 values of rank r.
template <int B, int DT, int R>
__device__ __forceinline__ void allreduce16_tile(const uint32_t (&raw)[R][8], uint16_t *y, long long base,
                                                 long long n, bool full) {
    float2 acc[8];
#pragma unroll
    for (int r = 0; r < R; ++r) accumulate_rank<B, DT>(raw[r], acc, r == 0);
    finish_tile<B, DT>(acc, y, base, n, full);
}

template <int B, int DT, int R>
__global__ void __launch_bounds__(kThreads16, 4) allreduce16_kernel(ConstPtrs x, long long n, uint16_t *y,
                                                                    long long T) {
    chain_entry();
    const int k = threadIdx.x;
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const long long base = t * kTileValues + 16 * k;
        const bool full = (t + 1) * kTileValues <= n;
        uint32_t raw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) load16(static_cast<const uint16_t *>(x.p[r]), base, n, full, raw[r]);
        allreduce16_tile<B, DT, R>(raw, y, base, n, full);
    }
}

// The per-tile steps of the fused kernel as a policy for the staged kernel
// (staged_allreduce_kernel in qr_staged.cuh): one rank's quantize-and-sum,
// the requantize-and-store of a full tile, and the ragged last tile.
template <int B, int DT>
struct QrTile {
    static __device__ __forceinline__ void accumulate(const uint32_t (&w)[8], float2 (&acc)[8], bool first) {
        accumulate_rank<B, DT>(w, acc, first);
    }
    static __device__ __forceinline__ void finish(const float2 (&acc)[8], uint16_t *y, long long base, long long n,
                                                  bool swapped) {
        finish_tile<B, DT>(acc, y, base, n, true, swapped);
    }
    // Bounds-checked loads of the last, partial tile.  Not inlined: its 8R
    // conditional loads would otherwise set the register budget of the whole
    // staged kernel and push its main loop into spills.
    template <int R>
    static __device__ __noinline__ void ragged(const ConstPtrs &x, long long n, uint16_t *y, long long base) {
        uint32_t raw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) load16(static_cast<const uint16_t *>(x.p[r]), base, n, false, raw[r]);
        allreduce16_tile<B, DT, R>(raw, y, base, n, false);
    }
};

}  // namespace qrk
