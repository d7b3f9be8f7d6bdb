// qr_kernels.cuh -- the fused two-shot kernels, templated on the code width
// B and the storage type DT (0 = fp16, 1 = bf16).  (The standalone encode,
// reduce and decode kernels are in qr_kernels32.cuh.)
//
// Every kernel is a grid-stride loop over 2048-value tiles; tiles are
// independent, so any grid size gives the same bytes.  No kernel waits on
// another CTA, allocates, or uses global scratch memory; the staged kernel's
// threads wait only on their own CTA's shared-memory barriers.
#pragma once

#include "qr_device.cuh"
#include "qr_pipeline.cuh"

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

// The same computation with the inputs staged through shared memory by the
// bulk-copy engine, so that HBM reads stay in flight while the warps compute
// (a register-fed kernel at 100+ registers per thread has too few warps per
// SM to keep enough loads outstanding).  Persistent: one CTA per SM made of
// G groups of 128 threads; each group is an independent pipeline over its
// own tiles t = blockIdx.x + gridDim.x * (g + G * j), j = 0, 1, ..., with a
// private ring of SG stages (stage = the R ranks' 4 KiB slices of one tile).
//   - The group's leader thread fills a stage with R bulk copies whose
//     completion is counted on the stage's mbarrier; the first SG tiles are
//     issued up front.
//   - For tile j the group waits on stage j % SG, quantizes and sums ranks
//     0..K-1 straight from the stage, copies the other R-K ranks' 32 bytes
//     per thread into registers (lanes with bit 2 set read the two 16-byte
//     halves in the other order, so that every 8 lanes cover the 32 banks
//     once; their values stay exchanged up to the store), and meets at a
//     named barrier that also
//     ANDs every thread's "my wait completed" (so the group leaves the loop
//     together, never stranding a thread in a hardware barrier); the leader
//     then refills the stage with tile j + SG and the group computes while
//     that copy is in flight.
//   - A stage is only ever filled and drained by its own group, in order, so
//     every parity wait refers to an unambiguous phase.
//   - The ragged last tile (n not a multiple of 2048) is not staged: group 0
//     of CTA 0 reads it with bounds-checked loads after its loop.
// Every mbarrier wait gives up after one second; the group then adds one to
// *timeouts, its leader waits (bounded again) for the copies it issued, and
// the group returns.
// The ragged last tile for the staged kernel, read with bounds-checked loads.
// Not inlined: its 8R conditional loads would otherwise set the register
// budget of the whole kernel and push the main loop into spills.
template <int B, int DT, int R>
__device__ __noinline__ void allreduce16_ragged_tile(const ConstPtrs &x, long long n, uint16_t *y, long long base) {
    uint32_t raw[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) load16(static_cast<const uint16_t *>(x.p[r]), base, n, false, raw[r]);
    allreduce16_tile<B, DT, R>(raw, y, base, n, false);
}

template <int B, int DT, int R, int G, int SG, int K>
__global__ void __launch_bounds__(128 * G, 1) allreduce16_staged_kernel(ConstPtrs x, long long n, uint16_t *y,
                                                                        long long full_tiles, unsigned *timeouts) {
    static_assert(G >= 1 && G <= 15 && SG >= 1, "named barriers 1..G, at least one stage per group");
    static_assert(K >= 0 && K < R, "ranks taken from shared memory before the stage is released");
    constexpr uint32_t kSlice = kTileValues * 2;  // bytes of one rank's tile
    constexpr uint32_t kStageBytes = R * kSlice;
    extern __shared__ __align__(128) uint8_t ring[];  // G * SG * R * kSlice bytes
    __shared__ __align__(8) uint64_t full[G * SG];
    __shared__ const uint8_t *src[R];  // the ranks' inputs, read by the leaders at each refill

    if (threadIdx.x == 0) {
        for (int s = 0; s < G * SG; ++s) mbar_init(&full[s], 1);
        for (int r = 0; r < R; ++r) src[r] = static_cast<const uint8_t *>(x.p[r]);
        mbar_init_fence();
    }
    __syncthreads();

    const int g = threadIdx.x / 128, k = threadIdx.x & 127;
    const bool leader = k == 0;
    // this group's tiles: t = first + j * stride, j < tiles (32-bit: a group
    // never has 2^31 tiles)
    const long long first = blockIdx.x + static_cast<long long>(gridDim.x) * g;
    const long long stride = static_cast<long long>(gridDim.x) * G;
    const int tiles = full_tiles > first ? static_cast<int>((full_tiles - first + stride - 1) / stride) : 0;
    uint8_t *my_ring = ring + static_cast<size_t>(g) * SG * kStageBytes;
    uint64_t *my_full = full + g * SG;
    // this thread's 32 bytes in a stage, first and second 16-byte half
    // (exchanged in lanes with bit 2 set: see lds32)
    const bool swap = (k >> 2) & 1;
    const uint32_t mine = smem_addr(my_ring) + 32u * k;
    const uint32_t half_a = mine + (swap ? 16u : 0u), half_b = mine + (swap ? 0u : 16u);

    auto issue = [&](int j) {  // leader only: stage j % SG <- tile j
        const int s = j % SG;
        const long long off = (first + j * stride) * kSlice;
        uint8_t *dst = my_ring + static_cast<size_t>(s) * kStageBytes;
        mbar_arrive_expect_tx(&my_full[s], kStageBytes);
#pragma unroll
        for (int r = 0; r < R; ++r) bulk_copy_g2s(dst + r * kSlice, src[r] + off, kSlice, &my_full[s]);
    };

    int issued = 0;
    if (leader)
        for (; issued < tiles && issued < SG; ++issued) issue(issued);

    int j = 0;
    for (; j < tiles; ++j) {
        const int s = j % SG;
        const bool ok = mbar_wait(&my_full[s], static_cast<uint32_t>((j / SG) & 1));
        const uint32_t at = static_cast<uint32_t>(s) * kStageBytes;
        float2 acc[8];
#pragma unroll
        for (int r = 0; r < K; ++r) {  // straight from the stage (garbage if !ok: never stored)
            uint32_t w[8];
            lds_rank<kSlice>(half_a + at, half_b + at, r, w);
            accumulate_rank<B, DT>(w, acc, r == 0);
        }
        uint32_t rest[R - K][8];
#pragma unroll
        for (int r = K; r < R; ++r) lds_rank<kSlice>(half_a + at, half_b + at, r, rest[r - K]);
        if (!group_all(1 + g, ok)) break;  // also: every thread is done reading stage s
        if (leader && issued < tiles) issue(issued++);
#pragma unroll
        for (int r = K; r < R; ++r) accumulate_rank<B, DT>(rest[r - K], acc, r == 0);
        finish_tile<B, DT>(acc, y, (first + j * stride) * kTileValues + 16 * k, n, true, swap);
    }
    if (j < tiles) {  // a wait ran out
        if (leader) {
            atomicAdd(timeouts, 1u);
            for (int i = j; i < issued; ++i)  // copies still in flight into this group's stages
                if (!mbar_wait(&my_full[i % SG], static_cast<uint32_t>((i / SG) & 1))) break;
        }
        return;
    }
    if (blockIdx.x == 0 && g == 0 && full_tiles * kTileValues < n)
        allreduce16_ragged_tile<B, DT, R>(x, n, y, full_tiles * kTileValues + 16 * k);
}

}  // namespace qrk
