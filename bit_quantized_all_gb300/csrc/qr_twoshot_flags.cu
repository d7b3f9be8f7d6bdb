// qr_twoshot_flags.cu -- the two-shot all-reduce of qr_twoshot.cu in one
// cooperative launch, its phases joined by ready flags (one pair per chunk
// of C tiles) instead of launch boundaries: the protocol a multi-GPU version runs between ranks
// (peers store wire tiles into the owner's buffer and raise a flag the owner
// waits on), here between CTAs of one GPU ([QR] Design Highlights: Phase-1
// sends, Phase-1B owner reduction, Phase-2 gather; [FC] key machinery).
//
// Work units (a chunk of C consecutive 2048-value tiles, 64 threads, one
// 32-value block of each tile per thread):
//   phase 1: (sender j, chunk c): quantize rank j's tiles of chunk c into
//            their owners' receive buffers recv[k][j] (owner k = t / seg),
//            then add one to sent[c] (a release);
//   phase 2: chunk c: wait until sent[c] == R (an acquire), reduce the R
//            copies of each tile into the gathered wire, set reduced[c] (a
//            release);
//   phase 3: (rank j, chunk c): wait for reduced[c], decode the chunk's
//            gathered tiles into y[j].
// Every CTA runs all its phase-1 units, then its phase-2 units, then its
// phase-3 units, and a cooperative launch keeps every CTA resident, so a
// wait only ever waits for work that itself never waits (phase 1) or waits
// only for phase 1: no cycle.  Tiles flow through the three phases as soon
// as their inputs are ready.  Data written by other CTAs during the kernel
// is read with L2 (.cg) loads after the acquire.
//
// Every wait is bounded (one second of %globaltimer).  On expiry the CTA
// raises the workspace's abort word, and the CTA that raised it first adds
// one to the library's timeout counter (so a failed launch counts exactly
// one timeout); every other wait sees the word and returns at once, so a
// failed launch ends promptly with incomplete outputs and the context usable.
// For a self-test, one sender's announcements can be left out (its tiles are
// still written), which makes the owners' waits run out.
#include <cstdint>

#include "qr_kernels32.cuh"
#include "qr_launch.h"

namespace qrk {

namespace {

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void add_release(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void store_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Thread 0 waits (bounded) until *flag >= target, then the CTA proceeds
// together; false if the wait ran out or another CTA gave up.
__device__ __forceinline__ bool cta_wait(const uint32_t *flag, uint32_t target, uint32_t *abort_word,
                                         unsigned *timeouts) {
    __shared__ int ok;
    if (threadIdx.x == 0) {
        int good = 1;
        if (ld_acquire(flag) < target) {
            const unsigned long long t0 = global_ns();
            while (ld_acquire(flag) < target) {
                if (*static_cast<volatile uint32_t *>(abort_word) != 0) {
                    good = 0;
                    break;
                }
                if (global_ns() - t0 > kWaitLimitNs) {
                    if (atomicExch(abort_word, 1u) == 0u) atomicAdd(timeouts, 1u);
                    good = 0;
                    break;
                }
            }
        }
        ok = good;
    }
    __syncthreads();
    const bool r = ok != 0;
    __syncthreads();  // `ok` is rewritten by the next wait
    return r;
}

// One block's codes and scale from a tile written during this kernel (L2 loads).
template <int B>
__device__ __forceinline__ void load_block_cg(const uint8_t *tile, int g, BlockWords<B> &c, uint32_t &sb) {
    if constexpr (B == 8) {
        const uint4 a = __ldcg(reinterpret_cast<const uint4 *>(tile + 32 * g));
        const uint4 b = __ldcg(reinterpret_cast<const uint4 *>(tile + 32 * g + 16));
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
        c.w[4] = b.x; c.w[5] = b.y; c.w[6] = b.z; c.w[7] = b.w;
    } else if constexpr (B == 4) {
        const uint4 a = __ldcg(reinterpret_cast<const uint4 *>(tile + 16 * g));
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
    } else if constexpr (B == 3) {
        const uint2 a = __ldcg(reinterpret_cast<const uint2 *>(tile + 8 * g));
        c.w[0] = a.x; c.w[1] = a.y;
        c.w[2] = __ldcg(reinterpret_cast<const unsigned int *>(tile + 512 + 4 * g));
    } else {
        const uint4 a = __ldcg(reinterpret_cast<const uint4 *>(tile + 16 * g));
        const uint2 b = __ldcg(reinterpret_cast<const uint2 *>(tile + 1024 + 8 * g));
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
        c.w[4] = b.x; c.w[5] = b.y;
    }
    sb = __ldcg(reinterpret_cast<const unsigned short *>(tile + Codec<B>::kCodeBytes + 2 * g));
}

// Work unit = a chunk of C consecutive tiles (one block of each per thread,
// all their loads issued before any arithmetic); flags are per chunk.
template <int B, int DT, int R, int C>
__global__ void __launch_bounds__(64) twoshot_flags_kernel(ConstPtrs x, long long n, MutPtrs y, uint8_t *ws,
                                                           long long T, long long seg, uint32_t *flags,
                                                           unsigned *timeouts, int drop_sender) {
    constexpr long long kTile = Codec<B>::kTileBytes;
    const int k = threadIdx.x;  // the block of each tile this thread works on
    const long long chunks = (T + C - 1) / C;
    uint32_t *sent = flags, *reduced = flags + T, *abort_word = flags + 2 * T;
    uint8_t *red = ws + static_cast<long long>(R) * R * seg * kTile;
    const auto recv_tile = [&](long long t, int j) {  // owner(t)'s copy of sender j's tile t
        const long long owner = t / seg;
        return ws + ((owner * R + j) * seg + (t - owner * seg)) * kTile;
    };

    // phase 1: sends, chunk-major so that early chunks become ready early
    for (long long u = blockIdx.x; u < R * chunks; u += gridDim.x) {
        const long long c = u / R;
        const int j = static_cast<int>(u - c * R);
        const uint16_t *xj = static_cast<const uint16_t *>(row_pointer(x.p, j));
        uint32_t raw[C][16];
#pragma unroll
        for (int i = 0; i < C; ++i)
            if (c * C + i < T) load_block_values(xj, (c * C + i) * kTileValues + 32 * k, n, raw[i]);
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const long long t = c * C + i;
            if (t < T) {
                float2 v[16], f[16];
                widen_block<DT>(raw[i], v);
                const BlockScale2 sc = block_scale2<B>(block_absmax(v));
                quantize_block_magic<B>(v, sc.r, sc.low_clip, f);
                BlockWords<B> cw;
                pack_block<B>(f, cw);
                uint8_t *dst = recv_tile(t, j);
                store_block_codes<B>(dst, k, cw);
                store_block_scale<B>(dst, k, sc.bits);
            }
        }
        __syncthreads();
        if (k == 0 && j != drop_sender) add_release(&sent[c], 1u);
    }
    // phase 2: the owners' reductions, chunk by chunk as the copies arrive
    for (long long c = blockIdx.x; c < chunks; c += gridDim.x) {
        if (!cta_wait(&sent[c], R, abort_word, timeouts)) return;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const long long t = c * C + i;
            if (t < T) {
                BlockWords<B> cw[R];
                uint32_t sb[R];
#pragma unroll
                for (int j = 0; j < R; ++j) load_block_cg<B>(recv_tile(t, j), k, cw[j], sb[j]);
                // INT4 from six ranks keeps the fp32 sum: with the exact
                // integer sum the kernel took 95 registers a thread, fewer of
                // its cooperative CTAs were resident, and R = 8 ran at 0.92
                // of the copy bandwidth instead of 0.96 (2^27 bf16 values per
                // rank); at INT6 and at INT4 up to R = 4 the exact sum was faster.
                reduce_block<B, R, (B == 4 && R >= 6)>(cw, sb, red + t * kTile, k);
            }
        }
        __syncthreads();
        if (k == 0) store_release(&reduced[c], 1u);
    }
    // phase 3: every rank decodes the gathered wire, chunk by chunk as it is reduced
    for (long long u = blockIdx.x; u < R * chunks; u += gridDim.x) {
        const long long c = u / R;
        const int j = static_cast<int>(u - c * R);
        if (!cta_wait(&reduced[c], 1u, abort_word, timeouts)) return;
        uint16_t *yj = static_cast<uint16_t *>(row_pointer(y.p, j));
        const bool y32 = (reinterpret_cast<uintptr_t>(yj) & 31u) == 0;
        BlockWords<B> cw[C];
        uint32_t sb[C];
#pragma unroll
        for (int i = 0; i < C; ++i)
            if (c * C + i < T) load_block_cg<B>(red + (c * C + i) * kTile, k, cw[i], sb[i]);
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const long long t = c * C + i;
            if (t >= T) continue;
            const float s = f16_bits_to_float(sb[i]);
            const float2 s2 = make_float2(s, s);
            float2 q[16];
            unpack_block_q<B>(cw[i], q);
            uint32_t w[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float2 o = __fmul2_rn(q[m], s2);
                w[m] = narrow2<DT>(o.x, o.y);
            }
            const long long base = t * kTileValues + 32 * k;
            if (base + 32 <= n) {
                if (y32) {  // whole 32-byte sectors per store
                    const uint32_t lo[8] = {w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]};
                    const uint32_t hi[8] = {w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]};
                    st_global32(yj + base, lo);
                    st_global32(yj + base + 16, hi);
                } else {
                    uint4 *p = reinterpret_cast<uint4 *>(yj + base);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        p[m] = make_uint4(w[4 * m], w[4 * m + 1], w[4 * m + 2], w[4 * m + 3]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    if (base + 2 * m < n) yj[base + 2 * m] = static_cast<uint16_t>(w[m] & 0xFFFFu);
                    if (base + 2 * m + 1 < n) yj[base + 2 * m + 1] = static_cast<uint16_t>(w[m] >> 16);
                }
            }
        }
    }
}

#ifndef QR_FLAGS_CHUNK_TILES
#define QR_FLAGS_CHUNK_TILES 2
#endif
constexpr int kFlagsChunkTiles = QR_FLAGS_CHUNK_TILES;  // tiles per work unit and per flag

template <int B, int DT, int R>
static cudaError_t run_flags(const ConstPtrs &xp, long long n, const MutPtrs &yp, uint8_t *ws, uint32_t *flags,
                             int drop_sender, cudaStream_t s) {
    const long long T = (n + kTileValues - 1) / kTileValues;
    long long seg = twoshot_segment_tiles(T, R);
    cudaError_t err = cudaSuccess;
    unsigned *timeouts = wait_timeout_counter(&err);
    if (!timeouts) return err;
    if ((err = cudaMemsetAsync(flags, 0, static_cast<size_t>(2 * T + 1) * sizeof(uint32_t), s)) != cudaSuccess)
        return err;
    auto kern = twoshot_flags_kernel<B, DT, R, kFlagsChunkTiles>;
    const int sms = sm_count(&err);
    if (sms <= 0) return err;
    int per_sm = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 64, 0)) != cudaSuccess) return err;
    long long grid = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
    const long long units = R * ((T + kFlagsChunkTiles - 1) / kFlagsChunkTiles);
    if (grid > units) grid = units;
    long long nn = n, TT = T;
    ConstPtrs xa = xp;
    MutPtrs ya = yp;
    int drop = drop_sender;
    void *args[] = {&xa, &nn, &ya, &ws, &TT, &seg, &flags, &timeouts, &drop};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(static_cast<unsigned>(grid)),
                                       dim3(64), args, 0, s);
}

template <int B, int DT>
static cudaError_t run_flags_r(int R, const ConstPtrs &xp, long long n, const MutPtrs &yp, uint8_t *ws,
                               uint32_t *flags, int drop, cudaStream_t s) {
    switch (R) {
        case 1: return run_flags<B, DT, 1>(xp, n, yp, ws, flags, drop, s);
        case 2: return run_flags<B, DT, 2>(xp, n, yp, ws, flags, drop, s);
        case 3: return run_flags<B, DT, 3>(xp, n, yp, ws, flags, drop, s);
        case 4: return run_flags<B, DT, 4>(xp, n, yp, ws, flags, drop, s);
        case 5: return run_flags<B, DT, 5>(xp, n, yp, ws, flags, drop, s);
        case 6: return run_flags<B, DT, 6>(xp, n, yp, ws, flags, drop, s);
        case 7: return run_flags<B, DT, 7>(xp, n, yp, ws, flags, drop, s);
        case 8: return run_flags<B, DT, 8>(xp, n, yp, ws, flags, drop, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

long long twoshot_flag_words(long long tiles) { return 2 * tiles + 1; }

cudaError_t launch_twoshot_flags(int bits, int dtype, int R, const void *const *x, long long n, void *const *y,
                                 void *ws, void *flags, int drop_sender, cudaStream_t s) {
    ConstPtrs xp{};
    MutPtrs yp{};
    for (int r = 0; r < R; ++r) {
        xp.p[r] = x[r];
        yp.p[r] = y[r];
    }
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *f = static_cast<uint32_t *>(flags);
#define QR_CASE(B)                                                                                  \
    case B:                                                                                         \
        return dtype ? run_flags_r<B, 1>(R, xp, n, yp, w, f, drop_sender, s)                       \
                     : run_flags_r<B, 0>(R, xp, n, yp, w, f, drop_sender, s);
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
