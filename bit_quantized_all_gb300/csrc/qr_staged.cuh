// qr_staged.cuh -- the fused all-reduce with its inputs staged through shared
// memory by bulk asynchronous copies, generic over the codec: a Tile policy
// supplies one rank's quantize-and-sum (accumulate), the requantize-and-store
// of a full tile (finish), and the ragged last tile (ragged<R>); QrTile
// (qr_kernels.cuh) and FcTile (qr_kernels_fc.cuh) are the two codecs.  Every
// Tile works on 16 values per thread, 128 threads per 2048-value tile, and
// its steps before the store are per value or over whole blocks / groups, so
// a thread may hold its two 8-value halves exchanged.
#pragma once

#include "qr_device.cuh"
#include "qr_launch.h"
#include "qr_pipeline.cuh"

namespace qrk {

// The fused all-reduce with the inputs staged through shared memory by the
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
template <class Tile, int R, int G, int SG, int K>
__global__ void __launch_bounds__(128 * G, 1) staged_allreduce_kernel(ConstPtrs x, long long n, uint16_t *y,
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
    chain_entry();  // the rest reads and writes global memory

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
            Tile::accumulate(w, acc, r == 0);
        }
        uint32_t rest[R - K][8];
#pragma unroll
        for (int r = K; r < R; ++r) lds_rank<kSlice>(half_a + at, half_b + at, r, rest[r - K]);
        if (!group_all<128>(1 + g, ok)) break;  // also: every thread is done reading stage s
        if (leader && issued < tiles) issue(issued++);
#pragma unroll
        for (int r = K; r < R; ++r) Tile::accumulate(rest[r - K], acc, r == 0);
        Tile::finish(acc, y, (first + j * stride) * kTileValues + 16 * k, n, swap);
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
        Tile::template ragged<R>(x, n, y, full_tiles * kTileValues + 16 * k);
}

// Launch shape for R ranks: five groups of 128 threads (20 warps: at 96
// registers a thread, the most that five warps in each of the SM's four
// register quadrants allow), each with as many stages (at most 4) as fit in
// 192 KiB of shared memory at R * 4 KiB per stage; each group sums the first
// R/2 ranks straight from shared memory and copies the other R/2 into
// registers before it releases the stage.  The 192 KiB bound matters only at
// R = 5, where two stages (200 KiB) ran at 0.93-0.94 of the copy bandwidth
// and one stage at 1.00-1.03 (2^27 / 2^28 bf16 values per rank); one stage
// instead of the most that fit changed R = 4 by < 0.5% and cost R = 3 2-3%,
// and summing (R+1)/2 ranks from shared memory instead of R/2 helped at no
// R.  Measured on GB300 with the symmetric codec at R=8 (2^27 bf16 values
// per rank, INT4 and INT3, back-to-back launches):
//   groups x early ranks:  5 x 0: 6.65 TB/s   5 x 2: 6.92   5 x 4: 6.99
//                          5 x 6: 6.84        6 x 4: 6.75   6 x 6: 6.98
//                          7 x 4: 6.50        7 x 6: 6.65   4 x 4: 6.75
// (one to three groups with deeper rings: 4.4-5.5 TB/s, too few warps to
// issue the arithmetic); the register-fed kernel 6.36 TB/s.
template <int R>
struct StagedShape {
    static constexpr int kGroups = 5;
    static constexpr int kFit = (192 * 1024) / (kGroups * R * kTileValues * 2);
    static constexpr int kStages = kFit >= 4 ? 4 : kFit;  // per group
    static constexpr int kSmemBytes = kGroups * kStages * R * kTileValues * 2;
    static constexpr int kEarlyRanks = R / 2;  // summed from shared memory before the stage is released
    static_assert(kStages >= 1, "at least one stage per group");
};

// The staged kernel with min(ctas or #SMs, #SMs, full tiles) CTAs, at least
// one; every x[r] and y 32-byte aligned.
template <class Tile, int R>
cudaError_t launch_staged(const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    using Shape = StagedShape<R>;
    auto kern = staged_allreduce_kernel<Tile, R, Shape::kGroups, Shape::kStages, Shape::kEarlyRanks>;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (sms <= 0) return err;
    if ((err = allow_dynamic_smem(reinterpret_cast<const void *>(kern), Shape::kSmemBytes)) != cudaSuccess)
        return err;
    unsigned *timeouts = wait_timeout_counter(&err);
    if (!timeouts) return err;
    const long long full_tiles = n / kTileValues;
    long long grid = ctas > 0 ? ctas : sms;  // persistent: at most one CTA per SM
    if (grid > sms) grid = sms;
    if (grid > full_tiles) grid = full_tiles;
    if (grid < 1) grid = 1;  // a message shorter than one tile: CTA 0 does the ragged tile
    return launch_chained(kern, static_cast<int>(grid), 128 * Shape::kGroups, Shape::kSmemBytes, s, xp, n,
                          static_cast<uint16_t *>(y), full_tiles, timeouts);
}

template <class Tile>
cudaError_t launch_staged(int R, const ConstPtrs &xp, long long n, void *y, int ctas, cudaStream_t s) {
    switch (R) {
        case 1: return launch_staged<Tile, 1>(xp, n, y, ctas, s);
        case 2: return launch_staged<Tile, 2>(xp, n, y, ctas, s);
        case 3: return launch_staged<Tile, 3>(xp, n, y, ctas, s);
        case 4: return launch_staged<Tile, 4>(xp, n, y, ctas, s);
        case 5: return launch_staged<Tile, 5>(xp, n, y, ctas, s);
        case 6: return launch_staged<Tile, 6>(xp, n, y, ctas, s);
        case 7: return launch_staged<Tile, 7>(xp, n, y, ctas, s);
        case 8: return launch_staged<Tile, 8>(xp, n, y, ctas, s);
    }
    return cudaErrorInvalidValue;
}

// Where the library's default takes the staged kernel: full tiles per SM from
// which it was faster than the register-fed kernel in back-to-back launches
// on GB300 (bf16, 2^20..2^28 values per rank), per codec.
//   Symmetric (INT4): with R <= 2 the register-fed kernel has warps enough
//   and stays ahead at every size; R = 3 from ~200 tiles per SM, R >= 4 from
//   ~50 (at 2^27 values per rank: +14% at R=4 and R=6, +7% at R=8).
//   Asymmetric group-128: R = 2 from ~200 tiles per SM (at 2^27: 0.91 of the
//   HBM bandwidth against 0.86, at 2^24 0.63 against 0.69), R >= 3 from ~50.
inline long long staged_min_tiles_per_sm(int R, bool asymmetric) {
    if (asymmetric) return R <= 1 ? -1 : (R == 2 ? 128 : 48);
    return R <= 2 ? -1 : (R == 3 ? 128 : 48);
}

inline bool take_staged(int R, long long n, bool asymmetric, cudaError_t *err) {
    *err = cudaSuccess;
    const long long per_sm = staged_min_tiles_per_sm(R, asymmetric);
    if (per_sm < 0) return false;
    const int sms = sm_count(err);
    return sms > 0 && n / kTileValues >= per_sm * sms;
}

}  // namespace qrk
