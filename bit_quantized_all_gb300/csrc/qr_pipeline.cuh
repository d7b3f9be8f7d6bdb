// qr_pipeline.cuh -- the pieces of a shared-memory staging ring fed by the
// bulk-copy (TMA) engine: mbarrier set-up, arrive / expect-tx, bounded waits,
// and the global -> shared bulk copy, as inline PTX for sm_100-class GPUs.
//
// Every wait is bounded: after kWaitLimitNs of %globaltimer without the
// awaited phase completing, the wait gives up and returns false, and the
// caller records the event in the library's timeout counter (see
// qr_wait_timeouts in include/qr.h) and stops.  Nothing here traps.
#pragma once

#include <cstdint>

namespace qrk {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// One arrival plus the number of bytes the current phase still waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete; false if
// it has not completed after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; its completion counts
// the bytes against `bar`'s current phase.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Named barrier `id` over the kThreads threads of one group (a multiple of
// 32), returning whether `pred` holds in all of them.  Every thread of the
// group must arrive.
template <int kThreads>
__device__ __forceinline__ bool group_all(int id, bool pred) {
    static_assert(kThreads % 32 == 0, "whole warps");
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "n"(kThreads)
        : "memory");
    return out != 0;
}

// 32 bytes of rank slice `r` of a stage (two 16-byte shared loads) for a
// thread whose bytes start at shared address `lo` (first 16 bytes) and `hi`
// (second 16), the slice offset an immediate: with the halves exchanged
// (lo = start + 16, hi = start) w[0..3] holds bytes 16..31 and w[4..7] bytes
// 0..15.  Lanes that read 32 contiguous bytes each touch every bank twice
// per 16-byte access (lanes k and k+4 meet in the same banks); exchanging the
// order in lanes with bit 2 set makes each 8-lane phase cover all 32 banks
// once.  Two base registers and immediate offsets: R address registers kept
// live across the loop would cost as many registers as a rank's data.
template <int kOffset>
__device__ __forceinline__ void lds32(uint32_t lo, uint32_t hi, uint32_t (&w)[8]) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(lo), "n"(kOffset)
                 : "memory");
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "r"(hi), "n"(kOffset)
                 : "memory");
}

// lds32 of rank slice r (0 <= r < 8) of a stage, the slice offset
// r * kSlice as an immediate.
template <uint32_t kSlice>
__device__ __forceinline__ void lds_rank(uint32_t lo, uint32_t hi, int r, uint32_t (&w)[8]) {
    switch (r) {
        case 0: lds32<0 * kSlice>(lo, hi, w); break;
        case 1: lds32<1 * kSlice>(lo, hi, w); break;
        case 2: lds32<2 * kSlice>(lo, hi, w); break;
        case 3: lds32<3 * kSlice>(lo, hi, w); break;
        case 4: lds32<4 * kSlice>(lo, hi, w); break;
        case 5: lds32<5 * kSlice>(lo, hi, w); break;
        case 6: lds32<6 * kSlice>(lo, hi, w); break;
        default: lds32<7 * kSlice>(lo, hi, w); break;
    }
}

}  // namespace qrk
