// qr_device.cuh -- device-side building blocks of the block-quantized
// two-shot all-reduce codec for sm_103a.
//
// Sources:
//   [QR] "QuickReduce INT3 quantization and benchmarking on MI355" (AMD
//        blog), Design Highlights; Quantization and Dequantization Paths.
//   [FC] "Flash Communication" review record, arXiv 2412.04964, key machinery.
//
// Thread mapping: a CTA of 256 threads works on one 2048-value tile at a
// time; thread k owns slot k (values 8k..8k+7, one 16-byte load of fp16/bf16),
// so the 4 consecutive lanes of a quad own one 32-value block and share its
// absmax through two butterfly shuffles.  [QR] maps a block to "8 threads x 4
// fp16x2 lanes"; on sm_103a a quad of 16-byte slots keeps every load and
// store a full 128-bit access, and the wire bytes are the same either way.
//
// Rounding: every float operation on the quantization path is an explicit
// round-to-nearest intrinsic (__fmul_rn, __fadd_rn, __frcp_rn, __fmaf_rn), so
// no contraction can change a result; the library is also built -fmad=false.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace qrk {

// Entry of every kernel launched by launch_chained (qr_launch.h), before its
// first access to global memory: allow the next kernel on the stream to
// start launching (its CTAs take SMs as this grid's CTAs leave, and run up
// to their own entry), then wait until the previous kernel on the stream has
// completed and its writes are visible.  So a chained kernel sees everything
// its predecessor wrote, as with an ordinary launch, and the gap between
// back-to-back launches shrinks to the predecessor's last CTAs.  Launched
// without programmatic serialization both instructions return at once.
__device__ __forceinline__ void chain_entry() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace qrk

namespace qrk {

constexpr int kTileValues = 2048;
constexpr int kThreads = 256;  // one 8-value slot per thread
constexpr int kMaxRanks = 8;

// Adding 1.5*2^23 to |t| < 2^22 leaves an exact integer in the low mantissa
// bits, rounded half to even by the add itself (the fp32 spacing in
// [2^23, 2^24) is 1).  Adding the (even) bias as well gives the biased code.
constexpr float kRoundMagic = 12582912.0f;

template <int B>
struct Codec {
    static_assert(B == 3 || B == 4 || B == 6 || B == 8, "unsupported width");
    static constexpr int kBias = 1 << (B - 1);          // |qmin|: [-4,+3] -> [0,7] at INT3
    static constexpr int kCodeBytes = 256 * B;          // 2048 codes of B bits
    static constexpr int kTileBytes = 256 * B + 128;    // + 64 fp16 scales: 1152 (INT4), 896 (INT3)
    static constexpr float kQmin = -float(kBias);
    static constexpr float kQmax = float(kBias - 1);
    static constexpr float kInvBias = 1.0f / float(kBias);  // a power of two: exact
    static constexpr float kMagic = kRoundMagic + float(kBias);
};

// ---------------------------------------------------------------------------
// memory access
// ---------------------------------------------------------------------------

// 16-byte streaming load of read-once data (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_u16(const void *p) {
    return *reinterpret_cast<const uint16_t *>(p);
}

// ---------------------------------------------------------------------------
// fp16 / bf16 <-> fp32 (exact widening; round-half-even narrowing)
// ---------------------------------------------------------------------------

template <int DT>  // 0 = fp16, 1 = bf16
__device__ __forceinline__ void widen8(const uint4 raw, float (&v)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (DT == 1) {
            // bf16 -> fp32 is the pattern shifted into the top half [a shift, no conversion]
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

template <int DT>
__device__ __forceinline__ uint32_t narrow2(float a, float b) {
    if constexpr (DT == 1) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

template <int DT>
__device__ __forceinline__ uint16_t narrow1(float a) {
    if constexpr (DT == 1) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(a));
    } else {
        return __half_as_ushort(__float2half_rn(a));
    }
}

template <int DT>
__device__ __forceinline__ float widen1(uint16_t h) {
    if constexpr (DT == 1) {
        return __uint_as_float(uint32_t(h) << 16);
    } else {
        return __half2float(__ushort_as_half(h));
    }
}

// Slot `base` (8 values) of an n-value message; values at or past n read as
// +0 (the zero padding of the last tile).
template <int DT>
__device__ __forceinline__ void load_slot(const uint16_t *x, long long base, long long n,
                                          float (&v)[8]) {
    if (base + 8 <= n) {
        widen8<DT>(ld_stream16(x + base), v);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (base + j < n) ? widen1<DT>(x[base + j]) : 0.0f;
    }
}

template <int DT>
__device__ __forceinline__ void store_slot(uint16_t *y, long long base, long long n,
                                           const float (&v)[8]) {
    if (base + 8 <= n) {
        uint4 o;
        o.x = narrow2<DT>(v[0], v[1]);
        o.y = narrow2<DT>(v[2], v[3]);
        o.z = narrow2<DT>(v[4], v[5]);
        o.w = narrow2<DT>(v[6], v[7]);
        *reinterpret_cast<uint4 *>(y + base) = o;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (base + j < n) y[base + j] = narrow1<DT>(v[j]);
    }
}

// ---------------------------------------------------------------------------
// block scale and quantizer [QR Design Highlights; Quantization and
// Dequantization Paths: absmax -> fp16 scale -> scale, clip, round, bias]
// ---------------------------------------------------------------------------

// three-input minimum / maximum (sm_100+): one instruction for what two
// two-input ones do; exact, so the order of the operands does not matter.
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max |v[i]| over N values with three-input maxima.
template <int N>
__device__ __forceinline__ float absmax_n(const float *v) {
    static_assert(N >= 3, "at least three values");
    float a = fmax3(fabsf(v[0]), fabsf(v[1]), fabsf(v[2]));
    int i = 3;
#pragma unroll
    for (; i + 1 < N; i += 2) a = fmax3(a, fabsf(v[i]), fabsf(v[i + 1]));
    if (i < N) a = fmaxf(a, fabsf(v[i]));
    return a;
}

// Absolute maximum of the 32 values of this thread's block (4 lanes x 8).
// Every lane of the warp must call it (full-mask shuffles).
__device__ __forceinline__ float quad_absmax(const float (&v)[8]) {
    float a = absmax_n<8>(v);
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    return a;
}

struct BlockScale {
    float s;        // decode scale (an fp16 value, widened)
    float r;        // encode factor fp32_RN(1/s); 0 when s == 0
    uint32_t bits;  // the fp16 pattern written to the wire
};

template <int B>
__device__ __forceinline__ BlockScale block_scale(float absmax) {
    const float d = __fmul_rn(absmax, Codec<B>::kInvBias);  // absmax / |qmin|, exact
    uint32_t h = __half_as_ushort(__float2half_rn(d));
    if (h == 0x7C00u) h = 0x7BFFu;  // the fp16 scale saturates at 65504
    BlockScale sc;
    sc.bits = h;
    sc.s = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
    // s == 0 (zero block or fp16 underflow): r = 0 makes every t = 0, so
    // every code is the bias and the block decodes to +0.
    sc.r = (sc.s == 0.0f) ? 0.0f : __frcp_rn(sc.s);
    return sc;
}

// f[j] = clip(fp32_RN(v[j]*r), qmin, qmax) + 1.5*2^23 + bias, rounded half to
// even by the add: an exact integer whose low byte is the code u = q + bias.
// (Clipping before rounding equals rounding before clipping: the limits are
// integers.)
template <int B>
__device__ __forceinline__ void quantize8(const float (&v)[8], float r, float (&f)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float t = __fmul_rn(v[j], r);
        t = fminf(fmaxf(t, Codec<B>::kQmin), Codec<B>::kQmax);
        f[j] = __fadd_rn(t, Codec<B>::kMagic);
    }
}

// q = f - (1.5*2^23 + bias), exact.
template <int B>
__device__ __forceinline__ float magic_to_q(float f) {
    return __fadd_rn(f, -Codec<B>::kMagic);
}

// ---------------------------------------------------------------------------
// packing [QR Design Highlights: INT4 eight 4-bit codes per int32; INT3 low
// 2 bits in a uint16 q2w and the high bit in a uint8 q1w per slot]
// f[j] carry the codes in their low byte (see quantize8).
// ---------------------------------------------------------------------------

// byte_perm gathers the low bytes of a..d into one word [a0, b0, c0, d0].
__device__ __forceinline__ uint32_t gather_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    const uint32_t ab = __byte_perm(a, b, 0x0040);  // [a0, b0, a0, a0]
    const uint32_t cd = __byte_perm(c, d, 0x0040);  // [c0, d0, c0, c0]
    return __byte_perm(ab, cd, 0x5410);             // [a0, b0, c0, d0]
}

// codes of lanes 0,2,4,6 and 1,3,5,7, one per byte
__device__ __forceinline__ void even_odd_bytes(const float (&f)[8], uint32_t &even, uint32_t &odd) {
    even = gather_low_bytes(__float_as_uint(f[0]), __float_as_uint(f[2]), __float_as_uint(f[4]),
                            __float_as_uint(f[6]));
    odd = gather_low_bytes(__float_as_uint(f[1]), __float_as_uint(f[3]), __float_as_uint(f[5]),
                           __float_as_uint(f[7]));
}

// Compress the 2-bit fields at bits 4j (j = 0..7) of x into bits 2j.
__device__ __forceinline__ uint32_t compress_2_of_4(uint32_t x) {
    x &= 0x33333333u;
    x = (x | (x >> 2)) & 0x0F0F0F0Fu;
    x = (x | (x >> 4)) & 0x00FF00FFu;
    x = (x | (x >> 8)) & 0x0000FFFFu;
    return x;
}

// Inverse: the 2-bit fields at bits 2j of x (16 bits) to bits 4j.
__device__ __forceinline__ uint32_t spread_2_to_4(uint32_t x) {
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    return x;
}

// Compress the bits at 4j (j = 0..7) of x into bits j.
__device__ __forceinline__ uint32_t compress_1_of_4(uint32_t x) {
    x &= 0x11111111u;
    x = (x | (x >> 3)) & 0x03030303u;
    x = (x | (x >> 6)) & 0x000F000Fu;
    x = (x | (x >> 12)) & 0x000000FFu;
    return x;
}

// Inverse: bit j of x (8 bits) to bit 4j.
__device__ __forceinline__ uint32_t spread_1_to_4(uint32_t x) {
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;
    return x;
}

// Write the codes of slot k into the code section(s) of `tile`.
template <int B>
__device__ __forceinline__ void store_codes(uint8_t *tile, int k, const float (&f)[8]) {
    uint32_t even, odd;
    even_odd_bytes(f, even, odd);
    if constexpr (B == 8) {
        // bytes [u0..u7]
        uint2 w;
        w.x = __byte_perm(even, odd, 0x5140);  // [e0, o0, e1, o1] = [u0, u1, u2, u3]
        w.y = __byte_perm(even, odd, 0x7362);  // [u4, u5, u6, u7]
        *reinterpret_cast<uint2 *>(tile + 8 * k) = w;
    } else if constexpr (B == 4) {
        // lane j at bits 4j: byte m = u_{2m} | u_{2m+1} << 4
        *reinterpret_cast<uint32_t *>(tile + 4 * k) = even | (odd << 4);
    } else if constexpr (B == 3) {
        const uint32_t nib = even | (odd << 4);  // lane j's 3-bit code at bits 4j
        *reinterpret_cast<uint16_t *>(tile + 2 * k) = static_cast<uint16_t>(compress_2_of_4(nib));
        tile[512 + k] = static_cast<uint8_t>(compress_1_of_4(nib >> 2));
    } else {  // B == 6
        const uint32_t lo = (even & 0x0F0F0F0Fu) | ((odd & 0x0F0F0F0Fu) << 4);
        const uint32_t hi = ((even >> 4) & 0x03030303u) | (((odd >> 4) & 0x03030303u) << 4);
        // hi: lane j's top 2 bits at bits 4j (j = 2m at 8m, j = 2m+1 at 8m+4)
        *reinterpret_cast<uint32_t *>(tile + 4 * k) = lo;
        *reinterpret_cast<uint16_t *>(tile + 1024 + 2 * k) = static_cast<uint16_t>(compress_2_of_4(hi));
    }
}

// Byte m of w (m = 0..3) as the float 1.5*2^23 + w.byte[m]:
// the pattern 0x4B40_00xx.
template <int M>
__device__ __forceinline__ float byte_as_magic(uint32_t w) {
    return __uint_as_float(__byte_perm(w, 0x4B400000u, 0x7650 + M));
}

// Raw code words of one slot, as loaded from a wire tile.
struct SlotCodes {
    uint32_t a, b;  // B=8: bytes 0-3, 4-7; B=4: word; B=6: q4w, q2w; B=3: q2w, q1w
};

// The codes of lanes 0,2,4,6 (`even`) and 1,3,5,7 (`odd`) of a slot, one
// per byte.
template <int B>
__device__ __forceinline__ void slot_even_odd_codes(const SlotCodes c, uint32_t &even, uint32_t &odd) {
    if constexpr (B == 8) {
        even = __byte_perm(c.a, c.b, 0x6420);
        odd = __byte_perm(c.a, c.b, 0x7531);
    } else if constexpr (B == 4) {
        even = c.a & 0x0F0F0F0Fu;
        odd = (c.a >> 4) & 0x0F0F0F0Fu;
    } else if constexpr (B == 3) {
        const uint32_t nib = spread_2_to_4(c.a) | (spread_1_to_4(c.b) << 2);
        even = nib & 0x0F0F0F0Fu;
        odd = (nib >> 4) & 0x0F0F0F0Fu;
    } else {
        const uint32_t hi = spread_2_to_4(c.b);  // lane j's top 2 bits at 4j
        even = (c.a & 0x0F0F0F0Fu) | ((hi & 0x03030303u) << 4);
        odd = ((c.a >> 4) & 0x0F0F0F0Fu) | (((hi >> 4) & 0x03030303u) << 4);
    }
}

template <int B>
__device__ __forceinline__ void store_scale(uint8_t *tile, int k, uint32_t bits) {
    if ((k & 3) == 0)
        *reinterpret_cast<uint16_t *>(tile + Codec<B>::kCodeBytes + 2 * (k >> 2)) =
            static_cast<uint16_t>(bits);
}

// ---------------------------------------------------------------------------
// 16 values per thread (two slots, 32 bytes of fp16/bf16): two threads per
// block.  Used by the fused kernel when every pointer is 32-byte aligned.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ld_stream32(const void *p, uint32_t (&w)[8]) {
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(p));
}

__device__ __forceinline__ void st_global32(void *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 32 bytes = w[4..7] then w[0..3].
__device__ __forceinline__ void st_global32_swapped(void *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[4]), "r"(w[5]),
                 "r"(w[6]), "r"(w[7]), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
}

// 16 values at `base` of an n-value message as 8 packed words; values at or
// past n are +0.
__device__ __forceinline__ void load16(const uint16_t *x, long long base, long long n, bool full,
                                       uint32_t (&w)[8]) {
    if (full) {
        ld_stream32(x + base, w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (base + 2 * i < n) ? x[base + 2 * i] : 0u;
            const uint32_t hi = (base + 2 * i + 1 < n) ? x[base + 2 * i + 1] : 0u;
            w[i] = lo | (hi << 16);
        }
    }
}

template <int DT>
__device__ __forceinline__ void widen16(const uint32_t (&w)[8], float2 (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if constexpr (DT == 1) {
            v[i].x = __uint_as_float(w[i] << 16);
            v[i].y = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            v[i] = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        }
    }
}

// Absolute maximum of this thread's 16 values and its partner lane's.
__device__ __forceinline__ float pair_absmax(const float2 (&v)[8]) {
    const float a = absmax_n<16>(reinterpret_cast<const float *>(v));
    return fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
}

struct BlockScale2 {
    float s, r;
    uint32_t bits;
    bool low_clip;  // the lower clip can change a code for this block (see below)
};

// The block scale of block_scale(), plus whether the lower clip at qmin can
// matter.  For a normal, unsaturated fp16 scale, s = RN16(A/|qmin|) is within
// 2^-11 (relative) of A/|qmin|, so every t = RN(x * RN(1/s)) with |x| <= A is
// at least -|qmin|*(1 + 2^-10.9) > qmin - 1/2: it rounds to qmin or above and
// only the upper clip is needed.  A zero scale gives t = 0.  Only a subnormal
// scale (rounded far below A/|qmin|) or a saturated one (A/|qmin| > 65504)
// can take t below qmin - 1/2.
template <int B>
__device__ __forceinline__ BlockScale2 block_scale2(float absmax) {
    const float d = __fmul_rn(absmax, Codec<B>::kInvBias);
    uint32_t h = __half_as_ushort(__float2half_rn(d));
    BlockScale2 sc;
    sc.low_clip = (h == 0x7C00u) || (h - 1u < 0x3FFu);  // saturated, or subnormal and nonzero
    if (h == 0x7C00u) h = 0x7BFFu;
    sc.bits = h;
    sc.s = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
    sc.r = (h == 0u) ? 0.0f : __frcp_rn(sc.s);
    return sc;
}

// q = RNE(clip(RN(v * r), qmin, qmax)) as exact integer floats, two at a time.
// `low_clip` must be uniform across the warp.
template <int B>
__device__ __forceinline__ void quantize16(const float2 (&v)[8], float r, bool low_clip, float2 (&q)[8]) {
    const float2 r2 = make_float2(r, r);
    const float2 m2 = make_float2(kRoundMagic, kRoundMagic);
    const float2 nm2 = make_float2(-kRoundMagic, -kRoundMagic);
    if (low_clip) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float2 t = __fmul2_rn(v[i], r2);
            t.x = fminf(fmaxf(t.x, Codec<B>::kQmin), Codec<B>::kQmax);
            t.y = fminf(fmaxf(t.y, Codec<B>::kQmin), Codec<B>::kQmax);
            q[i] = __fadd2_rn(__fadd2_rn(t, m2), nm2);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float2 t = __fmul2_rn(v[i], r2);
            t.x = fminf(t.x, Codec<B>::kQmax);
            t.y = fminf(t.y, Codec<B>::kQmax);
            q[i] = __fadd2_rn(__fadd2_rn(t, m2), nm2);
        }
    }
}

template <int DT>
__device__ __forceinline__ void store16(uint16_t *y, long long base, long long n, bool full,
                                        const float2 (&o)[8], bool swapped_halves = false) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = narrow2<DT>(o[i].x, o[i].y);
    if (full) {
        if (swapped_halves)  // o[0..3] are values 8..15, o[4..7] values 0..7
            st_global32_swapped(y + base, w);
        else
            st_global32(y + base, w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (base + 2 * i < n) y[base + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
            if (base + 2 * i + 1 < n) y[base + 2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
        }
    }
}

// ---------------------------------------------------------------------------
// kernel parameter blocks (R pointers travel by value)
// ---------------------------------------------------------------------------
struct ConstPtrs {
    const void *p[kMaxRanks];
};
struct MutPtrs {
    void *p[kMaxRanks];
};

// p[i] for a run-time i without indexing the kernel-parameter array (which
// would copy it to local memory): one select per rank.
template <class P>
__device__ __forceinline__ P row_pointer(const P (&p)[kMaxRanks], int i) {
    P v = p[0];
#pragma unroll
    for (int r = 1; r < kMaxRanks; ++r) v = (i == r) ? p[r] : v;
    return v;
}

}  // namespace qrk
