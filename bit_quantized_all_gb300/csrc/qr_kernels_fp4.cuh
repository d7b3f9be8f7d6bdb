// qr_kernels_fp4.cuh -- the FP4 codec: the INT4 block framework and tile
// (32 values per fp16 scale, nibble of lane j at bits 4j of the slot word,
// 1152-byte tiles) with E2M1 elements in place of the biased integers
// ([QR] introduction: an FP4 quantization path on MI355, "essentially
// interchangeable" with INT4; the pages give no format, and this is the
// library's reading of it, stated in include/qr.h):
//   s = fp16_RNE(fp32_RN(absmax / 6)) saturated at 65504 (6 is the largest
//   E2M1 magnitude); s == 0 stores +0 and every code is 0;
//   r = fp32_RN(1/s); code = the E2M1 value nearest to fp32_RN(x * r), ties
//   to the even code, saturating at +-6, sign kept (so -0 is a code);
//   decode = value(code) * s, exact in fp32.
// The elements go to and from E2M1 with the native conversions
// (cvt.rn.satfinite.e2m1x2.f32 and cvt.rn.f16x2.e2m1x2, two values each).
// Kernels: encode (one 32-value block per thread), decode (two threads per
// block), the Phase-1B policy of the staged reduce kernel, and the per-tile
// policy of the staged fused kernel.
#pragma once

#include "qr_kernels32.cuh"

namespace qrk {

struct Fp4Scale {
    float s, r;
    uint32_t bits;
};

__device__ __forceinline__ Fp4Scale fp4_scale(float absmax) {
    const float d = __fdiv_rn(absmax, 6.0f);
    uint32_t h = __half_as_ushort(__float2half_rn(d));
    if (h == 0x7C00u) h = 0x7BFFu;  // the fp16 scale saturates at 65504
    Fp4Scale sc;
    sc.bits = h;
    sc.s = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
    sc.r = (h == 0u) ? 0.0f : __frcp_rn(sc.s);
    return sc;
}

// The E2M1 codes of eight values (lanes 0..7) as one slot word, lane j in
// bits 4j..4j+3.  The conversion puts its first operand in the high nibble.
__device__ __forceinline__ uint32_t e2m1_word(const float2 &a, const float2 &b, const float2 &c, const float2 &d) {
    uint32_t w;
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(w)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
    return w;
}

// The values of a slot word's eight codes, pairwise (q[m] = lanes 2m, 2m+1):
// the conversion yields both values of a byte as an fp16 pair, low nibble in
// the low half, exactly.
__device__ __forceinline__ void e2m1_word_values(uint32_t w, float2 (&q)[4]) {
    uint32_t h[4];
    e2m1_pairs_to_f16x2(w, h);
#pragma unroll
    for (int m = 0; m < 4; ++m) q[m] = __half22float2(*reinterpret_cast<const __half2 *>(&h[m]));
}

// t = fp32_RN(v * r), or +0 for a zero scale (every code 0, not -0).
__device__ __forceinline__ float2 fp4_scaled(const float2 &v, const Fp4Scale &sc) {
    const float2 t = __fmul2_rn(v, make_float2(sc.r, sc.r));
    return sc.bits == 0u ? make_float2(0.0f, 0.0f) : t;
}

// The codes of n2 = 4 * words value pairs as slot words.
template <int kWords>
__device__ __forceinline__ void fp4_quantize(const float2 *v, const Fp4Scale &sc, uint32_t (&w)[kWords]) {
#pragma unroll
    for (int k = 0; k < kWords; ++k)
        w[k] = e2m1_word(fp4_scaled(v[4 * k], sc), fp4_scaled(v[4 * k + 1], sc), fp4_scaled(v[4 * k + 2], sc),
                         fp4_scaled(v[4 * k + 3], sc));
}

// ---------------------------------------------------------------------------
// send path: one 32-value block per thread
// ---------------------------------------------------------------------------
// Block gb of x quantized into block gb & 63 of `tile`.
template <int DT>
__device__ __forceinline__ void fp4_encode_block(const uint16_t *__restrict__ x, long long n, long long gb,
                                                 uint8_t *tile) {
    uint32_t raw[16];
    load_block_values(x, gb * 32, n, raw);
    float2 v[16];
    widen_block<DT>(raw, v);
    const Fp4Scale sc = fp4_scale(block_absmax(v));
    BlockWords<4> c;
    fp4_quantize<4>(v, sc, c.w);
    store_block_codes<4>(tile, static_cast<int>(gb & 63), c);
    store_block_scale<4>(tile, static_cast<int>(gb & 63), sc.bits);
}

template <int DT>
__global__ void __launch_bounds__(kThreads32) fp4_encode_kernel(const uint16_t *__restrict__ x, long long n,
                                                                uint8_t *__restrict__ wire, long long NB) {
    chain_entry();
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb < NB; gb += S)
        fp4_encode_block<DT>(x, n, gb, wire + (gb >> 6) * Codec<4>::kTileBytes);
}

// ---------------------------------------------------------------------------
// receive path: two threads per block, 16 values and 32 output bytes each
// ---------------------------------------------------------------------------
template <int DT, bool Y32>  // Y32: y is 32-byte aligned (one 256-bit store per thread)
__device__ __forceinline__ void fp4_decode_run(const uint8_t *__restrict__ wire, long long n, uint16_t *__restrict__ y,
                                               long long NH) {
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long hb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; hb < NH; hb += S) {
        const long long gb = hb >> 1;
        const uint8_t *tile = wire + (gb >> 6) * Codec<4>::kTileBytes;
        HalfWords<4> c;
        load_half_codes<4>(tile, static_cast<int>(gb & 63), static_cast<int>(hb & 1), c);
        const float s = f16_bits_to_float(load_block_scale_bits<4>(tile, static_cast<int>(gb & 63)));
        const float2 s2 = make_float2(s, s);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float2 q[4];
            e2m1_word_values(c.w[k], q);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 o = __fmul2_rn(q[m], s2);
                w[4 * k + m] = narrow2<DT>(o.x, o.y);
            }
        }
        const long long base = hb * 16;
        if (base + 16 <= n) {
            if constexpr (Y32) {
                st_global32(y + base, w);
            } else {
                uint4 *p = reinterpret_cast<uint4 *>(y + base);
                p[0] = make_uint4(w[0], w[1], w[2], w[3]);
                p[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (base + 2 * i < n) y[base + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
                if (base + 2 * i + 1 < n) y[base + 2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
            }
        }
    }
}

template <int DT, bool Y32>
__global__ void __launch_bounds__(kThreads32) fp4_decode_kernel(const uint8_t *__restrict__ wire, long long n,
                                                                uint16_t *__restrict__ y, long long NH) {
    chain_entry();
    fp4_decode_run<DT, Y32>(wire, n, y, NH);
}

// ---------------------------------------------------------------------------
// Phase-1B: the policy of staged_reduce_kernel (one 32-value block per thread)
// ---------------------------------------------------------------------------
// The codes' fp16 values (from the native conversion) are scaled and summed
// by fp16-operand fmas into fp32 -- exact products, one rounding per add, the
// same as fp32 fmas of the widened operands; acc starts at -0, so the first
// fma returns the first rank's product exactly, signed zeros included (they
// decide E2M1 codes 0 and 8 on re-quantization).
// The re-quantized codes go to cw, the fp16 scale bits to scale_bits.
template <int R>
__device__ __forceinline__ void fp4_reduce_block_words(const BlockWords<4> (&c)[R], const uint32_t (&sb)[R],
                                                       BlockWords<4> &cw, uint32_t &scale_bits) {
    float2 acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = make_float2(-0.0f, -0.0f);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const unsigned short sh = static_cast<unsigned short>(sb[r]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h[4];
            e2m1_pairs_to_f16x2(c[r].w[k], h);
#pragma unroll
            for (int m = 0; m < 4; ++m) fma_f16x2_f16_f32(h[m], sh, acc[4 * k + m]);
        }
    }
    const Fp4Scale sc = fp4_scale(block_absmax(acc));
    fp4_quantize<4>(acc, sc, cw.w);
    scale_bits = sc.bits;
}

// fp4_reduce_block_words, written into `tile` as its block g.
template <int R>
__device__ __forceinline__ void fp4_reduce_block(const BlockWords<4> (&c)[R], const uint32_t (&sb)[R], uint8_t *tile,
                                                 int g) {
    BlockWords<4> cw;
    uint32_t bits;
    fp4_reduce_block_words<R>(c, sb, cw, bits);
    store_block_codes<4>(tile, g, cw);
    store_block_scale<4>(tile, g, bits);
}

struct Fp4Reduce {
    static constexpr int kThreads = 64;
    static constexpr int kCtaThreads = 640;
    static constexpr uint32_t kTileIn = Codec<4>::kTileBytes, kTileOut = Codec<4>::kTileBytes;
    template <int R>
    struct Regs {
        BlockWords<4> c[R];
        uint32_t sb[R];
    };
    template <int R>
    static __device__ __forceinline__ void load(const uint8_t *stage, int k, Regs<R> &g) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            load_block_codes<4>(stage + r * kTileIn, k, g.c[r]);
            g.sb[r] = load_block_scale_bits<4>(stage + r * kTileIn, k);
        }
    }
    template <int R>
    static __device__ __forceinline__ void reduce(const Regs<R> &g, uint8_t *tile_out, int k, long long, long long) {
        fp4_reduce_block<R>(g.c, g.sb, tile_out, k);
    }
};

// The FP4 per-block Phase-1B as a policy of reduce_ahead_kernel.
struct Fp4BlockReducer {
    static constexpr int kBits = 4;
    template <int R>
    static __device__ __forceinline__ void reduce(const BlockWords<4> (&c)[R], const uint32_t (&sb)[R],
                                                  uint8_t *tile, int g) {
        fp4_reduce_block<R>(c, sb, tile, g);
    }
};

// Where the FP4 Phase-1B of a long message (from 48 tiles per SM) runs
// reduce_ahead_kernel instead of the staged kernel, with how many CTAs per
// SM (0 = not).  Measured on GB300 at 2^27 (2^28) bf16 values per rank,
// fraction of the copy bandwidth, staged -> one block ahead: R=2 0.677
// (0.723) -> 0.732 (0.787), R=3 0.794 -> 0.826, R=8 0.898 (0.939) -> 0.974
// (0.994); at R = 4..7 the staged kernel was faster.
template <int R>
__host__ __device__ constexpr int fp4_reduce_ahead_min_blocks() {
    return R == 2 ? 4 : R == 3 ? 3 : R == 8 ? 2 : 0;
}

// ---------------------------------------------------------------------------
// the fused all-reduce: the per-tile policy of staged_allreduce_kernel
// (16 values per thread, two threads per block sharing the absmax)
// ---------------------------------------------------------------------------

// The E2M1 values nearest to a pair (the codes never leave the register the
// conversion writes: no packing into slot words on the way back).
__device__ __forceinline__ float2 e2m1_nearest(const float2 &t) {
    uint32_t h;
    asm("{ .reg .b8 b;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b; }"
        : "=r"(h)
        : "f"(t.x), "f"(t.y));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Quantize 16 values and return their decoded values (without the scale).
__device__ __forceinline__ void fp4_roundtrip16(const float2 (&v)[8], const Fp4Scale &sc, float2 (&q)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = e2m1_nearest(fp4_scaled(v[i], sc));
}

template <int DT>
__device__ __forceinline__ void fp4_accumulate_rank(const uint32_t (&w)[8], float2 (&acc)[8], bool first) {
    float2 v[8], q[8];
    widen16<DT>(w, v);
    const Fp4Scale sc = fp4_scale(pair_absmax(v));
    fp4_roundtrip16(v, sc, q);
    const float2 s2 = make_float2(sc.s, sc.s);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = first ? __fmul2_rn(q[i], s2) : __ffma2_rn(q[i], s2, acc[i]);
}

template <int DT>
__device__ __forceinline__ void fp4_finish_tile(const float2 (&acc)[8], uint16_t *y, long long base, long long n,
                                                bool full, bool swapped) {
    const Fp4Scale sc = fp4_scale(pair_absmax(acc));
    float2 q[8], o[8];
    fp4_roundtrip16(acc, sc, q);
    const float2 s2 = make_float2(sc.s, sc.s);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __fmul2_rn(q[i], s2);
    store16<DT>(y, base, n, full, o, swapped);
}

template <int DT>
struct Fp4Tile {
    static __device__ __forceinline__ void accumulate(const uint32_t (&w)[8], float2 (&acc)[8], bool first) {
        fp4_accumulate_rank<DT>(w, acc, first);
    }
    static __device__ __forceinline__ void finish(const float2 (&acc)[8], uint16_t *y, long long base, long long n,
                                                  bool swapped) {
        fp4_finish_tile<DT>(acc, y, base, n, true, swapped);
    }
    // Bounds-checked loads of the last, partial tile (not inlined, as for
    // the symmetric codec's tile).
    template <int R>
    static __device__ __noinline__ void ragged(const ConstPtrs &x, long long n, uint16_t *y, long long base) {
        uint32_t raw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) load16(static_cast<const uint16_t *>(x.p[r]), base, n, false, raw[r]);
        float2 acc[8];
#pragma unroll
        for (int r = 0; r < R; ++r) fp4_accumulate_rank<DT>(raw[r], acc, r == 0);
        fp4_finish_tile<DT>(acc, y, base, n, false, false);
    }
};

}  // namespace qrk
