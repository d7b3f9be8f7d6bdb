// qr_kernels32.cuh -- the standalone encode, Phase-1B reduce and decode
// kernels: one 32-value block per thread (encode32, reduce32, reduce_ahead)
// or two threads per block (decode16); the staged Phase-1B kernel
// (staged_reduce_kernel, wire tiles brought into shared memory by bulk
// copies) with the symmetric codec's policy QrReduce; and Phase-1B's exact
// integer sum.
//
// A block's codes are contiguous in each section of the wire tile (slots
// 4g..4g+3), so a thread reads or writes them with one vector access per
// section, computes the block absmax without shuffles, and the fp16 scale
// once.  Each thread works on U blocks that lie a grid stride apart and
// issues every load of all U before any arithmetic, to keep enough bytes in
// flight for HBM.  Consecutive lanes own consecutive blocks of one tile.
#pragma once

#include "qr_device.cuh"
#include "qr_pipeline.cuh"

namespace qrk {

constexpr int kThreads32 = 256;

// ---------------------------------------------------------------------------
// values: 32 fp16/bf16 values of block `gb` (64 bytes)
// ---------------------------------------------------------------------------

// Values at or past n read as +0.  Full blocks use four 16-byte loads
// (L1-cached: the four chunks of a thread share two 32-byte sectors).
__device__ __forceinline__ void load_block_values(const uint16_t *x, long long base, long long n,
                                                  uint32_t (&w)[16]) {
    if (base + 32 <= n) {
        const uint4 *p = reinterpret_cast<const uint4 *>(x + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 c = p[i];
            w[4 * i] = c.x;
            w[4 * i + 1] = c.y;
            w[4 * i + 2] = c.z;
            w[4 * i + 3] = c.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t lo = (base + 2 * i < n) ? x[base + 2 * i] : 0u;
            const uint32_t hi = (base + 2 * i + 1 < n) ? x[base + 2 * i + 1] : 0u;
            w[i] = lo | (hi << 16);
        }
    }
}

template <int DT>
__device__ __forceinline__ void widen_block(const uint32_t (&w)[16], float2 (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if constexpr (DT == 1) {
            v[i].x = __uint_as_float(w[i] << 16);
            v[i].y = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            v[i] = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        }
    }
}

__device__ __forceinline__ float block_absmax(const float2 (&v)[16]) {
    return absmax_n<32>(reinterpret_cast<const float *>(v));
}

// RN(RN(v * r) + m) in both lanes: a packed multiply, then the add as a
// packed fma by `one`, which must equal 1 without being a constant the
// compiler can see.  A packed multiply followed by a packed add was merged
// into one fma (one rounding), which changes the codes; a multiply feeding
// the multiplicand of an fma has no such merge.
__device__ __forceinline__ float2 mul_then_add2(float2 v, float r, float one, float m) {
    float2 d;
    asm("{\n\t.reg .b64 pv, pr, pt, po, pm, pd;\n\t"
        "mov.b64 pv, {%2, %3};\n\t"
        "mov.b64 pr, {%4, %4};\n\t"
        "mov.b64 po, {%5, %5};\n\t"
        "mov.b64 pm, {%6, %6};\n\t"
        "mul.rn.f32x2 pt, pv, pr;\n\t"
        "fma.rn.f32x2 pd, pt, po, pm;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(v.x), "f"(v.y), "f"(r), "f"(one), "f"(m));
    return d;
}

// INT6 codes leave the quantizer 64 above the code (kMagic6): a code of 64
// (one past the top code 63; the packing turns it into 63) then has bit 7 of
// its byte set, and no other code has.
constexpr float kMagic6 = Codec<6>::kMagic + 64.0f;

// f = clip(RN(v*r), qmin, qmax) + 1.5*2^23 + bias (the code in the low byte;
// INT6: plus 64), with the clip at qmin only where block_scale2 says it can
// matter.
//
// INT3 and INT6 without the lower clip leave the upper one to the packing:
// for a normal scale every t = RN(v*r) is at most |qmin|*(1 + 2^-10.9), so its
// code is at most |qmin| + bias (INT3: 8, INT6: 64), and the packing maps that
// one out-of-range code to qmax + bias (INT3: one subtraction per eight codes
// in pack_pair_q3's nibbles; INT6: a sign-replicating byte permute of the
// code bytes in pack_block) -- the same code as clipping t at qmax first (t
// <= qmax is unchanged by the clip; for t > qmax, RNE(t) + bias is qmax + bias
// or one more, and becomes qmax + bias, as RNE(qmax) + bias is).  That
// removes one float minimum (integer-pipe work) per value.  The product and
// the add are then two packed operations (mul_then_add2): contracted into one
// rounding they would change the codes.
template <int B>
__device__ __forceinline__ void quantize_block_magic(const float2 (&v)[16], float r, bool low_clip,
                                                     float2 (&f)[16]) {
    constexpr float kM = (B == 6) ? kMagic6 : Codec<B>::kMagic;
    const float2 r2 = make_float2(r, r);
    const float2 m2 = make_float2(kM, kM);
    if constexpr (B == 3 || B == 6) {
        if (!low_clip) {
            const float one = __fmaf_rn(r, 0.0f, 1.0f);  // 1: r is finite
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = mul_then_add2(v[i], r, one, kM);
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 t = __fmul2_rn(v[i], r2);
        if (low_clip) {
            t.x = fmaxf(t.x, Codec<B>::kQmin);
            t.y = fmaxf(t.y, Codec<B>::kQmin);
        }
        t.x = fminf(t.x, Codec<B>::kQmax);
        t.y = fminf(t.y, Codec<B>::kQmax);
        f[i] = __fadd2_rn(t, m2);
    }
}

// ---------------------------------------------------------------------------
// codes of one block: slot s = values 8s..8s+7 of the block = f[4s..4s+3]
// ---------------------------------------------------------------------------

// lanes 0,2,4,6 (the .x of the four pairs) and 1,3,5,7 (.y), one per byte
__device__ __forceinline__ void slot_even_odd(const float2 (&f)[16], int s, uint32_t &even, uint32_t &odd) {
    even = gather_low_bytes(__float_as_uint(f[4 * s].x), __float_as_uint(f[4 * s + 1].x),
                            __float_as_uint(f[4 * s + 2].x), __float_as_uint(f[4 * s + 3].x));
    odd = gather_low_bytes(__float_as_uint(f[4 * s].y), __float_as_uint(f[4 * s + 1].y),
                           __float_as_uint(f[4 * s + 2].y), __float_as_uint(f[4 * s + 3].y));
}

// Raw words of one block's codes, section by section:
//   B=8: w[0..7] (32 bytes at 32g)     B=4: w[0..3] (16 bytes at 16g)
//   B=3: w[0..1] q2w (8 bytes at 8g), w[2] q1w (4 bytes at 512 + 4g)
//   B=6: w[0..3] q4w (16 bytes at 16g), w[4..5] q2w (8 bytes at 1024 + 8g)
template <int B>
struct BlockWords {
    static constexpr int kWords = (B == 8) ? 8 : (B == 4) ? 4 : (B == 3) ? 3 : 6;
    uint32_t w[kWords];
};

// Four codes (each the low nibble of a magic float's bit pattern, lanes
// 0..3) packed little-endian into the low 16 bits of the result, bits above
// don't-care, by a chain of integer multiply-adds (which run on the FMA pipe
// and so leave the integer pipe, the bottleneck of Phase-1B, to the rest).
// A magic float is 0x4B40_0000 + u with u < 16, so its pattern equals u
// modulo 2^22; the multiplier equals 16 modulo 2^16 (its high half only
// keeps the compiler from turning it into shifts); so modulo 2^16 the chain
// is the base-16 Horner scheme u0 + 16 (u1 + 16 (u2 + 16 u3)).
__device__ __forceinline__ uint32_t nibbles4_lo16(float f0, float f1, float f2, float f3) {
    constexpr uint32_t kMul = 0x5A5A0010u;
    uint32_t t = __float_as_uint(f3) * kMul + __float_as_uint(f2);
    t = t * kMul + __float_as_uint(f1);
    return t * kMul + __float_as_uint(f0);
}

// The codes of slot s (lanes 0..7 = f[4s..4s+3] pairwise) as one word with
// lane j in bits 4j..4j+3 (each code below 16).
__device__ __forceinline__ uint32_t slot_nibbles(const float2 *f) {
    return __byte_perm(nibbles4_lo16(f[0].x, f[0].y, f[1].x, f[1].y),
                       nibbles4_lo16(f[2].x, f[2].y, f[3].x, f[3].y), 0x5410);
}

// The q2w / q1w fields of two slots from their codes in nibbles (nibble
// 4i+m of e / o: lane 2m / 2m+1 of slot i, every nibble a code 0..8): W = the
// two slots' q2w (slot 0 in bits 0..15), X = their q1w (slot 0 in bits 0..7,
// slot 1 in 8..15).  A code of 8 (a value quantize_block_magic left
// unclipped at qmax) becomes 7 by one subtraction per eight nibbles, the q2
// fields come out with one mask, and the q1 bits, masked to every fourth bit,
// are gathered by three shift-and-mask steps.
__device__ __forceinline__ void q3_fields_from_nibbles(uint32_t e, uint32_t o, uint32_t &W, uint32_t &X) {
    e -= (e >> 3) & 0x11111111u;  // 8 -> 7 (bit 3 of a nibble is set only by 8)
    o -= (o >> 3) & 0x11111111u;
    W = (e & 0x33333333u) | ((o << 2) & 0xCCCCCCCCu);
    uint32_t x = ((e >> 2) & 0x11111111u) | ((o >> 1) & 0x22222222u);
    x = (x | (x >> 2)) & 0x0F0F0F0Fu;
    x = (x | (x >> 4)) & 0x00FF00FFu;
    X = (x & 0xFFu) | ((x >> 8) & 0xFF00u);
}

// The INT3 fields of slots 2h and 2h+1 from their 16 magic floats (f[4s + m]
// = lanes 2m, 2m+1 of slot s; the code is each float's low byte), W and X as
// above.  The inverse of unpack_pair_q3: the codes go into nibbles (even
// lanes in one word, odd lanes in another) by multiply-add chains.
__device__ __forceinline__ void pack_pair_q3(const float2 (&f)[16], int h, uint32_t &W, uint32_t &X) {
    const int a = 8 * h, b = 8 * h + 4;  // f index of lane 0 of slot 2h, of slot 2h+1
    q3_fields_from_nibbles(__byte_perm(nibbles4_lo16(f[a].x, f[a + 1].x, f[a + 2].x, f[a + 3].x),
                                       nibbles4_lo16(f[b].x, f[b + 1].x, f[b + 2].x, f[b + 3].x), 0x5410),
                           __byte_perm(nibbles4_lo16(f[a].y, f[a + 1].y, f[a + 2].y, f[a + 3].y),
                                       nibbles4_lo16(f[b].y, f[b + 1].y, f[b + 2].y, f[b + 3].y), 0x5410),
                           W, X);
}

// pack_pair_q3 for magic floats paired by lane: F[L] = (lane L of slot 2h,
// lane L of slot 2h+1).
__device__ __forceinline__ void pack_pair_q3_lanes(const float2 (&F)[8], uint32_t &W, uint32_t &X) {
    q3_fields_from_nibbles(__byte_perm(nibbles4_lo16(F[0].x, F[2].x, F[4].x, F[6].x),
                                       nibbles4_lo16(F[0].y, F[2].y, F[4].y, F[6].y), 0x5410),
                           __byte_perm(nibbles4_lo16(F[1].x, F[3].x, F[5].x, F[7].x),
                                       nibbles4_lo16(F[1].y, F[3].y, F[5].y, F[7].y), 0x5410),
                           W, X);
}

// The INT6 sections of one slot from its codes as bytes (`even`: lanes
// 0,2,4,6, `odd`: lanes 1,3,5,7, each byte's low six bits a code; the bits
// above are not read): the q4w word
// (lane j's low nibble at bits 4j), and `y`, whose bytes 0 and 2 are the
// slot's q2w field (lane j's high two bits at bits 2j): byte k of c holds
// lanes 2k and 2k+1, and one shift-or pairs neighbouring bytes, so that a
// byte permute finishes the field (7 operations where three shift-and-mask
// compress steps took 12).
__device__ __forceinline__ void q6_slot_fields(uint32_t even, uint32_t odd, uint32_t &q4w, uint32_t &y) {
    q4w = (even & 0x0F0F0F0Fu) | ((odd & 0x0F0F0F0Fu) << 4);
    const uint32_t c = ((even >> 4) & 0x03030303u) | ((odd >> 2) & 0x0C0C0C0Cu);
    y = c | (c >> 4);
}

// Each byte of x replaced by 0xFF where its bit 7 is set, else 0 (one byte
// permute in its sign-replicating mode, which the __byte_perm intrinsic does
// not promise).
__device__ __forceinline__ uint32_t sign_bytes(uint32_t x) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %1, 0xBA98;" : "=r"(d) : "r"(x));
    return d;
}

template <int B>
__device__ __forceinline__ void pack_block(const float2 (&f)[16], BlockWords<B> &c) {
    if constexpr (B == 3) {
        uint32_t x01, x23;
        pack_pair_q3(f, 0, c.w[0], x01);
        pack_pair_q3(f, 1, c.w[1], x23);
        c.w[2] = x01 | (x23 << 16);
    } else if constexpr (B == 4) {
#pragma unroll
        for (int s = 0; s < 4; ++s) c.w[s] = slot_nibbles(&f[4 * s]);
    } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t even, odd;
            slot_even_odd(f, s, even, odd);
            if constexpr (B == 8) {
                c.w[2 * s] = __byte_perm(even, odd, 0x5140);
                c.w[2 * s + 1] = __byte_perm(even, odd, 0x7362);
            } else {  // slot s's q2w field into the low (even s) or high half of its word
                // code bytes are 64 + code, 0..64 (quantize_block_magic): bit 7
                // is set only by 64 + 64, whose six code bits become all ones
                even |= sign_bytes(even);
                odd |= sign_bytes(odd);
                uint32_t y;
                q6_slot_fields(even, odd, c.w[s], y);
                c.w[4 + s / 2] = s % 2 == 0 ? __byte_perm(y, 0u, 0x4420) : __byte_perm(c.w[4 + s / 2], y, 0x6410);
            }
        }
    }
}

template <int B>
__device__ __forceinline__ SlotCodes slot_codes(const BlockWords<B> &c, int s) {
    SlotCodes sc;
    if constexpr (B == 8) {
        sc.a = c.w[2 * s];
        sc.b = c.w[2 * s + 1];
    } else if constexpr (B == 4) {
        sc.a = c.w[s];
        sc.b = 0;
    } else if constexpr (B == 3) {
        sc.a = (c.w[s / 2] >> (16 * (s % 2))) & 0xFFFFu;
        sc.b = (c.w[2] >> (8 * s)) & 0xFFu;
    } else {
        sc.a = c.w[s];
        sc.b = (c.w[4 + s / 2] >> (16 * (s % 2))) & 0xFFFFu;
    }
    return sc;
}

template <int B>
__device__ __forceinline__ void store_block_codes(uint8_t *tile, int g, const BlockWords<B> &c) {
    if constexpr (B == 8) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + 32 * g);
        p[0] = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
        p[1] = make_uint4(c.w[4], c.w[5], c.w[6], c.w[7]);
    } else if constexpr (B == 4) {
        *reinterpret_cast<uint4 *>(tile + 16 * g) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
    } else if constexpr (B == 3) {
        *reinterpret_cast<uint2 *>(tile + 8 * g) = make_uint2(c.w[0], c.w[1]);
        *reinterpret_cast<uint32_t *>(tile + 512 + 4 * g) = c.w[2];
    } else {
        *reinterpret_cast<uint4 *>(tile + 16 * g) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
        *reinterpret_cast<uint2 *>(tile + 1024 + 8 * g) = make_uint2(c.w[4], c.w[5]);
    }
}

template <int B>
__device__ __forceinline__ void load_block_codes(const uint8_t *tile, int g, BlockWords<B> &c) {
    if constexpr (B == 8) {
        const uint4 *p = reinterpret_cast<const uint4 *>(tile + 32 * g);
        const uint4 a = p[0], b = p[1];
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
        c.w[4] = b.x; c.w[5] = b.y; c.w[6] = b.z; c.w[7] = b.w;
    } else if constexpr (B == 4) {
        const uint4 a = *reinterpret_cast<const uint4 *>(tile + 16 * g);
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
    } else if constexpr (B == 3) {
        const uint2 a = *reinterpret_cast<const uint2 *>(tile + 8 * g);
        c.w[0] = a.x; c.w[1] = a.y;
        c.w[2] = *reinterpret_cast<const uint32_t *>(tile + 512 + 4 * g);
    } else {
        const uint4 a = *reinterpret_cast<const uint4 *>(tile + 16 * g);
        const uint2 b = *reinterpret_cast<const uint2 *>(tile + 1024 + 8 * g);
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
        c.w[4] = b.x; c.w[5] = b.y;
    }
}

// The 8 signed codes of a slot as exact floats, pairwise (lanes 2i, 2i+1):
// each code goes into the low byte of 1.5*2^23 + bias by one byte permute,
// and one packed add per pair removes the offset.
template <int B>
__device__ __forceinline__ void unpack_slot_q2(const SlotCodes c, float2 (&q)[4]) {
    uint32_t even, odd;
    slot_even_odd_codes<B>(c, even, odd);
    const float2 nm = make_float2(-Codec<B>::kMagic, -Codec<B>::kMagic);
    q[0] = __fadd2_rn(make_float2(byte_as_magic<0>(even), byte_as_magic<0>(odd)), nm);
    q[1] = __fadd2_rn(make_float2(byte_as_magic<1>(even), byte_as_magic<1>(odd)), nm);
    q[2] = __fadd2_rn(make_float2(byte_as_magic<2>(even), byte_as_magic<2>(odd)), nm);
    q[3] = __fadd2_rn(make_float2(byte_as_magic<3>(even), byte_as_magic<3>(odd)), nm);
}

// The 3-bit codes of two consecutive INT3 slots in nibbles, from the slots'
// q2w (W: slot 0 in bits 0..15) and q1w (X: slot 0 in bits 0..7, slot 1 in
// 8..15; bits above 15 are ignored): e nibble 4i+m = lane 2m of slot i, o
// nibble 4i+m = lane 2m+1, each nibble q2 | q1 << 2.  The q1 bits are placed
// by two byte-permute lookups: a selector nibble of three q1 bits (lanes j,
// j+1, j+2) picks the table byte that holds lane j's bit at bit 2 and lane
// j+2's at bit 6 -- 8 integer operations where spreading the q1 byte by
// shifts and masks took 11.
__device__ __forceinline__ void q3_nibbles(uint32_t W, uint32_t X, uint32_t &e, uint32_t &o) {
    constexpr uint32_t kQ1Lo = 0x04000400u, kQ1Hi = 0x44404440u;  // byte k = (k & 1) << 2 | (k & 4) << 4
    e = (W & 0x33333333u) | __byte_perm(kQ1Lo, kQ1Hi, X & 0x7777u);
    o = ((W >> 2) & 0x33333333u) | __byte_perm(kQ1Lo, kQ1Hi, (X >> 1) & 0x7777u);
}

// The 16 signed INT3 codes of two consecutive slots as exact floats,
// pairwise (q[4i + m] = lanes 2m, 2m+1 of slot i).  W: the two slots' q2w
// (slot 0 in bits 0..15); X: their q1w (slot 0 in bits 0..7, slot 1 in
// 8..15; bits above 15 are ignored).  The q1 bits are merged with the q2
// fields into 3-bit codes in nibbles, even lanes in one word and odd lanes
// in another (q3_nibbles); each code's byte then goes into a magic float by
// one byte permute (which can take any byte, so the codes need no further
// ordering).
__device__ __forceinline__ void unpack_pair_q3(uint32_t W, uint32_t X, float2 (&q)[8]) {
    uint32_t e, o;  // nibble 4i+m: lane 2m / 2m+1 of slot i
    q3_nibbles(W, X, e, o);
    const uint32_t el = e & 0x0F0F0F0Fu, eh = (e >> 4) & 0x0F0F0F0Fu;          // byte t: nibble 2t / 2t+1
    const uint32_t ol = o & 0x0F0F0F0Fu, oh = (o >> 4) & 0x0F0F0F0Fu;
    const float2 nm = make_float2(-Codec<3>::kMagic, -Codec<3>::kMagic);
    q[0] = __fadd2_rn(make_float2(byte_as_magic<0>(el), byte_as_magic<0>(ol)), nm);  // slot 0 lanes 0, 1
    q[1] = __fadd2_rn(make_float2(byte_as_magic<0>(eh), byte_as_magic<0>(oh)), nm);  // lanes 2, 3
    q[2] = __fadd2_rn(make_float2(byte_as_magic<1>(el), byte_as_magic<1>(ol)), nm);  // lanes 4, 5
    q[3] = __fadd2_rn(make_float2(byte_as_magic<1>(eh), byte_as_magic<1>(oh)), nm);  // lanes 6, 7
    q[4] = __fadd2_rn(make_float2(byte_as_magic<2>(el), byte_as_magic<2>(ol)), nm);  // slot 1
    q[5] = __fadd2_rn(make_float2(byte_as_magic<2>(eh), byte_as_magic<2>(oh)), nm);
    q[6] = __fadd2_rn(make_float2(byte_as_magic<3>(el), byte_as_magic<3>(ol)), nm);
    q[7] = __fadd2_rn(make_float2(byte_as_magic<3>(eh), byte_as_magic<3>(oh)), nm);
}

// Four bytes of E2M1 code pairs (low nibble, high nibble) as four fp16 pairs
// (low half, high half), exactly, by the native conversion.
__device__ __forceinline__ void e2m1_pairs_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// acc += (q.lo * s, q.hi * s) for an fp16 pair q and an fp16 scale s, each
// product exact and each sum rounded once to fp32: the same result as an
// fp32 fma of the widened operands.
__device__ __forceinline__ void fma_f16x2_f16_f32(uint32_t q, unsigned short s, float2 &acc) {
    asm("{ .reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.f16 %0, lo, %3, %0;\n\t"
        "fma.rn.f32.f16 %1, hi, %3, %1; }"
        : "+f"(acc.x), "+f"(acc.y)
        : "r"(q), "h"(s));
}

// The 8 signed INT4 codes of a slot word (lane j in bits 4j) as exact fp16
// pairs q[m] = (lane m, lane m + 4): each code goes into the mantissa of the
// fp16 1024 in place (one logic operation per pair: lanes m and m + 4 sit 16
// bits apart), and one packed fp16 fma per pair removes the offset and the
// bias, scaling the nibbles at bits 4..7 of each half back by 1/16 --
// (1024 + u) - 1032 or (1024 + 16u) / 16 - 72, exact at every step.
__device__ __forceinline__ void unpack_word_q4_f16(uint32_t w, uint32_t (&q)[4]) {
    const uint32_t w8 = w >> 8;
    const uint32_t a = (w & 0x000F000Fu) | 0x64006400u, b = (w & 0x00F000F0u) | 0x64006400u;
    const uint32_t c = (w8 & 0x000F000Fu) | 0x64006400u, d = (w8 & 0x00F000F0u) | 0x64006400u;
    const __half2 one = __float2half2_rn(1.0f), sixteenth = __float2half2_rn(0.0625f);
    const __half2 off0 = __float2half2_rn(-1032.0f), off4 = __float2half2_rn(-72.0f);
    const auto h2 = [](uint32_t v) { return *reinterpret_cast<const __half2 *>(&v); };
    const auto u32 = [](__half2 v) { return *reinterpret_cast<const uint32_t *>(&v); };
    q[0] = u32(__hfma2(h2(a), one, off0));        // lanes 0, 4
    q[1] = u32(__hfma2(h2(b), sixteenth, off4));  // lanes 1, 5
    q[2] = u32(__hfma2(h2(c), one, off0));        // lanes 2, 6
    q[3] = u32(__hfma2(h2(d), sixteenth, off4));  // lanes 3, 7
}

// The codes of slot s from magic floats paired as (lane m, lane m + 4)
// (f[m] for m = 0..3), lane j in bits 4j (each code below 16).
__device__ __forceinline__ uint32_t slot_nibbles_m4(const float2 *f) {
    return __byte_perm(nibbles4_lo16(f[0].x, f[1].x, f[2].x, f[3].x),
                       nibbles4_lo16(f[0].y, f[1].y, f[2].y, f[3].y), 0x5410);
}

// The 16 signed INT3 codes of two consecutive slots (W, X as for
// unpack_pair_q3) as exact fp16 pairs, h[4i + m] = lanes 2m, 2m+1 of slot
// i.  Every INT3 value -4..3 is an E2M1 value, so after the q1 bits are
// merged into 3-bit codes in nibbles (even lanes in e, odd lanes in o), one
// byte permute per four codes looks each code's E2M1 code up in an 8-entry
// byte table (the low-nibble table for the even lanes, the same codes shifted
// into the high nibble for the odd lanes), an OR pairs them, and the native
// E2M1 conversion yields two fp16 values per byte.  8 integer operations
// per 8 values where the float path takes 14.
__device__ __forceinline__ void unpack_pair_q3_f16(uint32_t W, uint32_t X, uint32_t (&h)[8]) {
    // E2M1 codes of u - 4 for u = 0..7: -4, -3, -2, -1, 0, 1, 2, 3
    constexpr uint32_t kLo0 = 0x0A0C0D0Eu, kLo1 = 0x05040200u;  // bytes 0-3, 4-7
    constexpr uint32_t kHi0 = 0xA0C0D0E0u, kHi1 = 0x50402000u;
    uint32_t e, o;  // nibble 4i+m: lane 2m / 2m+1 of slot i
    q3_nibbles(W, X, e, o);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t ei = e >> (16 * i), oi = o >> (16 * i);  // the byte permute reads 4 selector nibbles
        const uint32_t pairs = __byte_perm(kLo0, kLo1, ei) | __byte_perm(kHi0, kHi1, oi);
        uint32_t hi[4];
        e2m1_pairs_to_f16x2(pairs, hi);
#pragma unroll
        for (int m = 0; m < 4; ++m) h[4 * i + m] = hi[m];
    }
}

// The 16 signed INT3 codes of two consecutive slots (W, X as for
// unpack_pair_q3) as exact fp16 pairs by lane, h[L] = (lane L of slot 0,
// lane L of slot 1): after the q1 bits are merged into nibbles (q3_nibbles),
// one logic operation puts two codes 16 bits apart into the mantissas of the
// fp16 pair (1024, 1024) and one packed fp16 fma removes the offset and the
// bias (and the factor 16 of a code in bits 4..7): exact at every step.
__device__ __forceinline__ void unpack_pair_q3_f16_lanes(uint32_t W, uint32_t X, uint32_t (&h)[8]) {
    uint32_t e, o;
    q3_nibbles(W, X, e, o);
    const __half2 one = __float2half2_rn(1.0f), sixteenth = __float2half2_rn(0.0625f);
    const __half2 off0 = __float2half2_rn(-1028.0f), off4 = __float2half2_rn(-68.0f);
    const auto fix = [](uint32_t t, __half2 m, __half2 a) {
        const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&t), m, a);
        return *reinterpret_cast<const uint32_t *>(&r);
    };
    const uint32_t e8 = e >> 8, o8 = o >> 8;
    h[0] = fix((e & 0x000F000Fu) | 0x64006400u, one, off0);         // lane 0: nibbles 0 and 4 of e
    h[2] = fix((e & 0x00F000F0u) | 0x64006400u, sixteenth, off4);   // lane 2: nibbles 1 and 5
    h[4] = fix((e8 & 0x000F000Fu) | 0x64006400u, one, off0);        // lane 4: nibbles 2 and 6
    h[6] = fix((e8 & 0x00F000F0u) | 0x64006400u, sixteenth, off4);  // lane 6: nibbles 3 and 7
    h[1] = fix((o & 0x000F000Fu) | 0x64006400u, one, off0);
    h[3] = fix((o & 0x00F000F0u) | 0x64006400u, sixteenth, off4);
    h[5] = fix((o8 & 0x000F000Fu) | 0x64006400u, one, off0);
    h[7] = fix((o8 & 0x00F000F0u) | 0x64006400u, sixteenth, off4);
}

// The 8 signed INT6 codes of a slot as exact fp16 pairs h[0..3] = lanes
// (0, 2), (4, 6), (1, 3), (5, 7): the 6-bit codes, one per byte (even and
// odd lanes apart), become the low bytes of two fp16 patterns 0x64xx
// (1024 + code) by one byte permute, and one packed fp16 fma per pair removes
// the offset and the bias -- half the byte permutes of the float path.
__device__ __forceinline__ void unpack_slot_q6_f16(const SlotCodes c, uint32_t (&h)[4]) {
    uint32_t even, odd;
    slot_even_odd_codes<6>(c, even, odd);
    const __half2 one = __float2half2_rn(1.0f), off = __float2half2_rn(-1056.0f);
    const auto fix = [&](uint32_t t) {
        const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&t), one, off);
        return *reinterpret_cast<const uint32_t *>(&r);
    };
    h[0] = fix(__byte_perm(even, 0x64646464u, 0x4140));
    h[1] = fix(__byte_perm(even, 0x64646464u, 0x4342));
    h[2] = fix(__byte_perm(odd, 0x64646464u, 0x4140));
    h[3] = fix(__byte_perm(odd, 0x64646464u, 0x4342));
}

// The 32 signed codes of a block as exact floats, pairwise.
template <int B>
__device__ __forceinline__ void unpack_block_q(const BlockWords<B> &c, float2 (&q)[16]) {
    if constexpr (B == 3) {
        float2 lo[8], hi[8];
        unpack_pair_q3(c.w[0], c.w[2], lo);        // slots 0, 1
        unpack_pair_q3(c.w[1], c.w[2] >> 16, hi);  // slots 2, 3
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[i] = lo[i];
            q[8 + i] = hi[i];
        }
    } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            float2 qs[4];
            unpack_slot_q2<B>(slot_codes<B>(c, s), qs);
#pragma unroll
            for (int i = 0; i < 4; ++i) q[4 * s + i] = qs[i];
        }
    }
}

template <int B>
__device__ __forceinline__ uint32_t load_block_scale_bits(const uint8_t *tile, int g) {
    return ld_u16(tile + Codec<B>::kCodeBytes + 2 * g);
}

template <int B>
__device__ __forceinline__ void store_block_scale(uint8_t *tile, int g, uint32_t bits) {
    *reinterpret_cast<uint16_t *>(tile + Codec<B>::kCodeBytes + 2 * g) = static_cast<uint16_t>(bits);
}

__device__ __forceinline__ float f16_bits_to_float(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// ---------------------------------------------------------------------------
// kernels.  NB = number of blocks = 64 * tiles (the zero padding of the last
// tile included); thread (CTA c, lane i) starts at block c*256 + i.
// ---------------------------------------------------------------------------

// Where tile t of a wire goes: contiguously (a plain wire) ...
struct ContigTiles {
    uint8_t *base;
    int tile_bytes;
    __device__ __forceinline__ uint8_t *operator()(long long t) const { return base + t * tile_bytes; }
};

// ... or into owner k's receive buffer for sender j (the two-shot exchange
// on one GPU): owner k = t / seg owns tiles [k*seg, (k+1)*seg); the R
// buffers of owner k sit back to back, each `seg` tiles long.
struct OwnerTiles {
    uint8_t *ws;
    long long seg;
    int ranks, sender, tile_bytes;
    __device__ __forceinline__ uint8_t *operator()(long long t) const {
        const long long k = t / seg;
        return ws + ((k * ranks + sender) * seg + (t - k * seg)) * tile_bytes;
    }
};

// Send path [QR Quantization and Dequantization Paths, CodecQ3::send].
// The body of each kernel below is a device function so that the two-shot
// path can run it once per rank (blockIdx.y) inside a single launch.
template <int B, int DT, int U, class Addr>
__device__ __forceinline__ void encode32_run(const uint16_t *__restrict__ x, long long n, Addr wire, long long NB) {
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb0 = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb0 < NB; gb0 += U * S) {
        uint32_t raw[U][16];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB) load_block_values(x, gb * 32, n, raw[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB) {
                float2 v[16], f[16];
                widen_block<DT>(raw[u], v);
                const BlockScale2 sc = block_scale2<B>(block_absmax(v));
                quantize_block_magic<B>(v, sc.r, sc.low_clip, f);
                BlockWords<B> c;
                pack_block<B>(f, c);
                uint8_t *tile = wire(gb >> 6);
                store_block_codes<B>(tile, static_cast<int>(gb & 63), c);
                store_block_scale<B>(tile, static_cast<int>(gb & 63), sc.bits);
            }
        }
    }
}

template <int B, int DT, int U, class Addr = ContigTiles>
__global__ void __launch_bounds__(kThreads32) encode32_kernel(const uint16_t *__restrict__ x, long long n,
                                                              Addr wire, long long NB) {
    chain_entry();
    encode32_run<B, DT, U, Addr>(x, n, wire, NB);
}

// Receive path / Phase-2 [QR Quantization and Dequantization Paths,
// CodecQ3::recv], with two threads per block (16 values, two slots each):
// every lane writes 32 contiguous bytes of output and neighbouring lanes
// write neighbouring bytes, so a warp's stores cover whole sectors once.
// Work unit = half-block hb: block hb/2, slots 2*(hb%2) and 2*(hb%2)+1.
template <int B>
struct HalfWords {  // the codes of two slots
    static constexpr int kWords = (B == 8) ? 4 : (B == 4) ? 2 : (B == 3) ? 2 : 3;
    uint32_t w[kWords];
};

template <int B>
__device__ __forceinline__ void load_half_codes(const uint8_t *tile, int g, int half, HalfWords<B> &c) {
    if constexpr (B == 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(tile + 32 * g + 16 * half);
        c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
    } else if constexpr (B == 4) {
        const uint2 a = *reinterpret_cast<const uint2 *>(tile + 16 * g + 8 * half);
        c.w[0] = a.x; c.w[1] = a.y;
    } else if constexpr (B == 3) {
        c.w[0] = *reinterpret_cast<const uint32_t *>(tile + 8 * g + 4 * half);       // two q2w
        c.w[1] = *reinterpret_cast<const uint16_t *>(tile + 512 + 4 * g + 2 * half); // two q1w
    } else {
        const uint2 a = *reinterpret_cast<const uint2 *>(tile + 16 * g + 8 * half);
        c.w[0] = a.x; c.w[1] = a.y;
        c.w[2] = *reinterpret_cast<const uint32_t *>(tile + 1024 + 8 * g + 4 * half);  // two q2w
    }
}

template <int B>
__device__ __forceinline__ SlotCodes half_slot_codes(const HalfWords<B> &c, int s) {
    SlotCodes sc;
    if constexpr (B == 8) {
        sc.a = c.w[2 * s];
        sc.b = c.w[2 * s + 1];
    } else if constexpr (B == 4) {
        sc.a = c.w[s];
        sc.b = 0;
    } else if constexpr (B == 3) {
        sc.a = (c.w[0] >> (16 * s)) & 0xFFFFu;
        sc.b = (c.w[1] >> (8 * s)) & 0xFFu;
    } else {
        sc.a = c.w[s];
        sc.b = (c.w[2] >> (16 * s)) & 0xFFFFu;
    }
    return sc;
}

template <int B, int DT, int U, bool Y32>  // Y32: y is 32-byte aligned (one 256-bit store per unit)
__device__ __forceinline__ void decode16_run(const uint8_t *__restrict__ wire, long long n, uint16_t *__restrict__ y,
                                             long long NH) {
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long hb0 = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; hb0 < NH; hb0 += U * S) {
        HalfWords<B> c[U];
        uint32_t sb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long hb = hb0 + u * S;
            if (hb < NH) {
                const long long gb = hb >> 1;
                const uint8_t *tile = wire + (gb >> 6) * Codec<B>::kTileBytes;
                load_half_codes<B>(tile, static_cast<int>(gb & 63), static_cast<int>(hb & 1), c[u]);
                sb[u] = load_block_scale_bits<B>(tile, static_cast<int>(gb & 63));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long hb = hb0 + u * S;
            if (hb < NH) {
                const float s = f16_bits_to_float(sb[u]);
                const float2 s2 = make_float2(s, s);
                float2 o[8];
                if constexpr (B == 3) {
                    float2 q[8];
                    unpack_pair_q3(c[u].w[0], c[u].w[1], q);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = __fmul2_rn(q[i], s2);
                } else {
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        float2 q[4];
                        unpack_slot_q2<B>(half_slot_codes<B>(c[u], sl), q);
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[4 * sl + i] = __fmul2_rn(q[i], s2);
                    }
                }
                const long long base = hb * 16;
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = narrow2<DT>(o[i].x, o[i].y);
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
    }
}

template <int B, int DT, int U, bool Y32>
__global__ void __launch_bounds__(kThreads32) decode16_kernel(const uint8_t *__restrict__ wire, long long n,
                                                              uint16_t *__restrict__ y, long long NH) {
    chain_entry();
    decode16_run<B, DT, U, Y32>(wire, n, y, NH);
}

// Codes of two slots (one half-block) from 16 magic floats f[0..7] (pairs):
// the asymmetric codec's INT4 and INT8 halves.
template <int B>
__device__ __forceinline__ void pack_half(const float2 (&f)[8], HalfWords<B> &c) {
    static_assert(B == 4 || B == 8, "half-block packing is used at INT4 and INT8");
    if constexpr (B == 4) {
        c.w[0] = slot_nibbles(&f[0]);
        c.w[1] = slot_nibbles(&f[4]);
    } else {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const uint32_t even = gather_low_bytes(__float_as_uint(f[4 * s].x), __float_as_uint(f[4 * s + 1].x),
                                                   __float_as_uint(f[4 * s + 2].x), __float_as_uint(f[4 * s + 3].x));
            const uint32_t odd = gather_low_bytes(__float_as_uint(f[4 * s].y), __float_as_uint(f[4 * s + 1].y),
                                                  __float_as_uint(f[4 * s + 2].y), __float_as_uint(f[4 * s + 3].y));
            c.w[2 * s] = __byte_perm(even, odd, 0x5140);
            c.w[2 * s + 1] = __byte_perm(even, odd, 0x7362);
        }
    }
}

template <int B>
__device__ __forceinline__ void store_half_codes(uint8_t *tile, int g, int half, const HalfWords<B> &c) {
    if constexpr (B == 8) {
        *reinterpret_cast<uint4 *>(tile + 32 * g + 16 * half) = make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]);
    } else if constexpr (B == 4) {
        *reinterpret_cast<uint2 *>(tile + 16 * g + 8 * half) = make_uint2(c.w[0], c.w[1]);
    } else if constexpr (B == 3) {
        *reinterpret_cast<uint32_t *>(tile + 8 * g + 4 * half) = c.w[0];
        *reinterpret_cast<uint16_t *>(tile + 512 + 4 * g + 2 * half) = static_cast<uint16_t>(c.w[1]);
    } else {
        *reinterpret_cast<uint2 *>(tile + 16 * g + 8 * half) = make_uint2(c.w[0], c.w[1]);
        *reinterpret_cast<uint32_t *>(tile + 1024 + 8 * g + 4 * half) = c.w[2];
    }
}

// ---------------------------------------------------------------------------
// Phase-1B by exact integer arithmetic
// ---------------------------------------------------------------------------
// Every decoded value q*s is exact in fp32 (a code of at most 6 bits times an
// fp16 scale), and every fp16 scale s_r >= smin is an integer multiple M_r of
// unit = 2^(floor(log2 smin) - 10), smin the block's smallest nonzero scale
// over the R ranks.  When M_r < 2^16 for every rank (the scales lie within
// about 5 binades of each other), every partial sum of the rank order is an
// integer multiple of unit below bias * R * 2^16 <= 2^24 units in magnitude,
// so the fp32 rank-order sum that defines Phase-1B rounds nothing: it equals
// the exact sum unit * S, S = sum_r M_r * q_r, in any order.  S is then summed in
// integers: the codes of two ranks for one value sit in adjacent bytes (one
// byte permute per four values), and one two-way dot product (dp2a: two
// 16x8-bit products and an add) takes both ranks' M_r * u_r.  u = q + bias is
// the stored code.  The accumulator starts at 1.5*2^23 - bias * sum_r M_r as
// an fp32 bit pattern, so it ends as the pattern of the float 1.5*2^23 + S,
// and one fma per value pair turns it into unit * S.  That needs |S| below
// 2^22, which holds at INT3 and INT4 (|S| <= 8 * 8 * 2^16).  INT6 with at
// most four ranks adds it to the condition: bias * sum_r M_r < 2^22, i.e.
// sum_r M_r < 2^17 (always true at R = 2; an INT6 block further spread takes
// the float path).  INT6 from five ranks, where outlier channels put many
// blocks past that sum, starts at -bias * sum_r M_r instead and ends as S
// (|S| < 2^24), converted exactly to fp32 and scaled by unit.  The result is the
// rank-order sum up to the sign of a zero, which the re-quantization does not
// see (a zero gives the same code with either sign).  Blocks outside the
// condition (scales further apart, a negative, infinite or NaN scale bit
// pattern, every scale zero) return false and take the float path.
constexpr uint32_t kExactLimit = 1u << 16;     // M_r < kExactLimit
constexpr uint32_t kExactSumLimit6 = 1u << 17;  // INT6, R <= 4: sum_r M_r < kExactSumLimit6

// The codes of one rank's block as 8 words of 4 byte-sized codes: word x,
// byte t is the code of value 2 * exact_pair<B>(x, t) + (x >= 4 at INT3,
// else x & 1).
// The 8 INT6 codes of a slot as bytes, lanes 0,2,4,6 in `even` and 1,3,5,7
// in `odd`, from the slot's low nibbles `a` (lane j at bits 4j) and its
// high-bit pairs in the low 16 bits of `b` (lane j at bits 2j): one byte
// permute looks each lane's two high bits up in a table of the four values
// already shifted to bits 4..5, with the lane's bits in the low bits of a
// selector nibble (the nibble's top bit is cleared: set, it would make the
// permute replicate a sign).  8 integer operations per slot where spreading
// the high bits by shifts and masks took 11.
__device__ __forceinline__ void q6_even_odd_bytes(uint32_t a, uint32_t b, uint32_t &even, uint32_t &odd) {
    constexpr uint32_t kHi = 0x30201000u;  // byte i = i << 4
    even = (a & 0x0F0F0F0Fu) | __byte_perm(kHi, kHi, b & 0x7777u);
    odd = ((a >> 4) & 0x0F0F0F0Fu) | __byte_perm(kHi, kHi, (b >> 2) & 0x7777u);
}

template <int B>
__device__ __forceinline__ void block_code_bytes(const BlockWords<B> &c, uint32_t (&X)[8]) {
    if constexpr (B == 6) {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
            q6_even_odd_bytes(c.w[sl], c.w[4 + sl / 2] >> (16 * (sl % 2)), X[2 * sl], X[2 * sl + 1]);
    } else if constexpr (B == 3) {
        uint32_t e01, o01, e23, o23;  // nibble 4i+m: lane 2m (e) / 2m+1 (o) of slot i (+2)
        q3_nibbles(c.w[0], c.w[2], e01, o01);
        q3_nibbles(c.w[1], c.w[2] >> 16, e23, o23);
        X[0] = e01 & 0x0F0F0F0Fu;
        X[1] = (e01 >> 4) & 0x0F0F0F0Fu;
        X[2] = e23 & 0x0F0F0F0Fu;
        X[3] = (e23 >> 4) & 0x0F0F0F0Fu;
        X[4] = o01 & 0x0F0F0F0Fu;
        X[5] = (o01 >> 4) & 0x0F0F0F0Fu;
        X[6] = o23 & 0x0F0F0F0Fu;
        X[7] = (o23 >> 4) & 0x0F0F0F0Fu;
    } else {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) slot_even_odd_codes<B>(slot_codes<B>(c, sl), X[2 * sl], X[2 * sl + 1]);
    }
}

// The value pair (index j: values 2j, 2j+1 of the block) of byte t of code
// word x, and whether the byte holds the pair's odd value.
template <int B>
__device__ __forceinline__ constexpr int exact_pair(int x, int t) {
    return B == 3 ? ((x & 1) + 8 * ((x >> 1) & 1) + 2 * t) : (4 * (x >> 1) + t);
}
template <int B>
__device__ __forceinline__ constexpr bool exact_odd(int x) {
    return B == 3 ? x >= 4 : (x & 1) != 0;
}

template <int B, int R>
__device__ __forceinline__ bool exact_int_sum(const BlockWords<B> (&c)[R], const uint32_t (&sb)[R],
                                              float2 (&acc)[16]) {
    // the largest scale pattern (unsigned: a sign bit, infinity and NaN all
    // compare above 0x7BFF) and the smallest nonzero one
    uint32_t hi = 0, lo_m1 = 0xFFFFFFFFu;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        hi = max(hi, sb[r]);
        lo_m1 = min(lo_m1, sb[r] - 1u);
    }
    if (hi > 0x7BFFu || lo_m1 == 0xFFFFFFFFu) return false;
    const uint32_t unit_bits = (__float_as_uint(f16_bits_to_float(lo_m1 + 1u)) & 0x7F800000u) - (10u << 23);
    const float unit = __uint_as_float(unit_bits), inv = __uint_as_float(0x7F000000u - unit_bits);  // 2^k, 2^-k
    if (!(__fmul_rn(f16_bits_to_float(hi), inv) < float(kExactLimit))) return false;
    // M_r in the low half of the pattern of 2^23 + M_r; the sum of the
    // scales (exact: multiples of unit below 2^19 units)
    uint32_t m[R];
    float ssum = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float s = f16_bits_to_float(sb[r]);
        m[r] = __float_as_uint(__fmaf_rn(s, inv, 8388608.0f));
        ssum = __fadd_rn(ssum, s);
    }
    constexpr bool kMagic = B != 6 || R <= 4;  // the accumulator as the pattern of 1.5*2^23 + S
    if constexpr (B == 6 && R > 2 && kMagic)
        if (!(__fmul_rn(ssum, inv) < float(kExactSumLimit6))) return false;
    uint32_t base;
    if constexpr (kMagic)  // the pattern of 1.5*2^23 - bias * sum M (exact: bias * sum M < 2^22)
        base = __float_as_uint(__fmaf_rn(ssum, -float(Codec<B>::kBias) * inv, kRoundMagic));
    else  // -bias * sum M (sum M < 2^19, from the pattern of 2^23 + sum M)
        base = (0x4B000000u - __float_as_uint(__fmaf_rn(ssum, inv, 8388608.0f))) * uint32_t(Codec<B>::kBias);
    uint32_t ax[16], ay[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) ax[j] = ay[j] = base;
#pragma unroll
    for (int r = 0; r + 1 < R; r += 2) {
        const uint32_t a = __byte_perm(m[r], m[r + 1], 0x5410);  // (M_r, M_r+1) as 16-bit halves
        uint32_t X0[8], X1[8];
        block_code_bytes<B>(c[r], X0);
        block_code_bytes<B>(c[r + 1], X1);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const uint32_t p01 = __byte_perm(X0[x], X1[x], 0x5140), p23 = __byte_perm(X0[x], X1[x], 0x7362);
            uint32_t *d = exact_odd<B>(x) ? ay : ax;
            d[exact_pair<B>(x, 0)] = __dp2a_lo(a, p01, d[exact_pair<B>(x, 0)]);
            d[exact_pair<B>(x, 1)] = __dp2a_hi(a, p01, d[exact_pair<B>(x, 1)]);
            d[exact_pair<B>(x, 2)] = __dp2a_lo(a, p23, d[exact_pair<B>(x, 2)]);
            d[exact_pair<B>(x, 3)] = __dp2a_hi(a, p23, d[exact_pair<B>(x, 3)]);
        }
    }
    if constexpr (R % 2 == 1) {  // the last rank alone: (M, 0) against bytes 0, 2 and 1, 3
        const uint32_t a = m[R - 1] & 0xFFFFu;
        uint32_t X0[8];
        block_code_bytes<B>(c[R - 1], X0);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            uint32_t *d = exact_odd<B>(x) ? ay : ax;
            d[exact_pair<B>(x, 0)] = __dp2a_lo(a, X0[x], d[exact_pair<B>(x, 0)]);
            d[exact_pair<B>(x, 2)] = __dp2a_hi(a, X0[x], d[exact_pair<B>(x, 2)]);
            d[exact_pair<B>(x, 1)] = __dp2a_lo(a, X0[x] >> 8, d[exact_pair<B>(x, 1)]);
            d[exact_pair<B>(x, 3)] = __dp2a_hi(a, X0[x] >> 8, d[exact_pair<B>(x, 3)]);
        }
    }
    const float2 u2 = make_float2(unit, unit);
    if constexpr (kMagic) {
        const float2 c2 = make_float2(-kRoundMagic * unit, -kRoundMagic * unit);  // exact: a power of two
#pragma unroll
        for (int j = 0; j < 16; ++j)
            acc[j] = __ffma2_rn(make_float2(__uint_as_float(ax[j]), __uint_as_float(ay[j])), u2, c2);
    } else {  // S exactly (|S| < 2^24), times unit (a power of two: exact)
#pragma unroll
        for (int j = 0; j < 16; ++j)
            acc[j] = __fmul2_rn(make_float2(__int2float_rn(static_cast<int>(ax[j])),
                                            __int2float_rn(static_cast<int>(ay[j]))), u2);
    }
    return true;
}

// Where Phase-1B takes the exact integer sum first (the float path below
// remains the fallback for blocks outside its condition).
template <int B, int R>
__host__ __device__ constexpr bool exact_sum_enabled() {
    return (B == 3 || B == 4 || B == 6) && R >= 2;
}

// Phase-1B of one 32-value block from its R ranks' codes c[r] and fp16 scale
// bits sb[r] (one thread per block): decode, add in fp32 in rank order
// (fma(q, s, acc) = RN(acc + q*s): q*s is exact), re-quantize; the block's
// codes go to cw and its fp16 scale bits to scale_bits.  The float path.
template <int B, int R>
__device__ __forceinline__ void reduce_block_words_float(const BlockWords<B> (&c)[R], const uint32_t (&sb)[R],
                                                         BlockWords<B> &cw, uint32_t &scale_bits) {
    float2 acc[16];
    if constexpr (B == 3 && R <= 4) {
        // codes decoded to fp16 through the fp16 1024 (logic operations and
        // packed fp16 fmas), paired by lane across two slots (A[h][L] = lane L
        // of slots 2h and 2h+1), scaled and summed by fp16-operand fmas into
        // fp32; acc starts at -0, so the first fma returns the first rank's
        // product exactly.  Measured against the E2M1 decode below at 2^27
        // values per rank: 6% faster at R = 2, 1% at R = 4, 9% slower at R = 8.
        float2 A[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int L = 0; L < 8; ++L) A[h][L] = make_float2(-0.0f, -0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned short sh = static_cast<unsigned short>(sb[r]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t hp[8];
                unpack_pair_q3_f16_lanes(c[r].w[h], h ? (c[r].w[2] >> 16) : c[r].w[2], hp);
#pragma unroll
                for (int L = 0; L < 8; ++L) fma_f16x2_f16_f32(hp[L], sh, A[h][L]);
            }
        }
        const BlockScale2 sc = block_scale2<B>(absmax_n<32>(reinterpret_cast<const float *>(A)));
        float2 F[2][8];
        quantize_block_magic<B>(reinterpret_cast<const float2(&)[16]>(A), sc.r, sc.low_clip,
                                reinterpret_cast<float2(&)[16]>(F));
        uint32_t x01, x23;
        pack_pair_q3_lanes(F[0], cw.w[0], x01);
        pack_pair_q3_lanes(F[1], cw.w[1], x23);
        cw.w[2] = x01 | (x23 << 16);
        scale_bits = sc.bits;
        return;
    } else if constexpr (B == 3) {
        // codes decoded to fp16 through E2M1, scaled and summed by fp16-operand
        // fmas into fp32 (acc starts at -0, so the first fma returns the first
        // rank's product exactly, signed zeros included).  (R <= 4 takes the
        // fp16-1024 decode above.)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = make_float2(-0.0f, -0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint32_t h[16];
            uint32_t lo[8], hi[8];
            unpack_pair_q3_f16(c[r].w[0], c[r].w[2], lo);        // slots 0, 1
            unpack_pair_q3_f16(c[r].w[1], c[r].w[2] >> 16, hi);  // slots 2, 3
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = lo[i];
                h[8 + i] = hi[i];
            }
            const unsigned short sh = static_cast<unsigned short>(sb[r]);
#pragma unroll
            for (int i = 0; i < 16; ++i) fma_f16x2_f16_f32(h[i], sh, acc[i]);
        }
    } else if constexpr (B == 4 && R >= 4) {
        // codes decoded to fp16 in place, summed by fp16-operand fmas; here
        // acc[4s + m] holds lanes m and m + 4 of slot s (as the decode gives them).
        // Measured against the float path at 2^27 / 2^28 values per rank: R = 8
        // 0.70 / 0.71 -> 0.75 / 0.77 of HBM, R = 4 0.63 / 0.66 -> 0.65 / 0.68,
        // R = 2 0.55 / 0.58 -> 0.54 / 0.56 (so R <= 3 keeps the float path).
        // acc starts at -0: the first fma returns the first rank's product.
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = make_float2(-0.0f, -0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned short sh = static_cast<unsigned short>(sb[r]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t q[4];
                unpack_word_q4_f16(c[r].w[k], q);
#pragma unroll
                for (int m = 0; m < 4; ++m) fma_f16x2_f16_f32(q[m], sh, acc[4 * k + m]);
            }
        }
    } else if constexpr (B == 6) {
        // codes decoded to fp16 by byte permutes, summed by fp16-operand fmas;
        // here acc[4s + i] holds lanes (0, 2), (4, 6), (1, 3), (5, 7) of slot s.
        // Measured against the float path at 2^27 / 2^28 bf16 values per rank:
        // R = 8 0.76 / 0.78 -> 0.82 / 0.84 of HBM, R = 2 0.57 / 0.60 -> 0.60 /
        // 0.62, R = 4 equal (0.67 / 0.69).  acc starts at -0 as above.
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = make_float2(-0.0f, -0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned short sh = static_cast<unsigned short>(sb[r]);
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                uint32_t h[4];
                unpack_slot_q6_f16(slot_codes<6>(c[r], sl), h);
#pragma unroll
                for (int i = 0; i < 4; ++i) fma_f16x2_f16_f32(h[i], sh, acc[4 * sl + i]);
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float s = f16_bits_to_float(sb[r]);
            const float2 s2 = make_float2(s, s);
            float2 q[16];
            unpack_block_q<B>(c[r], q);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = (r == 0) ? __fmul2_rn(q[i], s2) : __ffma2_rn(q[i], s2, acc[i]);
        }
    }
    const BlockScale2 sc = block_scale2<B>(block_absmax(acc));
    float2 f[16];
    quantize_block_magic<B>(acc, sc.r, sc.low_clip, f);
    if constexpr (B == 4 && R >= 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cw.w[k] = slot_nibbles_m4(&f[4 * k]);
    } else if constexpr (B == 6) {
        float2 fs[16];
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const float2 *g = &f[4 * sl];
            fs[4 * sl] = make_float2(g[0].x, g[2].x);      // lanes 0, 1
            fs[4 * sl + 1] = make_float2(g[0].y, g[2].y);  // lanes 2, 3
            fs[4 * sl + 2] = make_float2(g[1].x, g[3].x);  // lanes 4, 5
            fs[4 * sl + 3] = make_float2(g[1].y, g[3].y);  // lanes 6, 7
        }
        pack_block<B>(fs, cw);
    } else {
        pack_block<B>(f, cw);
    }
    scale_bits = sc.bits;
}

// Phase-1B of one block (as reduce_block_words_float): the exact integer sum
// where it applies, the float path otherwise; the same bytes either way.
template <int B, int R>
__device__ __forceinline__ void reduce_block_words(const BlockWords<B> (&c)[R], const uint32_t (&sb)[R],
                                                   BlockWords<B> &cw, uint32_t &scale_bits) {
    if constexpr (exact_sum_enabled<B, R>()) {
        float2 acc[16];
        if (exact_int_sum<B, R>(c, sb, acc)) {
            const BlockScale2 sc = block_scale2<B>(block_absmax(acc));
            float2 f[16];
            quantize_block_magic<B>(acc, sc.r, sc.low_clip, f);
            pack_block<B>(f, cw);
            scale_bits = sc.bits;
            return;
        }
    }
    reduce_block_words_float<B, R>(c, sb, cw, scale_bits);
}

// reduce_block_words, written into `tile` as its block g; kFloatOnly skips
// the exact integer sum (the same bytes, for a kernel that has no registers
// to spare for it).
template <int B, int R, bool kFloatOnly = false>
__device__ __forceinline__ void reduce_block(const BlockWords<B> (&c)[R], const uint32_t (&sb)[R], uint8_t *tile,
                                             int g) {
    BlockWords<B> cw;
    uint32_t bits;
    if constexpr (kFloatOnly)
        reduce_block_words_float<B, R>(c, sb, cw, bits);
    else
        reduce_block_words<B, R>(c, sb, cw, bits);
    store_block_codes<B>(tile, g, cw);
    store_block_scale<B>(tile, g, bits);
}

template <int B, int R, int U>
__device__ __forceinline__ void reduce32_run(ConstPtrs wires, uint8_t *out, long long NB) {
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    for (long long gb0 = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x; gb0 < NB; gb0 += U * S) {
        BlockWords<B> c[U][R];
        uint32_t sb[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB) {
                const long long off = (gb >> 6) * Codec<B>::kTileBytes;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint8_t *tile = static_cast<const uint8_t *>(wires.p[r]) + off;
                    load_block_codes<B>(tile, static_cast<int>(gb & 63), c[u][r]);
                    sb[u][r] = load_block_scale_bits<B>(tile, static_cast<int>(gb & 63));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long gb = gb0 + u * S;
            if (gb < NB)
                reduce_block<B, R>(c[u], sb[u], out + (gb >> 6) * Codec<B>::kTileBytes, static_cast<int>(gb & 63));
        }
    }
}

template <int B, int R, int U>
__global__ void __launch_bounds__(kThreads32) reduce32_kernel(ConstPtrs wires, uint8_t *out, long long NB) {
    chain_entry();
    reduce32_run<B, R, U>(wires, out, NB);
}

// The per-block Phase-1B of the symmetric codec, as a policy of
// reduce_ahead_kernel (the FP4 codec has its own, Fp4BlockReducer).
template <int B>
struct QrBlockReducer {
    static constexpr int kBits = B;
    template <int R>
    static __device__ __forceinline__ void reduce(const BlockWords<B> (&c)[R], const uint32_t (&sb)[R],
                                                  uint8_t *tile, int g) {
        reduce_block<B, R>(c, sb, tile, g);
    }
};

// Block gb's codes and scale from each of the R wires.
template <int B, int R>
__device__ __forceinline__ void load_block_ranks(const ConstPtrs &wires, long long gb, BlockWords<B> (&c)[R],
                                                 uint32_t (&sb)[R]) {
    const long long off = (gb >> 6) * Codec<B>::kTileBytes;
    const int g = static_cast<int>(gb & 63);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint8_t *tile = static_cast<const uint8_t *>(wires.p[r]) + off;
        load_block_codes<B>(tile, g, c[r]);
        sb[r] = load_block_scale_bits<B>(tile, g);
    }
}

// Phase-1B from registers, one block per thread and one block ahead: the
// loads of the thread's next block (a grid stride on) are issued before this
// block is reduced, so every thread has loads in flight while it computes;
// two register sets take turns.  MINB caps the registers (CTAs per SM).
// Same results as reduce32_kernel and staged_reduce_kernel.
template <class P, int R, int MINB>
__global__ void __launch_bounds__(kThreads32, MINB) reduce_ahead_kernel(ConstPtrs wires, uint8_t *out,
                                                                        long long NB) {
    chain_entry();
    constexpr int B = P::kBits;
    const long long S = static_cast<long long>(gridDim.x) * kThreads32;
    long long gb = static_cast<long long>(blockIdx.x) * kThreads32 + threadIdx.x;
    if (gb >= NB) return;
    BlockWords<B> ca[R], cb[R];
    uint32_t sa[R], sbb[R];
    load_block_ranks<B, R>(wires, gb, ca, sa);
    while (true) {
        if (gb + S < NB) load_block_ranks<B, R>(wires, gb + S, cb, sbb);
        P::template reduce<R>(ca, sa, out + (gb >> 6) * Codec<B>::kTileBytes, static_cast<int>(gb & 63));
        gb += S;
        if (gb >= NB) break;
        if (gb + S < NB) load_block_ranks<B, R>(wires, gb + S, ca, sa);
        P::template reduce<R>(cb, sbb, out + (gb >> 6) * Codec<B>::kTileBytes, static_cast<int>(gb & 63));
        gb += S;
        if (gb >= NB) break;
    }
}

// Where the symmetric codec's Phase-1B of a long message (from 48 tiles per
// SM) runs reduce_ahead_kernel, with how many CTAs per SM (0 = not: the
// staged kernel for INT4/6/8, reduce32_kernel for INT3).  Measured on GB300
// at 2^27 (2^28) bf16 values per rank, fraction of the copy bandwidth, with
// the exact integer sum: default kernel -> one block ahead, INT4 R=2 0.634
// (0.660) -> 0.685 (0.711) at three CTAs per SM, R=4 0.788 (0.822) -> 0.834
// (0.863), R=5 0.814 (0.842) -> 0.880 (0.911), R=6 0.898 (0.928) -> 0.940
// (0.976), R=7 0.928 (0.959) -> 0.950 (0.981), R=8 0.970 (1.000) -> 0.980
// (1.003); INT6 R=5 0.822 (0.844) -> 0.839 (0.859); INT3 R=7 0.610 (0.631)
// -> 0.626 (0.640), R=8 0.634 (0.652) -> 0.649 (0.663); and the other
// choices below still the fastest of 0, 2, 3 (and 4 at R = 2) CTAs per SM
// (INT6 R=2 three, R=3 and 4 two; INT4 R=3 three; INT3 R=2 two).  With the
// float sum, INT8 R=4 0.965 (0.992) -> 0.988 (1.013).  Elsewhere the one
// block ahead was slower or within 1%.
template <int B, int R>
__host__ __device__ constexpr int reduce_ahead_min_blocks() {
    return (B == 8 && R == 4)                       ? 2
           : (B == 6 && R == 2)                     ? 3
           : (B == 6 && R >= 3 && R <= 5)           ? 2
           : (B == 4 && (R == 2 || R == 3))         ? 3
           : (B == 4 && R >= 4)                     ? 2
           : (B == 3 && (R == 2 || R >= 7))         ? 2
                                                    : 0;
}

// Phase-1B's register-fed kernels take one block per thread.  (A kernel with
// two threads per block, the pair sharing the absmax by a shuffle, was
// faster for INT4 / INT6 at six or more ranks while the sum was in fp32;
// with the exact integer sum one thread per block was faster there too: at
// 2^23 values per rank 0.34-0.44 -> 0.39-0.46 of the copy bandwidth, and
// the two-shot's owner reductions at 2^27 0.89-0.94 -> 0.93-0.98.)
template <int R>
__host__ __device__ constexpr int reduce_units_per_thread() { return (R <= 2) ? 2 : 1; }

// The symmetric codec's Phase-1B as a policy for staged_reduce_kernel: one
// 32-value block per thread, 64 threads per tile.
template <int B>
struct QrReduce {
    static constexpr int kThreads = 64;
    static constexpr int kCtaThreads = (B == 4 || B == 6) ? 640 : 512;  // see StagedReduceShape
    static constexpr uint32_t kTileIn = Codec<B>::kTileBytes, kTileOut = Codec<B>::kTileBytes;
    template <int R>
    struct Regs {
        BlockWords<B> c[R];
        uint32_t sb[R];
    };
    template <int R>
    static __device__ __forceinline__ void load(const uint8_t *stage, int k, Regs<R> &g) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            load_block_codes<B>(stage + r * kTileIn, k, g.c[r]);
            g.sb[r] = load_block_scale_bits<B>(stage + r * kTileIn, k);
        }
    }
    template <int R>
    static __device__ __forceinline__ void reduce(const Regs<R> &g, uint8_t *tile_out, int k, long long, long long) {
        reduce_block<B, R>(g.c, g.sb, tile_out, k);
    }
};

// Phase-1B with the R ranks' wire tiles staged through shared memory by the
// bulk-copy engine (the same pipeline as the staged fused kernel in
// qr_staged.cuh), generic over the codec (a policy P: QrReduce, FcReduce):
// persistent, one CTA per SM of G groups of P::kThreads threads, one tile
// per group at a time.  Each group owns a ring of SG stages of R input
// tiles; its leader fills stage j % SG with the group's tile j (R bulk
// copies counted on the stage's mbarrier).  The group copies its share of
// the stage into registers, meets at a named barrier that also ANDs "my
// wait completed", the leader refills the stage with tile j + SG, and the
// group reduces and writes its part of the output tile while that copy is
// in flight.  A wire is whole tiles, so there is no ragged tile.  Every
// wait gives up after one second (the group then counts one timeout, its
// leader waits, bounded again, for its copies, and it returns).
template <class P, int R, int G, int SG>
__global__ void __launch_bounds__(P::kThreads * G, 1) staged_reduce_kernel(ConstPtrs wires, uint8_t *out,
                                                                          long long T, long long n,
                                                                          unsigned *timeouts) {
    chain_entry();
    static_assert(G >= 1 && G <= 15 && SG >= 1, "named barriers 1..G, at least one stage per group");
    constexpr uint32_t kStageBytes = R * P::kTileIn;
    extern __shared__ __align__(128) uint8_t ring[];  // G * SG * R * P::kTileIn bytes
    __shared__ __align__(8) uint64_t full[G * SG];
    __shared__ const uint8_t *src[R];

    if (threadIdx.x == 0) {
        for (int s = 0; s < G * SG; ++s) mbar_init(&full[s], 1);
        for (int r = 0; r < R; ++r) src[r] = static_cast<const uint8_t *>(wires.p[r]);
        mbar_init_fence();
    }
    __syncthreads();

    const int g = threadIdx.x / P::kThreads, k = threadIdx.x % P::kThreads;
    const bool leader = k == 0;
    const long long first = blockIdx.x + static_cast<long long>(gridDim.x) * g;
    const long long stride = static_cast<long long>(gridDim.x) * G;
    const int tiles = T > first ? static_cast<int>((T - first + stride - 1) / stride) : 0;
    uint8_t *my_ring = ring + static_cast<size_t>(g) * SG * kStageBytes;
    uint64_t *my_full = full + g * SG;

    auto issue = [&](int j) {  // leader only: stage j % SG <- tile j of every rank
        const int s = j % SG;
        const long long off = (first + j * stride) * P::kTileIn;
        uint8_t *dst = my_ring + static_cast<size_t>(s) * kStageBytes;
        mbar_arrive_expect_tx(&my_full[s], kStageBytes);
#pragma unroll
        for (int r = 0; r < R; ++r) bulk_copy_g2s(dst + r * P::kTileIn, src[r] + off, P::kTileIn, &my_full[s]);
    };

    int issued = 0;
    if (leader)
        for (; issued < tiles && issued < SG; ++issued) issue(issued);

    int j = 0;
    for (; j < tiles; ++j) {
        const int s = j % SG;
        const bool ok = mbar_wait(&my_full[s], static_cast<uint32_t>((j / SG) & 1));
        typename P::template Regs<R> regs;
        P::template load<R>(my_ring + static_cast<size_t>(s) * kStageBytes, k, regs);
        if (!group_all<P::kThreads>(1 + g, ok)) break;  // also: every thread is done reading stage s
        if (leader && issued < tiles) issue(issued++);
        const long long t = first + j * stride;
        P::template reduce<R>(regs, out + t * P::kTileOut, k, t, n);
    }
    if (j < tiles && leader) {  // a wait ran out
        atomicAdd(timeouts, 1u);
        for (int i = j; i < issued; ++i)
            if (!mbar_wait(&my_full[i % SG], static_cast<uint32_t>((i / SG) & 1))) break;
    }
}

// Most ring stages per group: four, but one for INT8 from four ranks (the
// memory-bound case, where a deeper ring measured slower): at 2^27 / 2^28
// bf16 values per rank, R = 5 0.92 / 0.93 -> 1.00 / 1.02 of HBM (was two
// stages), R = 4 0.96 / 0.97 -> 0.97 / 1.00 (was two).
template <class P, int R>
struct StagedReduceStageCap {
    static constexpr int value = 4;
};
template <int R>
struct StagedReduceStageCap<QrReduce<8>, R> {
    static constexpr int value = (R >= 4) ? 1 : 4;
};

// Launch shape of the staged Phase-1B kernel: P::kCtaThreads threads (groups
// of P::kThreads), each group with as many stages (at most 4) as fit in
// 200 KiB of shared memory at R * tile-bytes per stage.  Measured on GB300 at
// 2^27 bf16 values per rank against the register-fed kernels (fraction of the
// measured HBM bandwidth, 4 / 8 / 12 groups of 64 threads): INT8 R=8 0.96 ->
// 0.93 / 1.00 / 0.83, R=2 0.76 -> 0.69 / 0.92 / 0.89; INT6 R=8 0.64 -> 0.63 /
// 0.76 / 0.72; INT4 R=8 0.60 -> 0.54 / 0.67 / 0.69; INT3 R=8 0.34 -> 0.29 /
// 0.34 / 0.34 (bound by the integer pipe, not by memory: it stays on
// reduce32_kernel).  Ten groups (640 threads, 20 warps at up to 96
// registers) against eight: INT4 +2..4% at R = 2, 4, 8 (latency-bound: more
// warps hide more); INT6, once its Phase-1B decoded through fp16, +3% at
// R = 2, +9% at R = 6 (0.73 -> 0.80 at 2^28), equal at R = 4, 8; INT8 -7% at
// R = 8 (one stage per group left in 200 KiB); so ten for INT4 and INT6.
// Deeper rings do not pay: a 224 KiB budget (one more stage for INT8 at
// R = 3, 4, 6, INT4 / FP4 at R = 6, FC 8->8 at R = 5, 7) measured INT8
// -3 / -6 / -11%, FP4 -3.5%, FC 8->8 R = 7 -2.5%, INT4 equal.  The asymmetric codec's policy runs five
// groups of 128 threads (640), 5-10% faster than four at R = 4, 6, 8 for
// every width pair.
template <class P, int R>
struct StagedReduceShape {
    static constexpr int kGroups = P::kCtaThreads / P::kThreads;
    static constexpr int kFit = (200 * 1024) / (kGroups * R * P::kTileIn);
    static constexpr int kCap = StagedReduceStageCap<P, R>::value;
    static constexpr int kStages = kFit >= kCap ? kCap : (kFit < 1 ? 1 : kFit);
    static constexpr int kSmemBytes = kGroups * kStages * R * P::kTileIn;
    // the ring plus the kernel's static barriers and pointers within one CTA's 227 KB
    static_assert(kSmemBytes + 1024 <= 227 * 1024, "staged Phase-1B ring exceeds the shared memory of a CTA");
};

}  // namespace qrk
