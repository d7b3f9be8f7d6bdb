// qr_kernels_fc.cuh -- the Flash Communication codec: asymmetric quantization
// in groups of 128 values ("Flash Communication" review record, arXiv
// 2412.04964: key machinery "asymmetric group-128 scaling", re-quantization of
// the partial sums, INT4 reduce-scatter + INT8 all-gather as "INT6").
//
// Arithmetic (the same steps as the library's reference definition):
//   per group: lo = min x, hi = max x; s = RN(RN(hi - lo) / (2^b - 1)), 0 if
//   below 2^-126; z = lo + 0 (a zero minimum is +0); r = RN(1/s) (0 if s = 0);
//   u = RNE(RN(x - z) * r), the product taken exactly (one rounding: a fused
//   multiply-add with 1.5*2^23); decode = RN(u*s + z) (one fma);
//   Phase-1B: acc = decode_0, acc = RN(acc + decode_r), values past n reset to
//   0, re-quantized at the all-gather width.
// u never exceeds 2^b - 1: d <= range and d*r <= range * RN(1/RN(range/umax))
// <= umax * (1 + 2^-24) / (1 - 2^-24) < umax + 1/2, so no cap is applied.
//
// Tile (2048 values = 16 groups): codes as in the symmetric codec (INT4 /
// INT8), then 16 fp32 scales at 256*b and 16 fp32 zero points at 256*b + 64.
// Thread mapping: 128 threads per tile, thread i owns values 16i..16i+15
// (slots 2i and 2i+1), so lanes 8k..8k+7 own group k of their warp's tile
// quarter and combine min and max with three butterfly shuffles.
#pragma once

#include "qr_kernels32.cuh"

namespace qrk {

template <int B>
struct FcCodec {
    static_assert(B == 4 || B == 8, "the Flash Communication codec is INT4 or INT8");
    static constexpr int kUmax = (1 << B) - 1;
    static constexpr int kMeta = 256 * B;            // scales at kMeta, zero points at kMeta + 64
    static constexpr int kTileBytes = 256 * B + 128;
};

struct FcParams {
    float s, r, z;
};

// Group minimum and maximum across the 8 lanes of a group (every lane of the
// warp must call it).
__device__ __forceinline__ void group_minmax(const float2 (&v)[8], float &lo, float &hi) {
    lo = fminf(v[0].x, v[0].y);
    hi = fmaxf(v[0].x, v[0].y);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        lo = fmin3(lo, v[i].x, v[i].y);
        hi = fmax3(hi, v[i].x, v[i].y);
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, m));
        hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, m));
    }
}

template <int B>
__device__ __forceinline__ FcParams fc_params(float lo, float hi) {
    FcParams p;
    float s = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(FcCodec<B>::kUmax));
    if (!(s >= 0x1p-126f)) s = 0.0f;
    p.s = s;
    p.z = __fadd_rn(lo, 0.0f);  // -0 -> +0
    p.r = (s == 0.0f) ? 0.0f : __frcp_rn(s);
    return p;
}

// f = RN(d*r + 1.5*2^23) = RNE(d*r) + 1.5*2^23 with d = RN(x - z): the exact
// product rounded once to an integer (0 <= d*r < 2^22, and the fp32 spacing
// in [2^23, 2^24) is 1); the code is in the low byte.
template <int B>
__device__ __forceinline__ void fc_quantize16(const float2 (&v)[8], const FcParams &p, float2 (&f)[8]) {
    const float2 nz = make_float2(-p.z, -p.z);
    const float2 r2 = make_float2(p.r, p.r);
    const float2 m2 = make_float2(kRoundMagic, kRoundMagic);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __ffma2_rn(__fadd2_rn(v[i], nz), r2, m2);
}

// decode of magic floats: RN(u*s + z)
__device__ __forceinline__ void fc_dequant16(const float2 (&f)[8], const FcParams &p, float2 (&o)[8]) {
    const float2 nm = make_float2(-kRoundMagic, -kRoundMagic);
    const float2 s2 = make_float2(p.s, p.s);
    const float2 z2 = make_float2(p.z, p.z);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __ffma2_rn(__fadd2_rn(f[i], nm), s2, z2);
}

// The 16 codes of thread i's two slots as u (exact floats), pairwise.
template <int B>
__device__ __forceinline__ void fc_unpack16(const HalfWords<B> &c, float2 (&u)[8]) {
    const float2 nm = make_float2(-kRoundMagic, -kRoundMagic);
#pragma unroll
    for (int sl = 0; sl < 2; ++sl) {
        uint32_t even, odd;
        slot_even_odd_codes<B>(half_slot_codes<B>(c, sl), even, odd);
        u[4 * sl + 0] = __fadd2_rn(make_float2(byte_as_magic<0>(even), byte_as_magic<0>(odd)), nm);
        u[4 * sl + 1] = __fadd2_rn(make_float2(byte_as_magic<1>(even), byte_as_magic<1>(odd)), nm);
        u[4 * sl + 2] = __fadd2_rn(make_float2(byte_as_magic<2>(even), byte_as_magic<2>(odd)), nm);
        u[4 * sl + 3] = __fadd2_rn(make_float2(byte_as_magic<3>(even), byte_as_magic<3>(odd)), nm);
    }
}

// Thread i's packed codes and its group's (scale, zero point) into `tile`.
template <int B>
__device__ __forceinline__ void fc_store_packed16(uint8_t *tile, int i, const HalfWords<B> &c, const FcParams &p) {
    store_half_codes<B>(tile, i >> 1, i & 1, c);
    if ((i & 7) == 0) {
        const int g = i >> 3;
        *reinterpret_cast<float *>(tile + FcCodec<B>::kMeta + 4 * g) = p.s;
        *reinterpret_cast<float *>(tile + FcCodec<B>::kMeta + 64 + 4 * g) = p.z;
    }
}

template <int B>
__device__ __forceinline__ void fc_store16(uint8_t *tile, int i, const float2 (&f)[8], const FcParams &p) {
    HalfWords<B> c;
    pack_half<B>(f, c);
    fc_store_packed16<B>(tile, i, c, p);
}

template <int B>
__device__ __forceinline__ void fc_load16(const uint8_t *tile, int i, HalfWords<B> &c, float &s, float &z) {
    load_half_codes<B>(tile, i >> 1, i & 1, c);
    const int g = i >> 3;
    s = *reinterpret_cast<const float *>(tile + FcCodec<B>::kMeta + 4 * g);
    z = *reinterpret_cast<const float *>(tile + FcCodec<B>::kMeta + 64 + 4 * g);
}

// 16 values at `base` (32 bytes); past n they read as +0.  A32: 32-byte
// aligned pointer (one 256-bit load), else two 16-byte loads.
template <bool A32>
__device__ __forceinline__ void load16v(const uint16_t *x, long long base, long long n, uint32_t (&w)[8]) {
    if (base + 16 <= n) {
        if constexpr (A32) {
            ld_stream32(x + base, w);
        } else {
            const uint4 a = reinterpret_cast<const uint4 *>(x + base)[0];
            const uint4 b = reinterpret_cast<const uint4 *>(x + base)[1];
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (base + 2 * i < n) ? x[base + 2 * i] : 0u;
            const uint32_t hi = (base + 2 * i + 1 < n) ? x[base + 2 * i + 1] : 0u;
            w[i] = lo | (hi << 16);
        }
    }
}

template <int DT, bool A32>
__device__ __forceinline__ void store16v(uint16_t *y, long long base, long long n, const float2 (&o)[8]) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = narrow2<DT>(o[i].x, o[i].y);
    if (base + 16 <= n) {
        if constexpr (A32) {
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

// Values at or past n are zero in every phase (a padded zero does not decode
// back to exactly 0, so the Phase-1B sums there are reset).
__device__ __forceinline__ void zero_past_n(float2 (&a)[8], long long base, long long n) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (base + 2 * i >= n) a[i].x = 0.0f;
        if (base + 2 * i + 1 >= n) a[i].y = 0.0f;
    }
}

constexpr int kThreadsFc = 128;

// The fused two-shot all-reduce with the Flash Communication codec: quantize
// every rank at BRS bits, decode and add in rank order, re-quantize at BAG
// bits, decode into y.  Codes never leave registers.
template <int BRS, int BAG, int DT, int R, bool A32>
__global__ void __launch_bounds__(kThreadsFc, 4) fc_allreduce_kernel(ConstPtrs x, long long n, uint16_t *y,
                                                                     long long T) {
    chain_entry();
    const int i = threadIdx.x;
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        const long long base = t * kTileValues + 16 * i;
        uint32_t raw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) load16v<A32>(static_cast<const uint16_t *>(x.p[r]), base, n, raw[r]);
        float2 acc[8];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2 v[8], f[8], d[8];
            widen16<DT>(raw[r], v);
            float lo, hi;
            group_minmax(v, lo, hi);
            const FcParams p = fc_params<BRS>(lo, hi);
            fc_quantize16<BRS>(v, p, f);
            fc_dequant16(f, p, d);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = (r == 0) ? d[k] : __fadd2_rn(acc[k], d[k]);
        }
        if (base + 16 > n) zero_past_n(acc, base, n);
        float lo, hi;
        group_minmax(acc, lo, hi);
        const FcParams p = fc_params<BAG>(lo, hi);
        float2 f[8], o[8];
        fc_quantize16<BAG>(acc, p, f);
        fc_dequant16(f, p, o);
        store16v<DT, A32>(y, base, n, o);
    }
}

// The per-tile steps of fc_allreduce_kernel as a policy for the staged kernel
// (staged_allreduce_kernel in qr_staged.cuh).  Every step before the store
// is per value or over a whole group of 128, so a thread may hold its two
// 8-value halves exchanged; values past n only occur in the ragged tile.
template <int BRS, int BAG, int DT>
struct FcTile {
    static __device__ __forceinline__ void accumulate(const uint32_t (&w)[8], float2 (&acc)[8], bool first) {
        float2 v[8], f[8], d[8];
        widen16<DT>(w, v);
        float lo, hi;
        group_minmax(v, lo, hi);
        const FcParams p = fc_params<BRS>(lo, hi);
        fc_quantize16<BRS>(v, p, f);
        fc_dequant16(f, p, d);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = first ? d[k] : __fadd2_rn(acc[k], d[k]);
    }
    static __device__ __forceinline__ void finish(const float2 (&acc)[8], uint16_t *y, long long base, long long,
                                                  bool swapped) {
        float lo, hi;
        group_minmax(acc, lo, hi);
        const FcParams p = fc_params<BAG>(lo, hi);
        float2 f[8], o[8];
        fc_quantize16<BAG>(acc, p, f);
        fc_dequant16(f, p, o);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = narrow2<DT>(o[k].x, o[k].y);
        if (swapped)
            st_global32_swapped(y + base, w);
        else
            st_global32(y + base, w);
    }
    // The last, partial tile with bounds-checked loads (not inlined, so that
    // it does not set the register budget of the staged kernel's main loop).
    template <int R>
    static __device__ __noinline__ void ragged(const ConstPtrs &x, long long n, uint16_t *y, long long base) {
        float2 acc[8];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint32_t w[8];
            load16v<true>(static_cast<const uint16_t *>(x.p[r]), base, n, w);
            accumulate(w, acc, r == 0);
        }
        if (base + 16 > n) zero_past_n(acc, base, n);
        float lo, hi;
        group_minmax(acc, lo, hi);
        const FcParams p = fc_params<BAG>(lo, hi);
        float2 f[8], o[8];
        fc_quantize16<BAG>(acc, p, f);
        fc_dequant16(f, p, o);
        store16v<DT, true>(y, base, n, o);
    }
};

// Thread i's 16 values of tile t (values past n read as +0) quantized at B
// bits into `tile`: group min / max over 8 lanes, parameters, codes.
// Called by whole warps.
template <int B, int DT, bool A32>
__device__ __forceinline__ void fc_encode_tile16(const uint16_t *__restrict__ x, long long n, long long t, int i,
                                                 uint8_t *tile) {
    uint32_t raw[8];
    load16v<A32>(x, t * kTileValues + 16 * i, n, raw);
    float2 v[8], f[8];
    widen16<DT>(raw, v);
    float lo, hi;
    group_minmax(v, lo, hi);
    const FcParams p = fc_params<B>(lo, hi);
    fc_quantize16<B>(v, p, f);
    fc_store16<B>(tile, i, f, p);
}

// Send path: quantize into a BITS-wide Flash Communication wire.
template <int B, int DT, bool A32>
__global__ void __launch_bounds__(kThreadsFc) fc_encode_kernel(const uint16_t *__restrict__ x, long long n,
                                                               uint8_t *__restrict__ wire, long long T) {
    chain_entry();
    for (long long t = blockIdx.x; t < T; t += gridDim.x)
        fc_encode_tile16<B, DT, A32>(x, n, t, threadIdx.x, wire + t * FcCodec<B>::kTileBytes);
}

// Receive path / Phase-2: decode the first n values.
template <int B, int DT, bool A32>
__global__ void __launch_bounds__(kThreadsFc) fc_decode_kernel(const uint8_t *__restrict__ wire, long long n,
                                                               uint16_t *__restrict__ y, long long T) {
    chain_entry();
    const int i = threadIdx.x;
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        HalfWords<B> c;
        FcParams p;
        fc_load16<B>(wire + t * FcCodec<B>::kTileBytes, i, c, p.s, p.z);
        float2 u[8], o[8];
        fc_unpack16<B>(c, u);
        const float2 s2 = make_float2(p.s, p.s), z2 = make_float2(p.z, p.z);
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = __ffma2_rn(u[k], s2, z2);
        store16v<DT, A32>(y, t * kTileValues + 16 * i, n, o);
    }
}

// Phase-1B: decode R BIN-wide wires, add in rank order, reset values past n,
// re-quantize into a BOUT-wide wire.
// Phase-1B of one tile for thread i (values base..base+15): decode the R
// ranks' codes c[r] with their group scale s[r] and zero point z[r], add in
// rank order, reset values past n, re-quantize at BOUT bits: the magic
// floats of the codes in f, the group's parameters in p.  Called by whole
// warps (the group min / max spans 8 lanes).
template <int BIN, int BOUT, int R>
__device__ __forceinline__ void fc_reduce_values(const HalfWords<BIN> (&c)[R], const float (&s)[R],
                                                 const float (&z)[R], long long base, long long n, float2 (&f)[8],
                                                 FcParams &p) {
    float2 acc[8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float2 u[8];
        fc_unpack16<BIN>(c[r], u);
        const float2 s2 = make_float2(s[r], s[r]), z2 = make_float2(z[r], z[r]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 d = __ffma2_rn(u[k], s2, z2);
            acc[k] = (r == 0) ? d : __fadd2_rn(acc[k], d);
        }
    }
    if (base + 16 > n) zero_past_n(acc, base, n);
    float lo, hi;
    group_minmax(acc, lo, hi);
    p = fc_params<BOUT>(lo, hi);
    fc_quantize16<BOUT>(acc, p, f);
}

// fc_reduce_values, stored into tile_out.
template <int BIN, int BOUT, int R>
__device__ __forceinline__ void fc_reduce_tile(const HalfWords<BIN> (&c)[R], const float (&s)[R], const float (&z)[R],
                                               uint8_t *tile_out, int i, long long base, long long n) {
    float2 f[8];
    FcParams p;
    fc_reduce_values<BIN, BOUT, R>(c, s, z, base, n, f, p);
    fc_store16<BOUT>(tile_out, i, f, p);
}

// U tiles a grid stride apart per iteration, the loads of all U issued
// before any arithmetic (the kernel is bound by latency, not by a pipe: with
// one tile in flight its issue rate stayed near 0.63 of the peak).  The
// branch on t < T is uniform across the CTA, so whole warps reach the group
// shuffles.
template <int BIN, int BOUT, int R, int U>
__global__ void __launch_bounds__(kThreadsFc, 4) fc_reduce_kernel(ConstPtrs wires, long long n, uint8_t *out,
                                                                  long long T) {
    chain_entry();
    const int i = threadIdx.x;
    const long long S = gridDim.x;
    for (long long t0 = blockIdx.x; t0 < T; t0 += U * S) {
        HalfWords<BIN> c[U][R];
        float s[U][R], z[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long t = t0 + u * S;
            if (t < T) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    fc_load16<BIN>(static_cast<const uint8_t *>(wires.p[r]) + t * FcCodec<BIN>::kTileBytes, i,
                                   c[u][r], s[u][r], z[u][r]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long t = t0 + u * S;
            if (t < T)
                fc_reduce_tile<BIN, BOUT, R>(c[u], s[u], z[u], out + t * FcCodec<BOUT>::kTileBytes, i,
                                             t * kTileValues + 16 * i, n);
        }
    }
}

// One tile's R code words, scales and zero points, as one thread holds them.
template <int BIN, int R>
struct FcReduceSet {
    HalfWords<BIN> c[R];
    float s[R], z[R];
};

template <int BIN, int R>
__device__ __forceinline__ void fc_load_set(const ConstPtrs &wires, long long t, int i, FcReduceSet<BIN, R> &g) {
#pragma unroll
    for (int r = 0; r < R; ++r)
        fc_load16<BIN>(static_cast<const uint8_t *>(wires.p[r]) + t * FcCodec<BIN>::kTileBytes, i, g.c[r], g.s[r],
                       g.z[r]);
}

// Phase-1B one tile ahead: the loads of the CTA's next tile (a grid stride
// on) are issued before this tile is reduced, so every thread has loads in
// flight while it computes; two register sets take turns.  MINB caps the
// registers (CTAs per SM).  Same results as fc_reduce_kernel.
template <int BIN, int BOUT, int R, int MINB>
__global__ void __launch_bounds__(kThreadsFc, MINB) fc_reduce_ahead_kernel(ConstPtrs wires, long long n,
                                                                           uint8_t *out, long long T) {
    chain_entry();
    const int i = threadIdx.x;
    const long long S = gridDim.x;
    long long t = blockIdx.x;
    if (t >= T) return;
    FcReduceSet<BIN, R> a, b;
    fc_load_set<BIN, R>(wires, t, i, a);
    while (true) {
        if (t + S < T) fc_load_set<BIN, R>(wires, t + S, i, b);
        fc_reduce_tile<BIN, BOUT, R>(a.c, a.s, a.z, out + t * FcCodec<BOUT>::kTileBytes, i, t * kTileValues + 16 * i,
                                     n);
        t += S;
        if (t >= T) break;
        if (t + S < T) fc_load_set<BIN, R>(wires, t + S, i, a);
        fc_reduce_tile<BIN, BOUT, R>(b.c, b.s, b.z, out + t * FcCodec<BOUT>::kTileBytes, i, t * kTileValues + 16 * i,
                                     n);
        t += S;
        if (t >= T) break;
    }
}

// The Flash Communication Phase-1B as a policy for staged_reduce_kernel
// (qr_kernels32.cuh): 16 values per thread, 128 threads per tile.
template <int BIN, int BOUT>
struct FcReduce {
    static constexpr int kThreads = kThreadsFc;
    static constexpr int kCtaThreads = 640;  // five groups: 5-10% over four at R = 4..8
    static constexpr uint32_t kTileIn = FcCodec<BIN>::kTileBytes, kTileOut = FcCodec<BOUT>::kTileBytes;
    template <int R>
    struct Regs {
        HalfWords<BIN> c[R];
        float s[R], z[R];
    };
    template <int R>
    static __device__ __forceinline__ void load(const uint8_t *stage, int k, Regs<R> &g) {
#pragma unroll
        for (int r = 0; r < R; ++r) fc_load16<BIN>(stage + r * kTileIn, k, g.c[r], g.s[r], g.z[r]);
    }
    template <int R>
    static __device__ __forceinline__ void reduce(const Regs<R> &g, uint8_t *tile_out, int k, long long t,
                                                  long long n) {
        fc_reduce_tile<BIN, BOUT, R>(g.c, g.s, g.z, tile_out, k, t * kTileValues + 16 * k, n);
    }
};

}  // namespace qrk
