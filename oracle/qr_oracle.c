/*
 * qr_oracle.c -- slow, scalar CPU oracle for the block-quantized two-shot
 * all-reduce codec.  TEST INFRASTRUCTURE ONLY (see qr_oracle.h): the product
 * path never includes, links or calls this file.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off matters: every float operation below must round on its
 * own (x*r is rounded before the clip, the rank sum is rounded after each
 * add), exactly as written.
 *
 * Citations name the source page and section:
 *   [QR]  "QuickReduce INT3 quantization and benchmarking on MI355" (AMD blog)
 *   [FC]  "Flash Communication" review record, arXiv 2412.04964
 */
#include "qr_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define TILE 2048   /* values per tile: 1152 B = 2048/2 + 64*2 for INT4 [QR Design Highlights] */
#define BLOCK 32    /* values per fp16 scale [QR Design Highlights] */
#define NBLOCK (TILE / BLOCK)
#define NSLOT (TILE / 8)  /* one q2w uint16 / q1w uint8 per 8-value slot [QR Design Highlights] */

/* ------------------------------------------------------------------------ */
/* Number formats, written from the IEEE-754 definitions.  Every float is a  */
/* dyadic rational that a double holds exactly, so each conversion is done  */
/* on exact values: find the quantum (the spacing of representable values   */
/* at the input's magnitude), round |x|/quantum to the nearest integer with  */
/* ties to even, and assemble the bit pattern.                               */
/* ------------------------------------------------------------------------ */

/* Nearest multiple of `quantum` (a power of two) to a >= 0, ties to the even
 * multiple.  a/quantum is exact in double, so is its fractional part. */
static double round_to_quantum(double a, double quantum)
{
    double v = a / quantum;
    double fl = floor(v);
    double frac = v - fl;
    if (frac > 0.5) return (fl + 1.0) * quantum;
    if (frac < 0.5) return fl * quantum;
    return (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0) * quantum;
}

/* floor(log2(a)) for a > 0, exactly (frexp is exact). */
static int ilog2(double a)
{
    int e;
    frexp(a, &e);
    return e - 1;
}

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
 * Normal quantum 2^(E-10) for E >= -14, subnormal quantum 2^-24,
 * largest finite 65504; anything that rounds above it is infinity. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t fb;
    memcpy(&fb, &f, sizeof fb);
    uint16_t sign = (uint16_t)((fb >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int E = ilog2(a);
    double quantum = (E < -14) ? ldexp(1.0, -24) : ldexp(1.0, E - 10);
    double r = round_to_quantum(a, quantum);
    if (r > 65504.0) return (uint16_t)(sign | 0x7C00u);
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) /* subnormal: r = m * 2^-24, m < 1024 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    E = ilog2(r);
    double frac = r / ldexp(1.0, E) - 1.0; /* a multiple of 2^-10 in [0,1) */
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(frac * 1024.0));
}

float orc_f16_to_f32(uint16_t h)
{
    int sign = h >> 15;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (ex == 0x1F) v = man ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)man, -24);
    else v = ldexp((double)(1024 + man), ex - 25);
    return (float)(sign ? -v : v);
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.
 * Normal quantum 2^(E-7) for E >= -126, subnormal quantum 2^-133,
 * largest finite (2 - 2^-7) * 2^127. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t fb;
    memcpy(&fb, &f, sizeof fb);
    uint16_t sign = (uint16_t)((fb >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(f)) return (uint16_t)(sign | 0x7F80u);
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int E = ilog2(a);
    double quantum = (E < -126) ? ldexp(1.0, -133) : ldexp(1.0, E - 7);
    double r = round_to_quantum(a, quantum);
    if (r > ldexp(255.0, 120)) return (uint16_t)(sign | 0x7F80u); /* (2-2^-7)*2^127 */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -126))
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
    E = ilog2(r);
    double frac = r / ldexp(1.0, E) - 1.0; /* a multiple of 2^-7 in [0,1) */
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)(frac * 128.0));
}

float orc_bf16_to_f32(uint16_t h)
{
    int sign = h >> 15;
    int ex = (h >> 7) & 0xFF;
    int man = h & 0x7F;
    double v;
    if (ex == 0xFF) v = man ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)man, -133);
    else v = ldexp((double)(128 + man), ex - 134);
    return (float)(sign ? -v : v);
}

void orc_f32_to_f16_n(const float *f, size_t n, uint16_t *h)
{
    for (size_t i = 0; i < n; ++i) h[i] = orc_f32_to_f16(f[i]);
}

void orc_f16_to_f32_n(const uint16_t *h, size_t n, float *f)
{
    for (size_t i = 0; i < n; ++i) f[i] = orc_f16_to_f32(h[i]);
}

void orc_f32_to_bf16_n(const float *f, size_t n, uint16_t *h)
{
    for (size_t i = 0; i < n; ++i) h[i] = orc_f32_to_bf16(f[i]);
}

void orc_bf16_to_f32_n(const uint16_t *h, size_t n, float *f)
{
    for (size_t i = 0; i < n; ++i) f[i] = orc_bf16_to_f32(h[i]);
}

static float widen(int dtype, uint16_t h)
{
    return dtype == ORC_FP16 ? orc_f16_to_f32(h) : orc_bf16_to_f32(h);
}

static uint16_t narrow(int dtype, float f)
{
    return dtype == ORC_FP16 ? orc_f32_to_f16(f) : orc_f32_to_bf16(f);
}

/* ------------------------------------------------------------------------ */
/* Sizes and the tile layout                                                 */
/* ------------------------------------------------------------------------ */

static int bits_ok(int bits) { return bits == 3 || bits == 4 || bits == 6 || bits == 8; }

size_t orc_tile_values(void) { return TILE; }

/* Codes take bits*2048/8 = 256*bits bytes, then 64 fp16 scales (128 B):
 * INT4 1152 B and INT3 896 B as printed in [QR Design Highlights]. */
size_t orc_tile_bytes(int bits)
{
    return bits_ok(bits) ? (size_t)256 * (size_t)bits + 128 : 0;
}

size_t orc_wire_bytes(int bits, size_t n)
{
    return ((n + TILE - 1) / TILE) * orc_tile_bytes(bits);
}

static size_t scale_offset(int bits) { return (size_t)256 * (size_t)bits; }

static void put_u16(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)((v >> 8) & 0xFF);
}

static void put_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)((v >> 8) & 0xFF);
    p[2] = (uint8_t)((v >> 16) & 0xFF);
    p[3] = (uint8_t)((v >> 24) & 0xFF);
}

static uint32_t get_u16(const uint8_t *p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }

static uint32_t get_u32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* Slot k of a tile holds the codes u[0..7] of values 8k..8k+7. */
static void pack_slot(int bits, const uint8_t *u, uint8_t *tile, int k)
{
    uint32_t lo = 0, hi = 0;
    int j;
    switch (bits) {
    case 8: /* one byte per code */
        for (j = 0; j < 8; ++j) tile[8 * k + j] = u[j];
        break;
    case 4: /* eight 4-bit codes in one 32-bit word [QR Design Highlights] */
        for (j = 0; j < 8; ++j) lo |= (uint32_t)(u[j] & 0xF) << (4 * j);
        put_u32(tile + 4 * k, lo);
        break;
    case 3: /* low 2 bits -> uint16 q2w, high bit -> uint8 q1w [QR Design Highlights] */
        for (j = 0; j < 8; ++j) {
            lo |= (uint32_t)(u[j] & 0x3) << (2 * j);
            hi |= (uint32_t)((u[j] >> 2) & 0x1) << j;
        }
        put_u16(tile + 2 * k, lo);
        tile[512 + k] = (uint8_t)hi;
        break;
    case 6: /* INT3-style split: low 4 bits as INT4, high 2 bits as a q2w word */
        for (j = 0; j < 8; ++j) {
            lo |= (uint32_t)(u[j] & 0xF) << (4 * j);
            hi |= (uint32_t)((u[j] >> 4) & 0x3) << (2 * j);
        }
        put_u32(tile + 4 * k, lo);
        put_u16(tile + 1024 + 2 * k, hi);
        break;
    }
}

static void unpack_slot(int bits, const uint8_t *tile, int k, uint8_t *u)
{
    uint32_t lo, hi;
    int j;
    switch (bits) {
    case 8:
        for (j = 0; j < 8; ++j) u[j] = tile[8 * k + j];
        break;
    case 4:
        lo = get_u32(tile + 4 * k);
        for (j = 0; j < 8; ++j) u[j] = (uint8_t)((lo >> (4 * j)) & 0xF);
        break;
    case 3:
        lo = get_u16(tile + 2 * k);
        hi = tile[512 + k];
        for (j = 0; j < 8; ++j)
            u[j] = (uint8_t)(((lo >> (2 * j)) & 0x3) | (((hi >> j) & 0x1) << 2));
        break;
    case 6:
        lo = get_u32(tile + 4 * k);
        hi = get_u16(tile + 1024 + 2 * k);
        for (j = 0; j < 8; ++j)
            u[j] = (uint8_t)(((lo >> (4 * j)) & 0xF) | (((hi >> (2 * j)) & 0x3) << 4));
        break;
    }
}

int orc_pack_codes(int bits, const uint8_t *u, size_t ntiles, uint8_t *wire)
{
    if (!bits_ok(bits)) return -1;
    size_t tb = orc_tile_bytes(bits);
    for (size_t t = 0; t < ntiles; ++t)
        for (int k = 0; k < NSLOT; ++k)
            pack_slot(bits, u + t * TILE + 8 * (size_t)k, wire + t * tb, k);
    return 0;
}

int orc_unpack_codes(int bits, const uint8_t *wire, size_t ntiles, uint8_t *u)
{
    if (!bits_ok(bits)) return -1;
    size_t tb = orc_tile_bytes(bits);
    for (size_t t = 0; t < ntiles; ++t)
        for (int k = 0; k < NSLOT; ++k)
            unpack_slot(bits, wire + t * tb, k, u + t * TILE + 8 * (size_t)k);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The block quantizer [QR Design Highlights; Quantization and               */
/* Dequantization Paths]: absmax over the block -> fp16 scale -> scale,      */
/* clip to [qmin, qmax], round, bias to unsigned.                            */
/* ------------------------------------------------------------------------ */

/* Round half to even of a float of small magnitude (|t| <= 128 here). */
static float round_half_even(float t)
{
    double v = (double)t;
    double fl = floor(v);
    double frac = v - fl;
    if (frac > 0.5) return (float)(fl + 1.0);
    if (frac < 0.5) return (float)fl;
    return (float)(fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);
}

int orc_quantize_block(int bits, const float *x, uint8_t *u, uint16_t *scale)
{
    if (!bits_ok(bits)) return -1;
    const int bias = 1 << (bits - 1);  /* |qmin|: [-4,+3] -> [0,7] for INT3 */
    const float qmin = (float)(-bias);
    const float qmax = (float)(bias - 1);
    int i;

    float A = 0.0f; /* block absolute maximum */
    for (i = 0; i < BLOCK; ++i) {
        if (!isfinite(x[i])) return -1; /* non-finite input is outside the contract */
        float a = fabsf(x[i]);
        if (a > A) A = a;
    }
    float d = A / (float)bias; /* power-of-two divide: exact unless it underflows */
    uint16_t sh = orc_f32_to_f16(d);
    if (sh == 0x7C00u) sh = 0x7BFFu; /* the fp16 scale saturates at 65504 */
    float s = orc_f16_to_f32(sh);
    if (s == 0.0f) { /* zero block, or a scale below the fp16 range */
        *scale = 0;
        for (i = 0; i < BLOCK; ++i) u[i] = (uint8_t)bias;
        return 0;
    }
    float r = 1.0f / s; /* fp32 encode factor */
    for (i = 0; i < BLOCK; ++i) {
        float t = x[i] * r;
        if (t < qmin) t = qmin;
        if (t > qmax) t = qmax;
        float q = round_half_even(t);
        u[i] = (uint8_t)((int)q + bias);
    }
    *scale = sh;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tiles: encode (send path) and decode (receive path)                       */
/* ------------------------------------------------------------------------ */

/* x: 2048 fp32 values (already zero-padded). */
static int encode_tile(int bits, const float *x, uint8_t *tile)
{
    uint8_t u[TILE];
    for (int g = 0; g < NBLOCK; ++g) {
        uint16_t sh;
        if (orc_quantize_block(bits, x + BLOCK * g, u + BLOCK * g, &sh) != 0) return -1;
        put_u16(tile + scale_offset(bits) + 2 * (size_t)g, sh);
    }
    for (int k = 0; k < NSLOT; ++k) pack_slot(bits, u + 8 * k, tile, k);
    return 0;
}

/* Recombine the bits, remove the bias, multiply by the block's decode scale.
 * (u - bias) * s is exact in fp32: an 8-bit integer times an 11-bit
 * significand. */
static void decode_tile_f32(int bits, const uint8_t *tile, float *out)
{
    const int bias = 1 << (bits - 1);
    uint8_t u[TILE];
    for (int k = 0; k < NSLOT; ++k) unpack_slot(bits, tile, k, u + 8 * k);
    for (int g = 0; g < NBLOCK; ++g) {
        float s = orc_f16_to_f32((uint16_t)get_u16(tile + scale_offset(bits) + 2 * (size_t)g));
        for (int i = 0; i < BLOCK; ++i) {
            int q = (int)u[BLOCK * g + i] - bias;
            out[BLOCK * g + i] = (float)q * s;
        }
    }
}

int orc_encode_f32(int bits, const float *x, size_t n, uint8_t *wire)
{
    if (!bits_ok(bits)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? x[idx] : 0.0f; /* tail: zero padding */
        }
        if (encode_tile(bits, buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_encode(int bits, int dtype, const uint16_t *x, size_t n, uint8_t *wire)
{
    if (!bits_ok(bits) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? widen(dtype, x[idx]) : 0.0f;
        }
        if (encode_tile(bits, buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_decode_f32(int bits, const uint8_t *wire, size_t n, float *out)
{
    if (!bits_ok(bits)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        decode_tile_f32(bits, wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i) out[t * TILE + i] = buf[i];
    }
    return 0;
}

int orc_decode(int bits, int dtype, const uint8_t *wire, size_t n, uint16_t *y)
{
    if (!bits_ok(bits) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        decode_tile_f32(bits, wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i)
            y[t * TILE + i] = narrow(dtype, buf[i]); /* round half to even */
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Two-shot reduction [QR Quantization and Dequantization Paths: Phase-1B;   */
/* FC key machinery: sum locally, re-quantize the partial sums]              */
/* ------------------------------------------------------------------------ */

/* Phase-1B: decode the R rank copies of each tile, add them in fp32 in rank
 * order 0..R-1 (each add rounded to fp32), re-quantize the sums. */
int orc_segment_reduce(int bits, int R, const uint8_t *const *wires, size_t n,
                       uint8_t *out_wire)
{
    if (!bits_ok(bits) || R < 1) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_tile_bytes(bits);
    float acc[TILE], y[TILE];
    for (size_t t = 0; t < T; ++t) {
        decode_tile_f32(bits, wires[0] + t * tb, acc);
        for (int r = 1; r < R; ++r) {
            decode_tile_f32(bits, wires[r] + t * tb, y);
            for (int i = 0; i < TILE; ++i) acc[i] = acc[i] + y[i];
        }
        if (encode_tile(bits, acc, out_wire + t * tb) != 0) return -1;
    }
    return 0;
}

/* The whole two-shot all-reduce: quantize every rank (send), Phase-1B
 * reduction with re-quantization, Phase-2 dequantization of the reduced
 * wire.  Two quantization round trips in total [FC key machinery]. */
int orc_allreduce(int bits, int dtype, int R, const uint16_t *const *x,
                  size_t n, uint16_t *y)
{
    if (!bits_ok(bits) || R < 1 || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t W = orc_wire_bytes(bits, n);
    int rc = -1;
    uint8_t **wires = (uint8_t **)calloc((size_t)R, sizeof *wires);
    uint8_t *red = (uint8_t *)malloc(W ? W : 1);
    if (!wires || !red) goto done;
    for (int r = 0; r < R; ++r) {
        wires[r] = (uint8_t *)malloc(W ? W : 1);
        if (!wires[r]) goto done;
        if (orc_encode(bits, dtype, x[r], n, wires[r]) != 0) goto done;
    }
    if (orc_segment_reduce(bits, R, (const uint8_t *const *)wires, n, red) != 0) goto done;
    rc = orc_decode(bits, dtype, red, n, y);
done:
    if (wires)
        for (int r = 0; r < R; ++r) free(wires[r]);
    free(wires);
    free(red);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* The Flash Communication codec: asymmetric quantization in groups of 128   */
/* [FC key machinery "asymmetric group-128 scaling"; pith summary "group     */
/* size 128", "INT4 for the reduce stage and INT8 for the gather stage";     */
/* minor comments on "INT6" and Algorithm 1's Dequantize(M_q, z, s)].        */
/* ------------------------------------------------------------------------ */

#define FC_GROUP 128
#define FC_NGROUP (TILE / FC_GROUP)

static int fc_bits_ok(int bits) { return bits == 4 || bits == 8; }

size_t orc_fc_tile_bytes(int bits)
{
    return fc_bits_ok(bits) ? (size_t)256 * (size_t)bits + 128 : 0;
}

size_t orc_fc_wire_bytes(int bits, size_t n)
{
    return ((n + TILE - 1) / TILE) * orc_fc_tile_bytes(bits);
}

static void put_f32(uint8_t *p, float f)
{
    uint32_t v;
    memcpy(&v, &f, sizeof v);
    put_u32(p, v);
}

static float get_f32(const uint8_t *p)
{
    uint32_t v = get_u32(p);
    float f;
    memcpy(&f, &v, sizeof f);
    return f;
}

/* One group of 128 values: zero point = minimum, scale = range / (2^b - 1),
 * codes = nearest integer of (x - z) / s, ties to even, at most 2^b - 1. */
int orc_fc_quantize_group(int bits, const float *x, uint8_t *u, float *scale, float *zero)
{
    if (!fc_bits_ok(bits)) return -1;
    const int umax = (1 << bits) - 1;
    float lo = x[0], hi = x[0];
    int i;
    for (i = 0; i < FC_GROUP; ++i) {
        if (!isfinite(x[i])) return -1;
        if (x[i] < lo) lo = x[i];
        if (x[i] > hi) hi = x[i];
    }
    float range = hi - lo;
    if (!isfinite(range)) return -1; /* a range beyond fp32 is outside the contract */
    float s = range / (float)umax;
    if (!(s >= 0x1p-126f)) s = 0.0f; /* zero or subnormal: every code 0 */
    /* The zero point is the minimum as a value: -0 and +0 are the same value,
     * and a zero minimum is stored as +0 (lo + 0 turns -0 into +0 and leaves
     * every other value unchanged). */
    float z = lo + 0.0f;
    *zero = z;
    *scale = s;
    if (s == 0.0f) {
        for (i = 0; i < FC_GROUP; ++i) u[i] = 0;
        return 0;
    }
    float r = 1.0f / s;
    for (i = 0; i < FC_GROUP; ++i) {
        /* the nearest integer (ties to even) to the exact product (x - z) * r;
         * a double holds the product of two floats exactly */
        float d = x[i] - z;
        double t = (double)d * (double)r; /* >= 0 */
        double fl = floor(t), frac = t - fl;
        double q = frac > 0.5 ? fl + 1.0 : frac < 0.5 ? fl : (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);
        if (q > (double)umax) q = (double)umax;
        u[i] = (uint8_t)q;
    }
    return 0;
}

static int fc_encode_tile(int bits, const float *x, uint8_t *tile)
{
    uint8_t u[TILE];
    const size_t meta = (size_t)256 * (size_t)bits;
    for (int g = 0; g < FC_NGROUP; ++g) {
        float s, z;
        if (orc_fc_quantize_group(bits, x + FC_GROUP * g, u + FC_GROUP * g, &s, &z) != 0) return -1;
        put_f32(tile + meta + 4 * (size_t)g, s);
        put_f32(tile + meta + 64 + 4 * (size_t)g, z);
    }
    for (int k = 0; k < NSLOT; ++k) pack_slot(bits, u + 8 * k, tile, k);
    return 0;
}

/* decode = u*s + z with one rounding */
static void fc_decode_tile_f32(int bits, const uint8_t *tile, float *out)
{
    uint8_t u[TILE];
    const size_t meta = (size_t)256 * (size_t)bits;
    for (int k = 0; k < NSLOT; ++k) unpack_slot(bits, tile, k, u + 8 * k);
    for (int g = 0; g < FC_NGROUP; ++g) {
        float s = get_f32(tile + meta + 4 * (size_t)g);
        float z = get_f32(tile + meta + 64 + 4 * (size_t)g);
        for (int i = 0; i < FC_GROUP; ++i) out[FC_GROUP * g + i] = fmaf((float)u[FC_GROUP * g + i], s, z);
    }
}

int orc_fc_encode_f32(int bits, const float *x, size_t n, uint8_t *wire)
{
    if (!fc_bits_ok(bits)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? x[idx] : 0.0f;
        }
        if (fc_encode_tile(bits, buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_fc_encode(int bits, int dtype, const uint16_t *x, size_t n, uint8_t *wire)
{
    if (!fc_bits_ok(bits) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? widen(dtype, x[idx]) : 0.0f;
        }
        if (fc_encode_tile(bits, buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_fc_decode_f32(int bits, const uint8_t *wire, size_t n, float *out)
{
    if (!fc_bits_ok(bits)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        fc_decode_tile_f32(bits, wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i) out[t * TILE + i] = buf[i];
    }
    return 0;
}

int orc_fc_decode(int bits, int dtype, const uint8_t *wire, size_t n, uint16_t *y)
{
    if (!fc_bits_ok(bits) || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fc_tile_bytes(bits);
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        fc_decode_tile_f32(bits, wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i) y[t * TILE + i] = narrow(dtype, buf[i]);
    }
    return 0;
}

/* Phase-1B: decode the R rank copies (bits_in), add in fp32 in rank order,
 * re-quantize the sums (bits_out: 8 for the pages' "INT6" mixed scheme).
 * Values at or past n are zero in every phase: an asymmetric code does not
 * decode a padded zero back to exactly 0, so the sums there are set to 0
 * again before re-quantization. */
int orc_fc_segment_reduce(int bits_in, int bits_out, int R, const uint8_t *const *wires,
                          size_t n, uint8_t *out_wire)
{
    if (!fc_bits_ok(bits_in) || !fc_bits_ok(bits_out) || R < 1) return -1;
    size_t T = (n + TILE - 1) / TILE;
    size_t tbi = orc_fc_tile_bytes(bits_in), tbo = orc_fc_tile_bytes(bits_out);
    float acc[TILE], y[TILE];
    for (size_t t = 0; t < T; ++t) {
        fc_decode_tile_f32(bits_in, wires[0] + t * tbi, acc);
        for (int r = 1; r < R; ++r) {
            fc_decode_tile_f32(bits_in, wires[r] + t * tbi, y);
            for (int i = 0; i < TILE; ++i) acc[i] = acc[i] + y[i];
        }
        for (size_t i = 0; i < TILE; ++i)
            if (t * TILE + i >= n) acc[i] = 0.0f;
        if (fc_encode_tile(bits_out, acc, out_wire + t * tbo) != 0) return -1;
    }
    return 0;
}

/* quantize (bits_rs) -> all-to-all -> local sum -> re-quantize (bits_ag) ->
 * all-gather -> dequantize: two quantization round trips. */
int orc_fc_allreduce(int bits_rs, int bits_ag, int dtype, int R, const uint16_t *const *x,
                     size_t n, uint16_t *y)
{
    if (!fc_bits_ok(bits_rs) || !fc_bits_ok(bits_ag) || R < 1 ||
        (dtype != ORC_FP16 && dtype != ORC_BF16))
        return -1;
    size_t W = orc_fc_wire_bytes(bits_rs, n), W2 = orc_fc_wire_bytes(bits_ag, n);
    int rc = -1;
    uint8_t **wires = (uint8_t **)calloc((size_t)R, sizeof *wires);
    uint8_t *red = (uint8_t *)malloc(W2 ? W2 : 1);
    if (!wires || !red) goto done;
    for (int r = 0; r < R; ++r) {
        wires[r] = (uint8_t *)malloc(W ? W : 1);
        if (!wires[r]) goto done;
        if (orc_fc_encode(bits_rs, dtype, x[r], n, wires[r]) != 0) goto done;
    }
    if (orc_fc_segment_reduce(bits_rs, bits_ag, R, (const uint8_t *const *)wires, n, red) != 0) goto done;
    rc = orc_fc_decode(bits_ag, dtype, red, n, y);
done:
    if (wires)
        for (int r = 0; r < R; ++r) free(wires[r]);
    free(wires);
    free(red);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* The FP4 codec [QR introduction: a hardware-accelerated FP4 quantization   */
/* path on MI355, "FP4 and INT4 are essentially interchangeable"]: the INT4  */
/* block framework with E2M1 elements in place of the biased integers.      */
/* ------------------------------------------------------------------------ */

/* The E2M1 magnitudes by code (bits 0..2; bit 3 is the sign): exponent bits
 * 1..2 with bias 1, one mantissa bit, code 1 subnormal. */
static const float FP4_GRID[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_fp4_value(uint8_t code)
{
    float v = FP4_GRID[code & 7u];
    return (code & 8u) ? -v : v;
}

/* Nearest E2M1 value to t: at or beyond 6 that is 6 (saturation); below,
 * the grid magnitude closest to |t| (the distances of a float below 6 to
 * the grid are exact in double wherever two of them can be equal), a tie
 * going to the even code (mantissa bit 0).  The sign bit is t's sign, so a
 * negative t that rounds to zero gives code 8 (-0). */
uint8_t orc_fp4_round(float t)
{
    double a = fabs((double)t);
    int best = 7;
    if (a < 6.0) {
        double dbest = a;
        best = 0;
        for (int m = 1; m < 8; ++m) {
            double dm = fabs(a - (double)FP4_GRID[m]);
            if (dm < dbest || (dm == dbest && (m & 1) == 0 && (best & 1) != 0)) {
                best = m;
                dbest = dm;
            }
        }
    }
    return (uint8_t)((signbit(t) ? 8 : 0) | best);
}

void orc_fp4_round_n(const float *t, size_t n, uint8_t *code)
{
    for (size_t i = 0; i < n; ++i) code[i] = orc_fp4_round(t[i]);
}

/* One block of 32: A = max|x|; d = fp32_RN(A / 6) (6, the largest E2M1
 * magnitude, plays the role of |qmin|); s = fp16_RNE(d), saturated at
 * 65504; s == 0 stores +0 and every code is 0; r = fp32_RN(1/s);
 * code = orc_fp4_round(fp32_RN(x * r)). */
int orc_fp4_quantize_block(const float *x, uint8_t *code, uint16_t *scale)
{
    int i;
    float A = 0.0f;
    for (i = 0; i < BLOCK; ++i) {
        if (!isfinite(x[i])) return -1;
        float a = fabsf(x[i]);
        if (a > A) A = a;
    }
    float d = A / 6.0f; /* IEEE fp32 division, rounded to nearest even */
    uint16_t sh = orc_f32_to_f16(d);
    if (sh == 0x7C00u) sh = 0x7BFFu;
    float s = orc_f16_to_f32(sh);
    if (s == 0.0f) {
        *scale = 0;
        for (i = 0; i < BLOCK; ++i) code[i] = 0;
        return 0;
    }
    float r = 1.0f / s;
    for (i = 0; i < BLOCK; ++i) {
        float t = x[i] * r;
        code[i] = orc_fp4_round(t);
    }
    *scale = sh;
    return 0;
}

/* Tile: the INT4 layout (nibble of lane j at bits 4j of the u32 at 4k, 64
 * fp16 scales at 1024): 1152 bytes. */
size_t orc_fp4_tile_bytes(void) { return orc_tile_bytes(4); }
size_t orc_fp4_wire_bytes(size_t n) { return orc_wire_bytes(4, n); }

static int fp4_encode_tile(const float *x, uint8_t *tile)
{
    uint8_t c[TILE];
    for (int g = 0; g < NBLOCK; ++g) {
        uint16_t sh;
        if (orc_fp4_quantize_block(x + BLOCK * g, c + BLOCK * g, &sh) != 0) return -1;
        put_u16(tile + scale_offset(4) + 2 * (size_t)g, sh);
    }
    for (int k = 0; k < NSLOT; ++k) pack_slot(4, c + 8 * k, tile, k);
    return 0;
}

/* value(code) * s is exact in fp32: at most 2 significant bits times an
 * 11-bit significand. */
static void fp4_decode_tile_f32(const uint8_t *tile, float *out)
{
    uint8_t c[TILE];
    for (int k = 0; k < NSLOT; ++k) unpack_slot(4, tile, k, c + 8 * k);
    for (int g = 0; g < NBLOCK; ++g) {
        float s = orc_f16_to_f32((uint16_t)get_u16(tile + scale_offset(4) + 2 * (size_t)g));
        for (int i = 0; i < BLOCK; ++i) out[BLOCK * g + i] = orc_fp4_value(c[BLOCK * g + i]) * s;
    }
}

int orc_fp4_encode_f32(const float *x, size_t n, uint8_t *wire)
{
    size_t T = (n + TILE - 1) / TILE, tb = orc_fp4_tile_bytes();
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? x[idx] : 0.0f;
        }
        if (fp4_encode_tile(buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_fp4_encode(int dtype, const uint16_t *x, size_t n, uint8_t *wire)
{
    if (dtype != ORC_FP16 && dtype != ORC_BF16) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fp4_tile_bytes();
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        for (size_t i = 0; i < TILE; ++i) {
            size_t idx = t * TILE + i;
            buf[i] = idx < n ? widen(dtype, x[idx]) : 0.0f;
        }
        if (fp4_encode_tile(buf, wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_fp4_decode_f32(const uint8_t *wire, size_t n, float *out)
{
    size_t T = (n + TILE - 1) / TILE, tb = orc_fp4_tile_bytes();
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        fp4_decode_tile_f32(wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i) out[t * TILE + i] = buf[i];
    }
    return 0;
}

int orc_fp4_decode(int dtype, const uint8_t *wire, size_t n, uint16_t *y)
{
    if (dtype != ORC_FP16 && dtype != ORC_BF16) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fp4_tile_bytes();
    float buf[TILE];
    for (size_t t = 0; t < T; ++t) {
        fp4_decode_tile_f32(wire + t * tb, buf);
        for (size_t i = 0; i < TILE && t * TILE + i < n; ++i) y[t * TILE + i] = narrow(dtype, buf[i]);
    }
    return 0;
}

/* Phase-1B as for the integer codes: decode the R copies, add in fp32 in rank
 * order, re-quantize. */
int orc_fp4_segment_reduce(int R, const uint8_t *const *wires, size_t n, uint8_t *out_wire)
{
    if (R < 1) return -1;
    size_t T = (n + TILE - 1) / TILE, tb = orc_fp4_tile_bytes();
    float acc[TILE], y[TILE];
    for (size_t t = 0; t < T; ++t) {
        fp4_decode_tile_f32(wires[0] + t * tb, acc);
        for (int r = 1; r < R; ++r) {
            fp4_decode_tile_f32(wires[r] + t * tb, y);
            for (int i = 0; i < TILE; ++i) acc[i] = acc[i] + y[i];
        }
        if (fp4_encode_tile(acc, out_wire + t * tb) != 0) return -1;
    }
    return 0;
}

int orc_fp4_allreduce(int dtype, int R, const uint16_t *const *x, size_t n, uint16_t *y)
{
    if (R < 1 || (dtype != ORC_FP16 && dtype != ORC_BF16)) return -1;
    size_t W = orc_fp4_wire_bytes(n);
    int rc = -1;
    uint8_t **wires = (uint8_t **)calloc((size_t)R, sizeof *wires);
    uint8_t *red = (uint8_t *)malloc(W ? W : 1);
    if (!wires || !red) goto done;
    for (int r = 0; r < R; ++r) {
        wires[r] = (uint8_t *)malloc(W ? W : 1);
        if (!wires[r]) goto done;
        if (orc_fp4_encode(dtype, x[r], n, wires[r]) != 0) goto done;
    }
    if (orc_fp4_segment_reduce(R, (const uint8_t *const *)wires, n, red) != 0) goto done;
    rc = orc_fp4_decode(dtype, red, n, y);
done:
    if (wires)
        for (int r = 0; r < R; ++r) free(wires[r]);
    free(wires);
    free(red);
    return rc;
}
