/*
 * qr_oracle.h -- slow, scalar CPU oracle for the block-quantized two-shot
 * all-reduce codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline / reference arm use it.  It shares no code,
 * header, table or constant with the CUDA library under
 * bit_quantized_all_gb300/csrc.
 *
 * What it computes, and where that is stated:
 *   - "QuickReduce INT3 quantization and benchmarking on MI355" (AMD blog),
 *     section "Design Highlights": blocks of 32 fp16/bf16 values share one
 *     fp16 scale; values are scaled, clipped to a symmetric range ([-4,+3] for
 *     INT3), rounded and biased to unsigned ([0,7]); INT4 packs eight 4-bit
 *     codes per int32; INT3 splits each code into a low-2-bit part (one
 *     uint16 "q2w" per thread slot) and a high bit (one uint8 "q1w" per slot);
 *     the per-rank tile is 1152 B (INT4) or 896 B (INT3).
 *   - same page, section "Quantization and Dequantization Paths": the send
 *     path takes the block absmax, derives the fp16 scale, scales / clips /
 *     rounds / biases, splits the bits and writes the scale; the receive path
 *     recombines the bits, removes the bias and multiplies by the scale.  The
 *     two-shot kernel uses the receive path in Phase-1B (in-segment
 *     reduction) and Phase-2 (gather).
 *   - "Flash Communication" review record (arXiv 2412.04964), key machinery:
 *     quantize, one all-to-all, local sum, re-quantize the partial sums, one
 *     all-gather, dequantize -- two quantization round trips in total.
 *
 * Conventions the pages leave open (each one is the plainest reading the
 * rest supports):
 *   - decode scale s = fp16_RNE(absmax / |qmin|); an fp16 overflow saturates
 *     to 65504; s == 0 (zero block or fp16 underflow) stores +0 and every code
 *     of the block is the bias;
 *   - encode factor r = fp32_RN(1/s); t = fp32_RN(x * r); clip t to
 *     [qmin, qmax]; round half to even; u = q + bias;
 *   - Phase-1B sums the decoded rank values in fp32, in rank order 0..R-1,
 *     and re-quantizes the fp32 sums with the same block rule;
 *   - tails are zero-padded to whole 2048-value tiles; decode writes only n;
 *   - wire layout of one tile (little-endian), slot k = values 8k..8k+7,
 *     lane j = value 8k+j, block g = values 32g..32g+31:
 *       INT8: byte 8k+j = u;                         scales at 2048
 *       INT6: u32 at 4k, bits 4j..4j+3 = u & 15;     u16 at 1024+2k,
 *             bits 2j..2j+1 = u >> 4;                scales at 1536
 *       INT4: u32 at 4k, bits 4j..4j+3 = u;          scales at 1024
 *       INT3: u16 at 2k, bits 2j..2j+1 = u & 3;      u8 at 512+k,
 *             bit j = u >> 2;                        scales at 768
 *     the scale of block g is the fp16 at (scale offset) + 2g.
 *
 * Parity pins: every function here is checked by the CPU test suite against
 * facts the pages print (tile sizes, ranges), hand-built known-answer tiles,
 * closed forms, brute force and error bounds.  The end-to-end pipeline has
 * no worked numeric example on the pages, so parity with the pages' own
 * implementation is unpinned beyond those invariants.
 */
#ifndef QR_ORACLE_H
#define QR_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_FP16 0
#define ORC_BF16 1

/* ---- number formats (IEEE-754 binary16 and bfloat16, round-half-even) ---- */
uint16_t orc_f32_to_f16(float f);
float    orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
float    orc_bf16_to_f32(uint16_t h);
/* the same conversions over arrays */
void orc_f32_to_f16_n(const float *f, size_t n, uint16_t *h);
void orc_f16_to_f32_n(const uint16_t *h, size_t n, float *f);
void orc_f32_to_bf16_n(const float *f, size_t n, uint16_t *h);
void orc_bf16_to_f32_n(const uint16_t *h, size_t n, float *f);

/* ---- sizes ---- */
size_t orc_tile_values(void);                 /* 2048 */
size_t orc_tile_bytes(int bits);              /* 256*bits + 128, 0 if unsupported */
size_t orc_wire_bytes(int bits, size_t n);    /* ceil(n/2048) * tile_bytes */

/* ---- code packing of whole tiles (no quantization) ----
 * u: 2048 codes per tile (values 0..2^bits-1), ntiles tiles back to back.
 * Writes / reads only the code section(s) of each tile. */
int orc_pack_codes(int bits, const uint8_t *u, size_t ntiles, uint8_t *wire);
int orc_unpack_codes(int bits, const uint8_t *wire, size_t ntiles, uint8_t *u);

/* ---- one 32-value block: the quantizer itself ----
 * x: 32 fp32 values.  Writes 32 codes and the fp16 scale bits. */
int orc_quantize_block(int bits, const float *x, uint8_t *u, uint16_t *scale);

/* ---- the codec (return 0 on success, -1 on bad arguments) ---- */
int orc_encode_f32(int bits, const float *x, size_t n, uint8_t *wire);
int orc_encode(int bits, int dtype, const uint16_t *x, size_t n, uint8_t *wire);
int orc_decode_f32(int bits, const uint8_t *wire, size_t n, float *out);
int orc_decode(int bits, int dtype, const uint8_t *wire, size_t n, uint16_t *y);
int orc_segment_reduce(int bits, int R, const uint8_t *const *wires, size_t n,
                       uint8_t *out_wire);
int orc_allreduce(int bits, int dtype, int R, const uint16_t *const *x,
                  size_t n, uint16_t *y);

/* ---- the Flash Communication codec (asymmetric, groups of 128) ----------
 * "Flash Communication" review record (arXiv 2412.04964): activations are
 * quantized "with asymmetric group-128 scaling" to 4-8 bits, exchanged,
 * summed locally, "re-quantizes the partial sums to INT8", all-gathered and
 * dequantized; "INT6" names the mixed scheme INT4 for the reduce-scatter and
 * INT8 for the all-gather; Algorithm 1 dequantizes from the codes, a zero
 * point z and a scale s.  Readings (the pages fix no more than that):
 *   per group of 128: lo = min x, hi = max x (fp32, exact);
 *   s = fp32_RN(fp32_RN(hi - lo) / (2^b - 1));  z = lo (a zero minimum, of
 *   either sign, stored as +0);
 *   s below 2^-126 (zero or subnormal) is stored as 0 and every code is 0;
 *   r = fp32_RN(1/s);  u = min(RNE(fp32_RN(x - z) * r), 2^b - 1), the
 *   product taken exactly (the nearest integer to it, one rounding);
 *   decode = fp32_RN(u*s + z) (one rounding, a fused multiply-add);
 *   Phase-1B: acc = decode_0, acc = fp32_RN(acc + decode_r), r = 1..R-1;
 *   values at or past n are zero in every phase (Phase-1B sets the sums
 *   there back to 0: a padded zero does not decode to exactly 0);
 *   s and z are stored as fp32 (every fp16/bf16 input and every fp32 partial
 *   sum fits); b is 4 or 8.
 * Tile of 2048 values = 16 groups: codes as in the symmetric codec (INT4
 * nibbles lane j at bits 4j of the u32 at 4k; INT8 bytes), then 16 fp32
 * scales at 256*b, then 16 fp32 zero points at 256*b + 64: 256*b + 128 bytes.
 */
size_t orc_fc_tile_bytes(int bits);           /* 256*bits + 128, 0 unless bits is 4 or 8 */
size_t orc_fc_wire_bytes(int bits, size_t n);
int orc_fc_quantize_group(int bits, const float *x, uint8_t *u, float *scale, float *zero);
int orc_fc_encode_f32(int bits, const float *x, size_t n, uint8_t *wire);
int orc_fc_encode(int bits, int dtype, const uint16_t *x, size_t n, uint8_t *wire);
int orc_fc_decode_f32(int bits, const uint8_t *wire, size_t n, float *out);
int orc_fc_decode(int bits, int dtype, const uint8_t *wire, size_t n, uint16_t *y);
int orc_fc_segment_reduce(int bits_in, int bits_out, int R, const uint8_t *const *wires,
                          size_t n, uint8_t *out_wire);
int orc_fc_allreduce(int bits_rs, int bits_ag, int dtype, int R, const uint16_t *const *x,
                     size_t n, uint16_t *y);

/* ---- the FP4 codec --------------------------------------------------------
 * "QuickReduce INT3 quantization and benchmarking on MI355", introduction: a
 * hardware-accelerated FP4 quantization path on MI355, with FP4 and INT4
 * "essentially interchangeable".  The pages give no format; the reading
 * here keeps the INT4 block framework and tile (32 values per fp16 scale,
 * nibble of lane j at bits 4j, 1152-byte tiles) with E2M1 elements (sign,
 * 2 exponent bits with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6) in place of the biased integers:
 *   A = max|x|; d = fp32_RN(A / 6); s = fp16_RNE(d) saturated at 65504;
 *   s == 0 stores +0 and every code is 0; r = fp32_RN(1/s);
 *   code = nearest E2M1 value to fp32_RN(x * r), ties to the even code,
 *   saturating at +-6, the sign bit taken from the product (-0 possible);
 *   decode = value(code) * s (exact in fp32);
 *   Phase-1B and Phase-2 as for the integer codes.
 * The pins check this reading (element rounding against an independent
 * E2M1 implementation, the scale against torch, closed forms); parity with
 * the pages' own FP4 path is unpinned, since the pages give no format.
 */
float   orc_fp4_value(uint8_t code);
uint8_t orc_fp4_round(float t);
void    orc_fp4_round_n(const float *t, size_t n, uint8_t *code);
size_t  orc_fp4_tile_bytes(void);              /* 1152 */
size_t  orc_fp4_wire_bytes(size_t n);
int orc_fp4_quantize_block(const float *x, uint8_t *code, uint16_t *scale);
int orc_fp4_encode_f32(const float *x, size_t n, uint8_t *wire);
int orc_fp4_encode(int dtype, const uint16_t *x, size_t n, uint8_t *wire);
int orc_fp4_decode_f32(const uint8_t *wire, size_t n, float *out);
int orc_fp4_decode(int dtype, const uint8_t *wire, size_t n, uint16_t *y);
int orc_fp4_segment_reduce(int R, const uint8_t *const *wires, size_t n, uint8_t *out_wire);
int orc_fp4_allreduce(int dtype, int R, const uint16_t *const *x, size_t n, uint16_t *y);

#ifdef __cplusplus
}
#endif
#endif /* QR_ORACLE_H */
