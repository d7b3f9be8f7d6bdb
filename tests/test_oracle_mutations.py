"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a temporary copy of the oracle's C
source (a dropped term, a wrong sign, index or offset, a transposed bit
order, the wrong rounding or denominator, ...), compiles it with gcc, and runs
the pin battery of the other oracle test modules against it: at least one pin
must fail.  Nothing here touches a GPU.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_formats as F
import test_oracle_layout as L
import test_oracle_quantizer as Q
import test_oracle_fc as FC
import test_oracle_reduce as Rd
import test_oracle_fp4 as P4

SRC = os.path.join(os.path.dirname(oracle.__file__), "qr_oracle.c")

# (name, [(old, new), ...]) -- every `old` must occur in the source; all
# occurrences are replaced.
MUTATIONS = [
    ("scale_over_qmax_not_qmin", [("float d = A / (float)bias;", "float d = A / (float)(bias - 1);")]),
    ("round_half_up_not_even",
     [("return (float)(fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);", "return (float)(fl + 1.0);")]),
    ("reduce_drops_rank0", [("decode_tile_f32(bits, wires[0] + t * tb, acc);", "memset(acc, 0, sizeof acc);")]),
    ("reduce_drops_last_rank", [("for (int r = 1; r < R; ++r) {", "for (int r = 1; r < R - 1; ++r) {")]),
    ("reduce_in_reverse_rank_order",
     [("decode_tile_f32(bits, wires[0] + t * tb, acc);", "decode_tile_f32(bits, wires[R - 1] + t * tb, acc);"),
      ("decode_tile_f32(bits, wires[r] + t * tb, y);", "decode_tile_f32(bits, wires[R - 1 - r] + t * tb, y);")]),
    ("decode_bias_sign_flipped",
     [("int q = (int)u[BLOCK * g + i] - bias;", "int q = bias - (int)u[BLOCK * g + i];")]),
    ("nibble_order_reversed", [("(4 * j)", "(4 * (7 - j))")]),
    ("q2w_order_reversed", [("(2 * j)", "(2 * (7 - j))")]),
    ("q1w_at_wrong_offset", [("512 + k", "520 + k")]),
    ("int6_high_bits_at_wrong_offset", [("1024 + 2 * k", "1026 + 2 * k")]),
    ("no_lower_clip", [("if (t < qmin) t = qmin;", "")]),
    ("no_upper_clip", [("if (t > qmax) t = qmax;", "")]),
    ("no_scale_saturation", [("if (sh == 0x7C00u) sh = 0x7BFFu;", "")]),
    ("absmax_without_abs", [("float a = fabsf(x[i]);", "float a = x[i];")]),
    ("fp16_rounds_ties_up", [("return (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0) * quantum;", "return (fl + 1.0) * quantum;")]),
    ("scales_after_a_gap", [("static size_t scale_offset(int bits) { return (size_t)256 * (size_t)bits; }",
                             "static size_t scale_offset(int bits) { return (size_t)256 * (size_t)bits + 2; }")]),
    ("tail_padded_with_ones", [("buf[i] = idx < n ? widen(dtype, x[idx]) : 0.0f;",
                                "buf[i] = idx < n ? widen(dtype, x[idx]) : 1.0f;")]),
    ("bf16_subnormal_quantum_wrong", [("ldexp(1.0, -133) : ldexp(1.0, E - 7)", "ldexp(1.0, -132) : ldexp(1.0, E - 7)")]),
    ("zero_scale_codes_not_bias", [("for (i = 0; i < BLOCK; ++i) u[i] = (uint8_t)bias;",
                                    "for (i = 0; i < BLOCK; ++i) u[i] = 0;")]),
    # the Flash Communication codec
    ("fc_zero_point_is_max", [("    float z = lo + 0.0f;", "    float z = hi + 0.0f;")]),
    ("fc_zero_point_sign_kept", [("    float z = lo + 0.0f;", "    float z = lo;")]),
    ("fc_scale_over_2b", [("float s = range / (float)umax;", "float s = range / (float)(umax + 1);")]),
    # (Removing the cap at 2^b - 1 is not a mistake the pins could catch: it
    # never fires, since t <= range * RN(1/RN(range/umax)) <= umax*(1+2^-24)^3
    # < umax + 1/2.)
    ("fc_decode_two_roundings", [("fmaf((float)u[FC_GROUP * g + i], s, z)", "(float)u[FC_GROUP * g + i] * s + z")]),
    ("fc_truncate_not_round", [("double q = frac > 0.5 ? fl + 1.0 : frac < 0.5 ? fl : (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);",
                                "double q = fl;")]),
    ("fc_product_rounded_to_fp32_first", [("double t = (double)d * (double)r; /* >= 0 */",
                                           "double t = (double)(d * r); /* >= 0 */")]),
    ("fc_reduce_drops_rank0", [("fc_decode_tile_f32(bits_in, wires[0] + t * tbi, acc);",
                                "memset(acc, 0, sizeof acc);")]),
    ("fc_reduce_reverse_order",
     [("fc_decode_tile_f32(bits_in, wires[0] + t * tbi, acc);",
       "fc_decode_tile_f32(bits_in, wires[R - 1] + t * tbi, acc);"),
      ("fc_decode_tile_f32(bits_in, wires[r] + t * tbi, y);",
       "fc_decode_tile_f32(bits_in, wires[R - 1 - r] + t * tbi, y);")]),
    ("fc_tail_not_repadded", [("            if (t * TILE + i >= n) acc[i] = 0.0f;", "            ;")]),
    ("fc_zero_points_at_wrong_offset", [("meta + 64 + 4 * (size_t)g", "meta + 60 + 4 * (size_t)g")]),
    ("fc_reduce_reencodes_at_input_width", [("if (fc_encode_tile(bits_out, acc, out_wire + t * tbo) != 0) return -1;",
                                             "if (fc_encode_tile(bits_in, acc, out_wire + t * tbo) != 0) return -1;")]),
    # the FP4 codec
    ("fp4_ties_to_odd", [("(dm == dbest && (m & 1) == 0 && (best & 1) != 0)", "(dm == dbest && (m & 1) != 0)")]),
    ("fp4_ties_away_from_zero", [("(dm == dbest && (m & 1) == 0 && (best & 1) != 0)", "(dm == dbest)")]),
    ("fp4_grid_4_read_as_5", [("{0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f}",
                               "{0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 5.0f, 6.0f}")]),
    ("fp4_no_saturation_branch", [("    if (a < 6.0) {\n        double dbest = a;", "    if (a < 1e38) {\n        double dbest = a;")]),
    ("fp4_sign_dropped", [("return (uint8_t)((signbit(t) ? 8 : 0) | best);", "return (uint8_t)best;")]),
    ("fp4_scale_over_4", [("float d = A / 6.0f;", "float d = A / 4.0f;")]),
    ("fp4_scale_not_saturated", [("    float d = A / 6.0f; /* IEEE fp32 division, rounded to nearest even */\n"
                                  "    uint16_t sh = orc_f32_to_f16(d);\n    if (sh == 0x7C00u) sh = 0x7BFFu;",
                                  "    float d = A / 6.0f; /* IEEE fp32 division, rounded to nearest even */\n"
                                  "    uint16_t sh = orc_f32_to_f16(d);")]),
    ("fp4_reduce_reverse_order",
     [("fp4_decode_tile_f32(wires[0] + t * tb, acc);", "fp4_decode_tile_f32(wires[R - 1] + t * tb, acc);"),
      ("fp4_decode_tile_f32(wires[r] + t * tb, y);", "fp4_decode_tile_f32(wires[R - 1 - r] + t * tb, y);")]),
]


def _battery(orc):
    golden = L._golden_cases()
    yield lambda: L.test_tile_sizes_printed_on_the_page(orc)
    for c in golden:
        for d in (0, 1):
            yield lambda c=c, d=d: L.test_known_answer_tiles(orc, c, d)
    for b in (3, 4, 6, 8):
        yield lambda b=b: Q.test_closed_form_all_equal_blocks(orc, b)
        yield lambda b=b: Q.test_zero_block(orc, b, 1)
        yield lambda b=b: Q.test_tail_is_zero_padded(orc, b, 0)
        yield lambda b=b: Q.test_scale_saturates_and_underflows_bf16(orc, b)
        yield lambda b=b: Rd.test_identical_ranks_scale_by_R(orc, b, 4, 1)
        yield lambda b=b: Rd.test_error_bound_against_exact_sum(orc, b, 3)
        yield lambda b=b: Q.test_codes_are_nearest_integers_clipped(orc, b)
        yield lambda b=b: Q.test_error_bound(orc, b)
    yield lambda: Q.test_int3_example_values(orc)
    yield lambda: Rd.test_sum_runs_in_rank_order(orc, 0)
    yield lambda: Rd.test_workload_c1_crafted_blocks(orc)
    yield lambda: F.test_f16_widen_every_pattern(orc)
    yield lambda: F.test_bf16_widen_every_pattern(orc)
    for fmt in ("f16", "bf16"):
        yield lambda fmt=fmt: F.test_narrow_ties_and_neighbours(orc, fmt)
        yield lambda fmt=fmt: F.test_narrow_roundtrips_every_value(orc, fmt)
    # the Flash Communication codec
    for c in FC._cases():
        for d in (0, 1):
            yield lambda c=c, d=d: FC.test_known_answer_tiles(orc, c, d)
    yield lambda: FC.test_decode_is_one_fused_rounding(orc)
    yield lambda: FC.test_zero_minimum_is_stored_as_plus_zero(orc)
    yield lambda: FC.test_code_is_nearest_integer_of_exact_product(orc)
    for b in (4, 8):
        yield lambda b=b: FC.test_constant_groups_are_exact(orc, b)
        yield lambda b=b: FC.test_min_decodes_exactly_and_codes_span_the_range(orc, b)
        yield lambda b=b: FC.test_codes_are_nearest_integers(orc, b)
        yield lambda b=b: FC.test_error_bound(orc, b)
        yield lambda b=b: FC.test_one_rank_and_mixed_widths(orc, b, 1)
        yield lambda b=b: FC.test_identical_ranks_on_exact_grids(orc, b, 4)
    yield lambda: FC.test_two_ranks_commute_and_rank_order(orc)
    for brs, bag in ((4, 8), (8, 8)):
        yield lambda brs=brs, bag=bag: FC.test_error_bound_against_exact_sum(orc, brs, bag, 3)
    # the FP4 codec
    yield lambda: P4.test_code_values_against_an_independent_decoder(orc)
    yield lambda: P4.test_ties_go_to_the_even_code(orc)
    yield lambda: P4.test_rounding_every_pattern_of_a_dense_range(orc)
    yield lambda: P4.test_rounding_random_patterns_of_every_magnitude(orc)
    yield lambda: P4.test_block_scale_against_torch(orc)
    yield lambda: P4.test_known_answer_block_and_layout(orc)
    yield lambda: P4.test_rank_order_is_the_order_of_the_fp32_adds(orc)
    for R in (2, 4):
        yield lambda R=R: P4.test_identical_ranks_on_exact_grids_scale_by_R(orc, R)


@pytest.mark.parametrize("name,edits", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert old in src, f"mutation {name}: {old!r} not in the oracle source"
        src = src.replace(old, new)
    c = tmp_path / "qr_oracle.c"
    c.write_text(src)
    hdr = os.path.join(os.path.dirname(SRC), "qr_oracle.h")
    (tmp_path / "qr_oracle.h").write_text(open(hdr).read())
    so = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    str(c), "-o", str(so), "-lm"], check=True, capture_output=True)
    caught = None
    with oracle.using_library(str(so)):
        for check in _battery(oracle):
            try:
                check()
            except (AssertionError, ValueError) as e:  # a pin failed
                caught = e
                break
    assert caught is not None, f"planted mistake {name!r} passed every pin"
