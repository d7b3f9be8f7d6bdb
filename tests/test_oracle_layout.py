"""Pins of the oracle's wire layout.

- Tile sizes: 1152 B (INT4) and 896 B (INT3), about 22% smaller, as printed in
  "QuickReduce INT3 quantization and benchmarking on MI355", Design Highlights.
- INT3 q2w/q1w split: brute force over all 8^8 code patterns of one slot.
- Per-lane exhaustive round trips for INT4 / INT6 / INT8.
- Hand-built known-answer tiles (tests/golden/known_answer_tiles.json) whose
  expected bytes were worked out by hand from the layout and the page's facts.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "known_answer_tiles.json")


def test_tile_sizes_printed_on_the_page(orc):
    assert orc.tile_values() == 2048
    assert orc.tile_bytes(4) == 1152
    assert orc.tile_bytes(3) == 896
    # "a reduction of about 22%"
    assert abs((1 - 896 / 1152) - 0.22) < 0.005
    # the same block framework for the other widths: codes + 64 fp16 scales
    assert orc.tile_bytes(8) == 2048 + 128
    assert orc.tile_bytes(6) == 1536 + 128
    assert orc.tile_bytes(5) == 0 and orc.tile_bytes(2) == 0
    for b in (3, 4, 6, 8):
        assert orc.tile_bytes(b) % 16 == 0
        assert orc.wire_bytes(b, 1) == orc.tile_bytes(b)
        assert orc.wire_bytes(b, 2048) == orc.tile_bytes(b)
        assert orc.wire_bytes(b, 2049) == 2 * orc.tile_bytes(b)
        assert orc.wire_bytes(b, 2048 * 7 + 37) == 8 * orc.tile_bytes(b)


def test_int3_brute_force_every_slot_pattern(orc):
    """All 8^8 = 16,777,216 code patterns of one 8-value slot pack into
    (q2w, q1w) and unpack to the same codes; the packing is injective."""
    p = np.arange(8**8, dtype=np.uint32)
    codes = np.empty((8**8, 8), np.uint8)
    for j in range(8):
        codes[:, j] = (p >> (3 * j)) & 7
    wire = orc.pack_codes(3, codes.reshape(-1))
    back = orc.unpack_codes(3, wire).reshape(-1, 8)
    assert np.array_equal(back, codes)
    assert back.max() <= 7  # [0, 7] after biasing
    tiles = wire.reshape(-1, 896)
    q2w = tiles[:, :512].reshape(-1, 256, 2).astype(np.uint32)
    q2w = (q2w[..., 0] | (q2w[..., 1] << 8)).reshape(-1)
    q1w = tiles[:, 512:768].reshape(-1).astype(np.uint32)
    key = q2w | (q1w << 16)
    assert np.unique(key).size == 8**8
    # the low two bits all live in q2w, the high bit in q1w
    assert np.array_equal((q2w >> 0) & 3, codes[:, 0] & 3)
    assert np.array_equal(q1w & 1, codes[:, 0] >> 2)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_every_code_in_every_lane(orc, bits):
    """Each code value in each lane position, with random neighbours."""
    rng = np.random.Generator(np.random.PCG64(bits))
    ncode = 1 << bits
    u = rng.integers(0, ncode, size=(ncode * 8, 2048), dtype=np.uint8)
    for c in range(ncode):
        for j in range(8):
            u[c * 8 + j, j::8] = c
    u = u.reshape(-1)
    w = orc.pack_codes(bits, u)
    assert np.array_equal(orc.unpack_codes(bits, w), u)


@pytest.mark.parametrize("bits", [3, 4, 6, 8])
def test_codes_land_in_their_sections(orc, bits):
    """Packing touches only the code section(s); the 128-byte scale section
    at the end of the tile stays as it was."""
    rng = np.random.Generator(np.random.PCG64(100 + bits))
    u = rng.integers(0, 1 << bits, size=3 * 2048, dtype=np.uint8)
    w = orc.pack_codes(bits, u).reshape(3, -1)
    assert np.all(w[:, 256 * bits:] == 0)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("dtype", [0, 1], ids=["fp16", "bf16"])
def test_known_answer_tiles(orc, case, dtype):
    bits = case["bits"]
    bias = 1 << (bits - 1)
    x = np.zeros(2048, np.float32)
    if "slot_codes" in case:
        s = case["scale"]
        u = np.full(32, case["fill_code"], np.int32)
        for k, codes in case["slot_codes"].items():
            u[8 * int(k): 8 * int(k) + 8] = codes
        x[:32] = (u - bias) * s
        expect_dec = x.copy()
    elif "values_block0" in case:
        v = case["values_block0"]
        x[: len(v)] = v
        expect_dec = np.zeros(2048, np.float32)
        expect_dec[: len(v)] = case["expect_decoded"]
    else:
        x[:32] = case["values_block0_all"]
        expect_dec = np.zeros(2048, np.float32)
        expect_dec[:32] = case["expect_decoded_all"]
    xin = orc.narrow(dtype, x)
    assert np.array_equal(orc.widen(dtype, xin), x)  # every value is exact in both formats
    wire = orc.encode(bits, dtype, xin)
    assert wire.size == orc.tile_bytes(bits)
    for off, hexstr in case["expect_hex"].items():
        off = int(off)
        got = wire[off: off + len(hexstr) // 2].tobytes().hex()
        assert got == hexstr, f"{case['name']} bytes at {off}: {got} != {hexstr}"
    assert np.array_equal(orc.decode_f32(bits, wire, 2048), expect_dec)
    assert np.array_equal(orc.decode(bits, dtype, wire, 2048), orc.narrow(dtype, expect_dec))
