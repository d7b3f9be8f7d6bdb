"""The CUDA path against the hand-built known-answer tiles of tests/golden/,
with no oracle in between: the encode kernels' bytes at the hand-worked
offsets, the decode kernels' values, and for tiles whose blocks all hold
qmin, R identical ranks through the fused all-reduce giving exactly R * x
(the reduced scale is R * s, a power of two, so every code is unchanged).

Sources of the expected values: the tile layout and the facts of
"QuickReduce INT3 quantization and benchmarking on MI355" (Design
Highlights; Quantization and Dequantization Paths) and of the Flash
Communication review record (key machinery: asymmetric group-128 scaling),
as worked out by hand in the fixtures.
"""
import json
import os

import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr

pytestmark = pytest.mark.gpu

HERE = os.path.join(os.path.dirname(__file__), "golden")
TORCH_DT = {0: torch.float16, 1: torch.bfloat16}


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)["cases"]


def _to_dev(x: np.ndarray, dtype: int) -> torch.Tensor:
    t = torch.from_numpy(x.astype(np.float32)).to(TORCH_DT[dtype])
    assert torch.equal(t.float(), torch.from_numpy(x.astype(np.float32))), "fixture value not exact in the format"
    return t.cuda()


def _bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_bytes(wire: torch.Tensor, expect_hex: dict, what: str):
    w = wire.cpu().numpy()
    for off, hexstr in expect_hex.items():
        off = int(off)
        got = w[off: off + len(hexstr) // 2].tobytes().hex()
        assert got == hexstr, f"{what}: bytes at {off}: {got} != {hexstr}"


def _symmetric_case(case):
    """Inputs and the expected decoded values of one symmetric-codec case
    (the same construction as the fixture's description)."""
    bits = case["bits"]
    bias = 1 << (bits - 1)
    x = np.zeros(2048, np.float32)
    if "slot_codes" in case:
        u = np.full(32, case["fill_code"], np.int32)
        for k, codes in case["slot_codes"].items():
            u[8 * int(k): 8 * int(k) + 8] = codes
        x[:32] = (u - bias) * case["scale"]
        return x, x.copy()
    expect = np.zeros(2048, np.float32)
    if "values_block0" in case:
        v = case["values_block0"]
        x[: len(v)] = v
        expect[: len(v)] = case["expect_decoded"]
    else:
        x[:32] = case["values_block0_all"]
        expect[:32] = case["expect_decoded_all"]
    return x, expect


SYM = _load("known_answer_tiles.json")
FC = _load("fc_known_answer_tiles.json")


@pytest.mark.parametrize("case", SYM, ids=lambda c: c["name"])
@pytest.mark.parametrize("dtype", [0, 1], ids=["fp16", "bf16"])
def test_encode_decode_known_answer_tiles(case, dtype):
    bits = case["bits"]
    x, expect = _symmetric_case(case)
    wire = qr.qr_encode(bits, _to_dev(x, dtype))
    assert wire.numel() == qr.qr_tile_bytes(bits)
    _check_bytes(wire, case["expect_hex"], case["name"])
    y = qr.qr_decode(bits, wire, 2048, dtype=TORCH_DT[dtype])
    want = torch.from_numpy(expect).to(TORCH_DT[dtype])
    assert np.array_equal(_bits16(y), _bits16(want)), case["name"]


@pytest.mark.parametrize("case", [c for c in SYM if "slot_codes" in c], ids=lambda c: c["name"])
@pytest.mark.parametrize("R", [2, 4])
@pytest.mark.parametrize("dtype", [0, 1], ids=["fp16", "bf16"])
def test_identical_ranks_sum_exactly(case, R, dtype):
    bits = case["bits"]
    x, _ = _symmetric_case(case)
    xs = [_to_dev(x, dtype) for _ in range(R)]
    want = _bits16(torch.from_numpy(R * x).to(TORCH_DT[dtype]))
    assert np.array_equal(_bits16(qr.qr_allreduce(bits, xs)), want), f"{case['name']} fused R={R}"
    red = qr.qr_segment_reduce(bits, [qr.qr_encode(bits, t) for t in xs], 2048)
    assert np.array_equal(_bits16(qr.qr_decode(bits, red, 2048, dtype=TORCH_DT[dtype])), want), \
        f"{case['name']} unfused R={R}"


def _fc_group0(case):
    i = np.arange(128)
    if case["bits"] == 4:
        u = i % 16
    else:
        u = 2 * i
        u[127] = 255
    x = np.zeros(2048, np.float32)
    x[:128] = (case["lo"] + u * case["d"]).astype(np.float32)
    return x


@pytest.mark.parametrize("case", FC, ids=lambda c: c["name"])
@pytest.mark.parametrize("dtype", [0, 1], ids=["fp16", "bf16"])
def test_fc_encode_decode_known_answer_tiles(case, dtype):
    bits = case["bits"]
    x = _fc_group0(case)
    wire = qr.qr_fc_encode(bits, _to_dev(x, dtype))
    assert wire.numel() == qr.qr_fc_tile_bytes(bits)
    _check_bytes(wire, case["expect_hex"], case["name"])
    y = qr.qr_fc_decode(bits, wire, 2048, dtype=TORCH_DT[dtype])
    want = torch.from_numpy(x).to(TORCH_DT[dtype])
    assert np.array_equal(_bits16(y), _bits16(want)), case["name"]
