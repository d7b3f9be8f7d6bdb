"""Phase-1B on long messages through the one-block-ahead kernel (the library
takes it from 48 tiles per SM at the rank counts and widths it names): the
reduced wire of every such case against the oracle's, on sampled tiles of
GPU-encoded wires (tiles are independent, so each sampled tile is checked
exactly), plus the first and last tiles; the staged kernel's wire must be
byte-identical.  Each thread of the kernel reduces several blocks, so both of
its register sets are used."""
import numpy as np
import pytest
import torch

import bit_quantized_all_gb300 as qr
import oracle
from qr_testlib import gather_wire_tiles, sample_tiles, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from bit_quantized_all_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    qr.lib()


def _ranks(R, n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for r in range(R):
        v = (rng.standard_normal(n) * (1 + r)).astype(np.float32)
        v[rng.integers(0, n, size=n // 500)] *= 30.0
        out.append(oracle.narrow(1, v))
    return out


def _long_n():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 2048 * (48 * sms + 301) + 7  # past the 48-tiles-per-SM threshold, a ragged tail


@pytest.mark.parametrize("bits,R", [(8, 4), (6, 2), (6, 3), (6, 4), (6, 5), (4, 2), (4, 3), (4, 4), (4, 5), (4, 6),
                                    (4, 7), (4, 8), (3, 2), (3, 7), (3, 8)])
def test_symmetric_phase1b_one_block_ahead(bits, R):
    n = _long_n()
    xs = [to_dev(x, 1) for x in _ranks(R, n, 40 + 7 * bits + R)]
    wires = [qr.qr_encode(bits, x) for x in xs]
    red = qr.qr_segment_reduce(bits, wires, n)
    T = -(-n // 2048)
    if bits != 3:
        staged = qr.qr_segment_reduce(bits, wires, n, staged=True)
        assert torch.equal(red, staged), f"INT{bits} R={R}: default and staged Phase-1B differ"
    tiles = np.unique(np.concatenate([sample_tiles(T, 96, seed=bits * 10 + R), [0, T - 1]]))
    w_t = [gather_wire_tiles(w, tiles, bits) for w in wires]
    red_t = gather_wire_tiles(red, tiles, bits)
    tb = qr.qr_tile_bytes(bits)
    for i, t in enumerate(tiles.tolist()):
        m = 2048 if t < T - 1 else n - 2048 * (T - 1)
        ref = oracle.segment_reduce(bits, [w[i * tb:(i + 1) * tb] for w in w_t], m)
        assert np.array_equal(red_t[i * tb:(i + 1) * tb], ref), f"INT{bits} R={R} tile {t}"
    assert qr.qr_wait_timeouts() == 0


@pytest.mark.parametrize("R", [2, 3, 8])
def test_fp4_phase1b_one_block_ahead(R):
    n = _long_n()
    xs = [to_dev(x, 1) for x in _ranks(R, n, 90 + R)]
    wires = [qr.qr_fp4_encode(x) for x in xs]
    red = qr.qr_fp4_segment_reduce(wires, n)
    staged = qr.qr_fp4_segment_reduce(wires, n, ctas=torch.cuda.get_device_properties(0).multi_processor_count)
    assert torch.equal(red, staged), f"FP4 R={R}: default and staged Phase-1B differ"
    T = -(-n // 2048)
    tiles = np.unique(np.concatenate([sample_tiles(T, 96, seed=R), [0, T - 1]]))
    tb = qr.qr_fp4_tile_bytes()
    idx = torch.as_tensor(tiles, device=red.device)
    rows = (idx[:, None] * tb + torch.arange(tb, device=red.device)[None, :]).reshape(-1)
    w_t = [w[rows].cpu().numpy() for w in wires]
    red_t = red[rows].cpu().numpy()
    for i, t in enumerate(tiles.tolist()):
        m = 2048 if t < T - 1 else n - 2048 * (T - 1)
        ref = oracle.fp4_segment_reduce([w[i * tb:(i + 1) * tb] for w in w_t], m)
        assert np.array_equal(red_t[i * tb:(i + 1) * tb], ref), f"FP4 R={R} tile {t}"
    assert qr.qr_wait_timeouts() == 0
