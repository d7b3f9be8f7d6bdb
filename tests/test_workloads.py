"""The seeded input generators hold the recipes the tests and the benchmark
state: shapes, the crafted blocks of c1, the outlier channels (the same on
every rank) of c2, c3 and the sweep, determinism, and the storage-type
conversion (fp16 clipped to the finite range, bf16 the top half of the
float32 pattern).  Checked by exact bit patterns where a value is fixed and
by robust statistics where it is drawn."""
import numpy as np
import pytest

import workloads as W

F16 = lambda v: int(np.float16(v).view(np.uint16))  # noqa: E731


def _values(bits: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == W.FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_to_bits_conversions():
    x = np.array([1.0, -0.75, 1e6, -1e6, 0.0, -0.0], np.float32)
    assert list(W.to_bits(x, W.FP16)) == [0x3C00, 0xBA00, 0x7BFF, 0xFBFF, 0x0000, 0x8000]
    assert list(W.to_bits(x, W.BF16)) == [0x3F80, 0xBF40, 0x4974, 0xC974, 0x0000, 0x8000]
    # bf16 keeps the top half (no rounding of the draw)
    assert W.to_bits(np.array([0x3F80FFFF], np.uint32).view(np.float32), W.BF16)[0] == 0x3F80


def test_generators_are_deterministic_and_ranks_differ():
    a, b = W.ranks(W.C1), W.ranks(W.C1)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
    assert not np.array_equal(a[0], a[1])
    s0, s1 = W.sweep_rank(0, 10000, W.BF16), W.sweep_rank(1, 10000, W.BF16)
    assert np.array_equal(s0, W.sweep_rank(0, 10000, W.BF16)) and not np.array_equal(s0, s1)
    assert not np.array_equal(s0, W.sweep_rank(0, 10000, W.BF16, seed=6))


def test_c1_crafted_blocks():
    xs = W.ranks(W.C1)
    assert len(xs) == 2 and all(x.size == 4096 and x.dtype == np.uint16 for x in xs)
    blk = lambda g: slice(32 * g, 32 * g + 32)  # noqa: E731
    for r, x in enumerate(xs):
        assert np.all(x[blk(64)] == 0x0000)                      # all-zero block (+0)
        assert x[32 * 65 + 7] == (F16(1000.0) if r == 0 else F16(-1000.0))  # opposite outliers
        assert x[32 * 66 + 7] == F16(1000.0)                     # the same outlier on both ranks
        assert np.all(x[blk(67)] == F16(0.7))
        assert np.all(x[blk(68)] == F16(-0.75))
        assert np.all(x[blk(69)] == F16(1.0))
        v = _values(x, W.FP16)
        plain = np.r_[v[:32 * 64], v[32 * 70:]]
        assert abs(plain.mean()) < 0.1 and 0.9 < plain.std() < 1.1  # N(0,1) elsewhere


def _outlier_columns(x: np.ndarray, k: int) -> set:
    """The k columns with the largest median |value| (robust to the draw)."""
    med = np.median(np.abs(x), axis=0)
    return set(np.argsort(med)[-k:].tolist())


@pytest.mark.parametrize("cfg, shape, k, factor", [
    (W.C2, (16, 8192), 82, 20.0),
    (W.C3, (1024, 5120), 8, 50.0),
])
def test_outlier_channels_are_shared_by_every_rank(cfg, shape, k, factor):
    xs = W.ranks(cfg)
    assert len(xs) == cfg["R"] and all(x.size == shape[0] * shape[1] for x in xs)
    cols = [_outlier_columns(_values(x, W.BF16).reshape(shape), k) for x in xs]
    assert all(c == cols[0] for c in cols)
    v = _values(xs[0], W.BF16).reshape(shape)
    inside = np.median(np.abs(v[:, sorted(cols[0])]))
    outside = np.median(np.abs(np.delete(v, sorted(cols[0]), axis=1)))
    assert factor / 2 < inside / outside < factor * 2


def test_sweep_outlier_channels_and_ragged_tail():
    n = 4096 * 64 + 37
    xs = [W.sweep_rank(r, n, W.FP16) for r in range(2)]
    rows = [_values(x[: 4096 * 64], W.FP16).reshape(64, 4096) for x in xs]
    cols = [_outlier_columns(v, 8) for v in rows]
    assert cols[0] == cols[1]
    v = rows[0]
    ratio = np.median(np.abs(v[:, sorted(cols[0])])) / np.median(np.abs(np.delete(v, sorted(cols[0]), axis=1)))
    assert 10 < ratio < 40
    # the tail continues the channel pattern: value index mod 4096
    for x in xs:
        tail = np.abs(_values(x[4096 * 64:], W.FP16))
        for c in range(37):
            if c not in cols[0]:
                assert tail[c] < 8.0  # an unscaled N(0,1) draw (6 sigma is ~1e-9 likely)
