"""Pins of the oracle's E4M3 codec against the OCP FP8 definition and an independent library cast."""
import numpy as np
import pytest
import torch

from oracle import e4m3


def test_decode_fixed_points():
    d = e4m3.decode(np.arange(256, dtype=np.uint8))
    assert d[0x00] == 0.0 and not np.signbit(d[0x00])
    assert d[0x80] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9          # smallest subnormal
    assert d[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert d[0x08] == 2.0 ** -6          # smallest normal
    assert d[0x38] == 1.0
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.count_nonzero(~np.isnan(d)) == 254


def test_positive_codes_strictly_increasing():
    d = e4m3.decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(d) > 0)


def test_round_trip_all_finite_codes():
    c = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(e4m3.encode(e4m3.decode(c).astype(np.float32)), c)


def test_ties_to_even_and_neighbours():
    d = e4m3.decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        mid = np.float32((d[c] + d[c + 1]) / 2)  # exact: needs 5 significant bits
        assert float(mid) == (d[c] + d[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert e4m3.encode(mid) == even
        assert e4m3.encode(np.nextafter(mid, np.float32(np.inf))) == c + 1
        assert e4m3.encode(np.nextafter(mid, np.float32(0))) == c
        assert e4m3.encode(-mid) == (even | 0x80)


def test_saturation():
    for v, code in [(448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E),
                    (-1e30, 0xFE), (-np.inf, 0xFE)]:
        assert e4m3.encode(np.float32(v)) == code


def test_signed_zero():
    assert e4m3.encode(np.float32(-0.0)) == 0x80
    assert e4m3.encode(np.float32(-1e-9)) == 0x80
    assert e4m3.encode(np.float32(1e-9)) == 0x00


def test_int4_values_are_exact():
    v = np.arange(-8, 8, dtype=np.float32)
    assert np.array_equal(e4m3.decode(e4m3.encode(v)), v.astype(np.float64))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_torch_cast_in_range(seed):
    # torch's float8_e4m3fn cast (round to nearest even) is an independent implementation;
    # in range it must agree bit for bit.
    rng = np.random.default_rng(seed)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(rng.uniform(0.001, 100)),
        rng.uniform(-448, 448, 20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-3).astype(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x), ref)
