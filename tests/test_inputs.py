"""The seeded generators: SplitMix64 against its published first output, ranges, independence of streams."""
import numpy as np

import inputs


def test_splitmix64_published_value():
    # SplitMix64 started from state 0: first output 0xE220A8397B1DCDAF
    assert int(inputs.mix64(np.array([inputs.GAMMA], np.uint64))[0]) == 0xE220A8397B1DCDAF


def test_counter_mode_is_slice_consistent():
    a = inputs.words(0, 3, 0, 1000)
    b = inputs.words(0, 3, 500, 500)
    assert np.array_equal(a[500:], b)
    assert not np.array_equal(inputs.words(0, 3, 0, 100), inputs.words(0, 4, 0, 100))
    assert not np.array_equal(inputs.words(0, 3, 0, 100), inputs.words(1, 3, 0, 100))


def test_int4_uniform_and_scales_in_range():
    b = inputs.packed_int4(0, 1, 0, 1 << 16)
    nib = np.concatenate([b & 0xF, b >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16
    s = inputs.scales(0, 2, 0, 1 << 16)
    assert s.dtype == np.float32 and s.min() >= np.float32(0.005) and s.max() < np.float32(0.02)
    u = inputs.uniform01(0, 2, 0, 10)
    assert np.array_equal(s[:10], (np.float32(0.005) + (np.float32(0.015) * u).astype(np.float32)))


def test_zipf_bias_popularity():
    lg = inputs.router_logits(0, 4096, 384, zipf=1.2)
    top1 = np.argmax(lg, axis=1)
    counts = np.sort(np.bincount(top1, minlength=384))[::-1]
    assert counts[0] > 20 * max(1, counts[192])  # a few hot experts, many cold ones


def test_bf16_helpers():
    x = np.array([1.0, 1.0 + 2 ** -8, -3.5, 1e-40], np.float32)
    b = inputs.to_bf16_bits(x)
    assert b.tolist()[:3] == [0x3F80, 0x3F80, 0xC060]
    assert np.array_equal(inputs.bf16_bits_to_f32(b[:3]), np.array([1.0, 1.0, -3.5], np.float32))
