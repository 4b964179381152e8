"""Pins of the per-token-group FP8 quantisation: closed forms and an independent torch route."""
import numpy as np
import torch

import oracle
from oracle import e4m3


def test_amax_maps_to_448():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 384)).astype(np.float32)
    q, s = oracle.quant_per_token_group(x)
    for r in range(5):
        for g in range(3):
            blk = x[r, g * 128:(g + 1) * 128]
            i = int(np.argmax(np.abs(blk)))
            assert q[r, g * 128 + i] == (0xFE if blk[i] < 0 else 0x7E)
            assert s[r, g] == np.float32(np.abs(blk).max()) / np.float32(448)


def test_zero_row_and_spike():
    x = np.zeros((2, 256), dtype=np.float32)
    x[1, 5] = 3.0
    x[1, 6] = np.float32(3.0 / 448 * 0.5)  # x / s rounds to 0.5 = code 0x30
    q, s = oracle.quant_per_token_group(x)
    assert np.all(q[0] == 0)
    assert s[0, 0] == np.float32(1e-12) / np.float32(448)
    assert q[1, 5] == 0x7E
    assert s[1, 0] == np.float32(3.0) / np.float32(448)
    assert q[1, 6] == 0x30
    assert np.all(q[1, 128:] == 0)


def test_matches_torch_route():
    # The same definition through torch ops and torch's fp8 cast (independent of oracle.e4m3).
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((17, 512)) * rng.uniform(0.01, 50, (17, 1))).astype(np.float32)
    q, s = oracle.quant_per_token_group(x)
    xt = torch.from_numpy(x).view(17, 4, 128)
    amax = xt.abs().amax(dim=2).clamp_min(1e-12)
    st = amax / 448.0
    qt = (xt / st[:, :, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(q, qt.reshape(17, 512).numpy())


def test_dequant_error_bound():
    # relative error of each element is at most half a code step: 2**-4 of the value (normals)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 256)).astype(np.float32)
    q, s = oracle.quant_per_token_group(x)
    xd = oracle.dequant(q, s)
    s_full = np.repeat(s.astype(np.float64), 128, axis=1)
    err = np.abs(xd - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s_full * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))
