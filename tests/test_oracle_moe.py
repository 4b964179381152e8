"""End-to-end pin of the oracle layer: a hand-worked 2-expert / 4-token example.

All scales are powers of two and every quantisation lands on an exact code, so
each intermediate below was derived by hand:

  H = I = 128, E = 2, k = 2, T = 4.
  x[t] = 448 at column 0 and 64 at column 1+t  ->  amax 448, scale 1,
         codes 0x7E (448) and 0x68 (64).
  w13 (scales 1 on gate rows, 2**-6 on up rows) gives, for every pair:
     gate row 0 = 64, gate row 2 = 64, gate row 1 = -64 for (expert 0, token 0) else 0,
     up row 0 = +(7 - t) for expert 0, -(7 - t) for expert 1,
     up row 1 = 3 (expert 0) / 5 (expert 1), up row 2 = 7, everything else 0.
  silu(64) = 64 and silu(0) = 0 exactly, silu(-64) ~ -1e-26 quantises to -0, so
     h = [64 (+-(7-t)), +-0, 448, 0, ...] with amax 448 and scale 1.
  w2 (scales 2**-6) is built so both experts give the same row:
     y2[n] = (7 - t) * ((n % 3) - 1) + 7 * ((n % 5) - 2),
  hence out[t, n] = y2[n] whatever the routing weights (they sum to 1).
"""
import math

import numpy as np

import oracle

H = I = 128
E, K_TOP, T = 2, 2, 4


def build():
    x = np.zeros((T, H), np.float32)
    x[:, 0] = 448.0
    for t in range(T):
        x[t, 1 + t] = 64.0
    logits = np.array([[0, 0], [0, 1], [3, -1], [-2, -2]], np.float32)
    w13 = np.zeros((E, 2 * I, H), np.int8)
    w13[0, 0, 1:5] = 1
    w13[0, 1, 1] = -1
    w13[0, 2, 1:5] = 1
    w13[0, I + 0, 0], w13[0, I + 0, 1:5] = 1, [0, -1, -2, -3]
    w13[0, I + 1, 1:5] = 3
    w13[0, I + 2, 0] = 1
    w13[1, 0, 0], w13[1, 0, 1:5] = 1, -6
    w13[1, 1, 0], w13[1, 1, 1:5] = 1, -7
    w13[1, 2, 0], w13[1, 2, 1:5] = 1, -6
    w13[1, I + 0, 0], w13[1, I + 0, 1:5] = -1, [0, 1, 2, 3]
    w13[1, I + 1, 1:5] = 5
    w13[1, I + 2, 0] = 1
    w13s = np.ones((E, 2 * I, 1), np.float32)
    w13s[:, I:, :] = 2.0 ** -6
    n = np.arange(H)
    w2 = np.zeros((E, H, I), np.int8)
    w2[0, :, 0] = (n % 3) - 1
    w2[1, :, 0] = 1 - (n % 3)
    w2[:, :, 2] = (n % 5) - 2
    w2s = np.full((E, H, 1), 2.0 ** -6, np.float32)
    return x, logits, w13, w13s, w2, w2s


def expected_out():
    n = np.arange(H)
    return np.stack([(7 - t) * ((n % 3) - 1) + 7 * ((n % 5) - 2) for t in range(T)]).astype(np.float64)


def test_hand_worked_layer():
    x, logits, w13, w13s, w2, w2s = build()
    r = oracle.moe_layer(x, logits, K_TOP, w13.__getitem__, w13s.__getitem__,
                         w2.__getitem__, w2s.__getitem__)
    assert r["ids"].tolist() == [[0, 1], [1, 0], [0, 1], [0, 1]]
    e = math.e
    assert np.allclose(r["w"], [[0.5, 0.5], [e / (1 + e), 1 / (1 + e)],
                                [1 / (1 + e ** -4), e ** -4 / (1 + e ** -4)], [0.5, 0.5]], rtol=1e-15)
    assert r["seg"].tolist() == [0, 4, 8]
    assert r["dst2src"].tolist() == [0, 3, 4, 6, 1, 2, 5, 7]
    assert r["src2dst"].tolist() == [0, 4, 5, 1, 2, 6, 3, 7]
    assert np.all(r["xs"] == 1.0)
    for t in range(T):
        row = np.zeros(H, np.uint8)
        row[0], row[1 + t] = 0x7E, 0x68
        assert np.array_equal(r["xq"][t], row)
    # permuted pair order: (t, e) for rows j = 0..7
    pairs = [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1), (1, 1), (2, 1), (3, 1)]
    for j, (t, ex) in enumerate(pairs):
        y13 = r["y13"][j]
        sgn = 1 if ex == 0 else -1
        want = np.zeros(2 * I)
        want[0] = 64
        want[1] = -64 if (ex, t) == (0, 0) else 0
        want[2] = 64
        want[I + 0] = sgn * (7 - t)
        want[I + 1] = 3 if ex == 0 else 5
        want[I + 2] = 7
        assert np.array_equal(y13, want), (j, t, ex)
        hq = np.zeros(I, np.uint8)
        hq[0] = [0x7E, 0x7C, 0x7A, 0x78][t] | (0 if ex == 0 else 0x80)
        hq[1] = 0x80 if (ex, t) == (0, 0) else 0x00
        hq[2] = 0x7E
        assert np.array_equal(r["hq"][j], hq), (j, t, ex)
        assert r["hs"][j, 0] == 1.0
        assert np.array_equal(r["y2"][j], expected_out()[t])
    assert np.array_equal(r["out"], expected_out())


def test_per_token_path_matches_layer():
    x, logits, w13, w13s, w2, w2s = build()
    out, ids, w = oracle.moe_tokens(x, logits, K_TOP, w13.__getitem__, w13s.__getitem__,
                                    w2.__getitem__, w2s.__getitem__)
    assert np.array_equal(out, expected_out())
    # and on random data, against the permuted layer
    rng = np.random.default_rng(21)
    T2, H2, I2, E2, k2 = 9, 256, 256, 4, 2
    xr = oracle.round_bf16(rng.standard_normal((T2, H2))).astype(np.float32)
    lg = rng.standard_normal((T2, E2)).astype(np.float32)
    W13 = rng.integers(-8, 8, (E2, 2 * I2, H2)).astype(np.int8)
    S13 = rng.uniform(0.005, 0.02, (E2, 2 * I2, H2 // 128)).astype(np.float32)
    W2 = rng.integers(-8, 8, (E2, H2, I2)).astype(np.int8)
    S2 = rng.uniform(0.005, 0.02, (E2, H2, I2 // 128)).astype(np.float32)
    full = oracle.moe_layer(xr, lg, k2, W13.__getitem__, S13.__getitem__, W2.__getitem__, S2.__getitem__)
    part, _, _ = oracle.moe_tokens(xr[3:6], lg[3:6], k2, W13.__getitem__, S13.__getitem__,
                                   W2.__getitem__, S2.__getitem__)
    assert np.array_equal(part, full["out"][3:6])
