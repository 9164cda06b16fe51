"""Pins of the oracle's quantisers and packed layout (CPU)."""
import os

import numpy as np
import pytest

from oracle import quant as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_pack_matches_worked_example():
    lines = [l.split() for l in open(os.path.join(GOLD, "q4_pack_example.txt")) if l.strip() and not l.startswith("#")]
    codes = np.array([int(v) for v in lines[0][1:]], dtype=np.int8)[None, :]
    words = np.array([int(v, 16) for v in lines[1][1:]], dtype=np.uint32)[None, :]
    assert np.array_equal(Q.pack_q4(codes), words)
    assert np.array_equal(Q.unpack_q4(words), codes)


def test_pack_roundtrip_random():
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, size=(7, 96)).astype(np.int8)
    assert np.array_equal(Q.unpack_q4(Q.pack_q4(q)), q)


def test_weight_quant_closed_form():
    # a group whose absmax is 7.0: the scale is exactly 1.0 and codes are rint(w) half-even
    w = np.zeros((1, 32), np.float32)
    w[0, :8] = [7.0, -7.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5]
    q, s = Q.quantize_weights_g32(w)
    assert s.dtype == np.float16 and float(s[0, 0]) == 1.0
    assert q[0, :8].tolist() == [7, -7, 2, 4, -2, 0, 2, 0]
    assert np.all(q[0, 8:] == 0)


def test_weight_quant_zero_group_and_extremes():
    rng = np.random.default_rng(1)
    w = rng.normal(0, 0.02, size=(3, 64)).astype(np.float32)
    w[1, 32:] = 0.0
    q, s = Q.quantize_weights_g32(w)
    assert float(s[1, 1]) == 0.0 and np.all(q[1, 32:] == 0)
    # the absmax element of every non-zero group lands on +-7
    g = w.reshape(3, 2, 32)
    for r in range(3):
        for j in range(2):
            if s[r, j] == 0:
                continue
            k = int(np.argmax(np.abs(g[r, j])))
            assert abs(int(q[r, 32 * j + k])) == 7
    # reconstruction error at most half a step
    dq = Q.dequantize_weights(q, s)
    step = np.repeat(s.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(dq - w) <= 0.5 * step * (1 + 1e-3) + 1e-12)


def test_weight_scale_is_fp16_of_absmax_over_7():
    rng = np.random.default_rng(2)
    w = rng.normal(0, 0.02, size=(4, 128)).astype(np.float32)
    _, s = Q.quantize_weights_g32(w)
    amax = np.abs(w.reshape(4, 4, 32)).max(axis=2)
    assert np.array_equal(s, (amax / np.float32(7)).astype(np.float32).astype(np.float16))


def test_act_quant_closed_form():
    x = np.array([[127.0, -63.5, 62.5, 0.5, 1.5, -127.0, 0.0, 3.0]], np.float32)
    q, s = Q.quantize_act_per_token(x)
    assert float(s[0]) == 1.0
    assert q[0].tolist() == [127, -64, 62, 0, 2, -127, 0, 3]
    z, sz = Q.quantize_act_per_token(np.zeros((1, 8), np.float32))
    assert float(sz[0]) == 0.0 and np.all(z == 0)


def test_act_quant_extremes_and_error():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5, 256)).astype(np.float32)
    q, s = Q.quantize_act_per_token(x)
    for t in range(5):
        k = int(np.argmax(np.abs(x[t])))
        assert abs(int(q[t, k])) == 127
        assert np.all(np.abs(q[t].astype(np.float64) * s[t] - x[t]) <= 0.5 * s[t] * (1 + 1e-5))


def test_act_quant_per_block_is_blockwise_per_token():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(3, 96)).astype(np.float32)
    q, s = Q.quantize_act_per_block32(x)
    assert s.shape == (3, 3)
    for b in range(3):
        qb, sb = Q.quantize_act_per_token(x[:, 32 * b:32 * b + 32])
        assert np.array_equal(q[:, 32 * b:32 * b + 32], qb) and np.array_equal(s[:, b], sb)
