"""Pins of the oracle's W4A8 matmul (CPU)."""
import numpy as np

import synth
from oracle import matmul as OMM
from oracle import quant as Q


def _brute_int(a_q, w_q):
    M, K = a_q.shape
    N = w_q.shape[0]
    out = np.zeros((M, N), dtype=np.int64)
    for t in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(a_q[t, k]) * int(w_q[n, k])
            out[t, n] = acc
    return out


def test_unit_scales_give_exact_integer_dot():
    rng = np.random.default_rng(5)
    M, K, N = 3, 96, 5
    a_q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    w_q = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    y = OMM.w4a8_matmul(a_q, np.ones(M, np.float32), Q.pack_q4(w_q), np.ones((N, K // 32), np.float16))
    assert np.array_equal(y, _brute_int(a_q, w_q).astype(np.float64))


def test_group_sums_brute_force():
    rng = np.random.default_rng(6)
    a_q = rng.integers(-127, 128, size=(2, 64)).astype(np.int8)
    w_q = rng.integers(-8, 8, size=(3, 64)).astype(np.int8)
    gs = OMM.group_sums(a_q, w_q)
    for g in range(2):
        assert np.array_equal(gs[:, :, g], _brute_int(a_q[:, 32 * g:32 * g + 32], w_q[:, 32 * g:32 * g + 32]))


def test_scales_apply_per_group_and_token():
    # one non-zero group per row: y = s_a * s_w[g] * isum[g]; pins the group and row indexing
    rng = np.random.default_rng(7)
    M, K, N = 2, 128, 3
    a_q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    w_q = np.zeros((N, K), np.int8)
    w_s = rng.uniform(0.001, 0.02, size=(N, K // 32)).astype(np.float16)
    a_s = rng.uniform(0.01, 0.1, size=M).astype(np.float32)
    for n in range(N):
        g = (n + 1) % 4
        w_q[n, 32 * g:32 * g + 32] = rng.integers(-8, 8, size=32)
    y = OMM.w4a8_matmul(a_q, a_s, Q.pack_q4(w_q), w_s)
    isum = _brute_int(a_q, w_q)
    for t in range(M):
        for n in range(N):
            g = (n + 1) % 4
            ref = float(a_s[t]) * float(w_s[n, g]) * isum[t, n]
            assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_m1_matches_blog_matvec_restatement():
    # the blog's portable matvec on the dequantised activation vector, f32 scales
    seed, K, N = 11, 128, 6
    q, s = synth.matmul_rows(seed, K, np.arange(N))
    x = synth.normal(seed, 3, 0, K, 1.0)[None, :]
    a_q, a_s = Q.quantize_act_per_token(x)
    y = OMM.w4a8_matmul(a_q, a_s, Q.pack_q4(q), s)[0]
    xv = a_q[0].astype(np.float64) * float(a_s[0])
    y2 = OMM.matvec_q4(Q.pack_q4(q), s.astype(np.float32), xv)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12)


def test_per_block_activation_scales():
    rng = np.random.default_rng(8)
    x = rng.normal(size=(2, 96)).astype(np.float32)
    a_q, a_s = Q.quantize_act_per_block32(x)
    w_q = rng.integers(-8, 8, size=(4, 96)).astype(np.int8)
    w_s = rng.uniform(0.001, 0.02, size=(4, 3)).astype(np.float16)
    y = OMM.w4a8_matmul(a_q, a_s, Q.pack_q4(w_q), w_s)
    gs = OMM.group_sums(a_q, w_q)
    ref = (gs * w_s.astype(np.float64)[None] * a_s.astype(np.float64)[:, None, :]).sum(axis=2)
    assert np.allclose(y, ref, rtol=1e-13, atol=0)


def test_matmul_rows_match_full_case():
    q, s, x = synth.matmul_case(3, 2, 64, 10)
    q2, s2 = synth.matmul_rows(3, 64, np.array([0, 4, 9]))
    assert np.array_equal(q[[0, 4, 9]], q2) and np.array_equal(s[[0, 4, 9]], s2)
