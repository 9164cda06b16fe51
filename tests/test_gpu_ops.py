"""GPU parity of the quantisers, the weight repack and the W4A8 matmul against the oracle.

Every GPU result here comes through the C ABI (libw4a8.so via the ctypes binding); the
oracle runs on the same seeded inputs drawn by ``synth``.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
import synth.cuda as SC
import w4a8_verify_gb300 as W
from oracle import matmul as OMM
from oracle import quant as Q

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    W.lib()
    SC.lib()


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _gpu_weights(q_codes, s16):
    """int8 codes [N][K] + fp16 scales -> tiled device layout via the library."""
    N, K = q_codes.shape
    wp2 = _to_dev(W.w4a8_pack_weights(q_codes).view(np.int32))
    sp2 = _to_dev(s16.view(np.int16))
    return W.w4a8_repack_weights(wp2, sp2, N, K)


def _tol(a_q, a_s, q, s, K, N):
    G = K // 32
    S = W.w4a8_matmul_slices(K, N)
    return (G + S + 2) * 2.0 ** -24 * OMM.abs_terms(a_q, a_s, q, s) + 1e-30


# ----------------------------------------------------------------------------- synth

def test_device_generator_matches_host():
    n = 100003
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    SC.normal(7, 3, 12345, out, 0.02)
    assert np.array_equal(out.cpu().numpy(), synth.normal(7, 3, 12345, n, 0.02))
    codes = torch.empty(n, dtype=torch.int8, device=DEV)
    SC.uniform_codes(7, 1, 999, codes)
    assert np.array_equal(codes.cpu().numpy(), synth.uniform_codes(7, 1, 999, n))
    sc = torch.empty(n, dtype=torch.int16, device=DEV)
    SC.uniform_scales(7, 2, 5, sc)
    assert np.array_equal(sc.cpu().numpy().view(np.float16), synth.uniform_scales(7, 2, 5, n))
    dw = torch.empty((50, 256), dtype=torch.float32, device=DEV)
    SC.dense_weight(synth.TINY, 1000, synth.layer_stream(1, synth.T_WG), 704, 256, 688, 256, dw, row0=650)
    ref = synth.dense_weight(synth.TINY, 1000, synth.layer_stream(1, synth.T_WG), 704, 256, 688, 256, row0=650, nrows=50)
    assert np.array_equal(dw.cpu().numpy(), ref)


# ----------------------------------------------------------------------------- quantisers

@pytest.mark.parametrize("N,K", [(64, 256), (688, 256), (256, 704), (3, 32)])
def test_quantize_weights_bit_exact(N, K):
    w = synth.dense_weight(synth.TINY, 1000, 5, N, K, N, K)
    if K >= 64:
        w[1, 32:64] = 0.0                               # a zero group
    if N > 2:
        w[2, K - 32:] = 1e-30                           # a group whose fp16 scale underflows to 0
    wq, ws = W.w4a8_quantize_weights(_to_dev(w))
    q_ref, s_ref = Q.quantize_weights_g32(w)
    assert np.array_equal(wq.cpu().numpy().view(np.uint32), Q.pack_q4(q_ref))
    assert np.array_equal(ws.cpu().numpy().view(np.uint16), s_ref.view(np.uint16))


@pytest.mark.parametrize("M,K", [(1, 256), (16, 4096), (5, 704), (16, 14336), (3, 32)])
def test_quantize_rows_per_token_bit_exact(M, K):
    x = synth.normal(21, 3, 0, M * K, 1.0).reshape(M, K)
    x[0, :] = 0.0 if M > 2 else x[0, :]
    q, s = W.w4a8_quantize_rows(_to_dev(x), 0)
    q_ref, s_ref = Q.quantize_act_per_token(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy(), s_ref)


def test_quantize_rows_per_block_bit_exact():
    x = synth.normal(22, 3, 0, 4 * 256, 3.0).reshape(4, 256)
    x[1, 64:96] = 0.0
    q, s = W.w4a8_quantize_rows(_to_dev(x), 1)
    q_ref, s_ref = Q.quantize_act_per_block32(x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy(), s_ref)


# ----------------------------------------------------------------------------- matmul

@pytest.mark.parametrize("M,K,N", [(1, 64, 32), (16, 96, 48), (7, 4096, 256), (16, 704, 272), (3, 32, 16)])
def test_matmul_unit_scales_are_exact_integers(M, K, N):
    rng = np.random.default_rng(M * 1000 + K + N)
    a_q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    a_q[0, :8] = [-128 + 1, 127, -127, 0, 1, -1, 16, -16]
    q = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s16 = np.ones((N, K // 32), np.float16)
    w_t, s_t = _gpu_weights(q, s16)
    y = W.w4a8_matmul(_to_dev(a_q), _to_dev(np.ones(M, np.float32)), w_t, s_t, N).cpu().numpy()
    ref = (a_q.astype(np.int64) @ q.astype(np.int64).T).astype(np.float64)
    assert np.array_equal(y.astype(np.float64), ref)


@pytest.mark.parametrize("M,K,N", [(1, 896, 4864), (8, 4864, 896), (16, 4096, 1024), (5, 704, 512), (16, 256, 4096),
                                   (2, 14336, 256), (13, 96, 80)])
def test_matmul_matches_oracle(M, K, N):
    seed = 2000 + M + K
    q, s, x = synth.matmul_case(seed, M, K, N)
    xd = _to_dev(x)
    a_q, a_s = W.w4a8_quantize_rows(xd, 0)
    a_q_ref, a_s_ref = Q.quantize_act_per_token(x)
    assert np.array_equal(a_q.cpu().numpy(), a_q_ref)
    w_t, s_t = _gpu_weights(q, s)
    y = W.w4a8_matmul(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64)
    ref = OMM.w4a8_matmul(a_q_ref, a_s_ref, Q.pack_q4(q), s)
    tol = _tol(a_q_ref, a_s_ref, q, s, K, N)
    assert np.all(np.abs(y - ref) <= tol), float(np.max(np.abs(y - ref) / tol))


@pytest.mark.parametrize("K,N", [(896, 4864), (4864, 896), (4096, 1152), (704, 256)])
def test_matmul_m_tokens_bitwise_equal_single_token_calls(K, N):
    M = 16
    q, s, x = synth.matmul_case(3000 + K, M, K, N)
    a_q, a_s = W.w4a8_quantize_rows(_to_dev(x), 0)
    w_t, s_t = _gpu_weights(q, s)
    y_all = W.w4a8_matmul(a_q, a_s, w_t, s_t, N)
    for m in (1, 2, 4, 8):
        y_m = W.w4a8_matmul(a_q[:m].contiguous(), a_s[:m].contiguous(), w_t, s_t, N)
        assert torch.equal(y_m, y_all[:m])
    for t in (0, 7, 8, 15):
        y1 = W.w4a8_matmul(a_q[t:t + 1].contiguous(), a_s[t:t + 1].contiguous(), w_t, s_t, N)
        assert torch.equal(y1[0], y_all[t])


@pytest.mark.parametrize("M,K,N", [(16, 4096, 14336), (1, 14336, 4096), (16, 4096, 128256), (4, 4864, 896)])
def test_matmul_full_size_sampled_rows(M, K, N):
    seed = 4000 + K + N
    q, s, x = synth.matmul_case(seed, M, K, N)
    a_q, a_s = W.w4a8_quantize_rows(_to_dev(x), 0)
    w_t, s_t = _gpu_weights(q, s)
    y = W.w4a8_matmul(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64)
    rows = np.unique(np.concatenate([np.arange(0, N, max(1, N // 97)), [N - 1, N - 16]]))
    qr, sr = synth.matmul_rows(seed, K, rows)
    a_q_ref, a_s_ref = Q.quantize_act_per_token(x)
    ref = OMM.w4a8_matmul(a_q_ref, a_s_ref, Q.pack_q4(qr), sr)
    tol = _tol(a_q_ref, a_s_ref, qr, sr, K, N)
    assert np.all(np.abs(y[:, rows] - ref) <= tol)


def test_matmul_repeated_calls_reuse_workspace():
    # the split-K tickets are restored by every call: repeated calls give identical bits
    M, K, N = 8, 4096, 512
    q, s, x = synth.matmul_case(77, M, K, N)
    a_q, a_s = W.w4a8_quantize_rows(_to_dev(x), 0)
    w_t, s_t = _gpu_weights(q, s)
    ws = torch.empty(W.w4a8_matmul_workspace_bytes(M, K, N), dtype=torch.uint8, device=DEV)
    ys = [W.w4a8_matmul(a_q, a_s, w_t, s_t, N, workspace=ws) for _ in range(4)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


# ------------------------------------------------------------- non-deterministic variant

@pytest.mark.parametrize("M,K,N", [(1, 896, 4864), (8, 4864, 896), (16, 4096, 1024), (3, 14336, 256), (5, 96, 48)])
def test_nondet_matmul_matches_oracle_within_the_same_bound(M, K, N):
    # the same exact integer group sums and slice chains; only the order of the S slice adds
    # differs, which the first-order bound (G + S + 2) 2^-24 sum|terms| already covers
    seed = 2500 + M + K
    q, s, x = synth.matmul_case(seed, M, K, N)
    a_q, a_s = W.w4a8_quantize_rows(_to_dev(x), 0)
    w_t, s_t = _gpu_weights(q, s)
    y = W.w4a8_matmul_nondet(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64)
    a_q_ref, a_s_ref = Q.quantize_act_per_token(x)
    ref = OMM.w4a8_matmul(a_q_ref, a_s_ref, Q.pack_q4(q), s)
    tol = _tol(a_q_ref, a_s_ref, q, s, K, N)
    assert np.all(np.abs(y - ref) <= tol), float(np.max(np.abs(y - ref) / tol))
    if W.w4a8_matmul_slices(K, N) == 1:   # a single slice: nothing to reorder, same bits
        assert np.array_equal(y, W.w4a8_matmul(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64))


# ------------------------------------------------------------------ per-32 activation scales

def _per32_case(seed, M, K, N):
    q, s, x = synth.matmul_case(seed, M, K, N)
    xd = _to_dev(x)
    a_q, a_s = W.w4a8_quantize_rows(xd, 1)              # one scale per block of 32 inputs
    a_q_ref, a_s_ref = Q.quantize_act_per_block32(x)
    assert np.array_equal(a_q.cpu().numpy(), a_q_ref) and np.array_equal(a_s.cpu().numpy(), a_s_ref)
    return q, s, a_q, a_s, a_q_ref, a_s_ref


@pytest.mark.parametrize("M,K,N", [(1, 896, 4864), (8, 4864, 896), (16, 4096, 1024), (5, 704, 512), (3, 96, 48)])
def test_per32_matmul_matches_oracle(M, K, N):
    q, s, a_q, a_s, a_q_ref, a_s_ref = _per32_case(5000 + M + K, M, K, N)
    w_t, s_t = _gpu_weights(q, s)
    y = W.w4a8_matmul_per32(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64)
    ref = OMM.w4a8_matmul(a_q_ref, a_s_ref, Q.pack_q4(q), s)
    # one more rounding than the per-token form: the product scale s_w * s_a of each group
    G = K // 32
    tol = (G + W.w4a8_matmul_slices(K, N) + 3) * 2.0 ** -24 * OMM.abs_terms(a_q_ref, a_s_ref, q, s) + 1e-30
    assert np.all(np.abs(y - ref) <= tol), float(np.max(np.abs(y - ref) / tol))


def test_per32_matmul_m_tokens_bitwise_equal_single_token_calls():
    M, K, N = 16, 4864, 896
    q, s, a_q, a_s, _, _ = _per32_case(5100, M, K, N)
    w_t, s_t = _gpu_weights(q, s)
    y_all = W.w4a8_matmul_per32(a_q, a_s, w_t, s_t, N)
    for t in (0, 5, 8, 15):
        y1 = W.w4a8_matmul_per32(a_q[t:t + 1].contiguous(), a_s[t:t + 1].contiguous(), w_t, s_t, N)
        assert torch.equal(y1[0], y_all[t])


def test_per32_with_equal_block_scales_is_the_per_token_product():
    # every block of a row with the per-token scale: the same products, the per-32 order
    # multiplies the scale into each group instead of the fold, so agreement is to rounding
    M, K, N = 4, 4096, 512
    q, s, x = synth.matmul_case(5200, M, K, N)
    a_q, a_s = W.w4a8_quantize_rows(_to_dev(x), 0)
    a_s32 = a_s[:, None].expand(M, K // 32).contiguous()
    w_t, s_t = _gpu_weights(q, s)
    y_tok = W.w4a8_matmul(a_q, a_s, w_t, s_t, N).cpu().numpy().astype(np.float64)
    y_32 = W.w4a8_matmul_per32(a_q, a_s32, w_t, s_t, N).cpu().numpy().astype(np.float64)
    a_q_ref, a_s_ref = Q.quantize_act_per_token(x)
    tol = 2 * (K // 32 + W.w4a8_matmul_slices(K, N) + 3) * 2.0 ** -24 * OMM.abs_terms(a_q_ref, a_s_ref, q, s)
    assert np.all(np.abs(y_32 - y_tok) <= tol)
