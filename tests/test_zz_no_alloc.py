"""The allocation-free matmul entry point (w4a8_matmul_noalloc) against w4a8_matmul.

Some callers cannot allocate device memory (code inside a stream capture, hosts that pass
only inputs and outputs); they use the variant whose scratch is the library's own static
device array.  This file is collected last on purpose: it checks that the shared array,
which keeps the previous call's contents, gives the same output as the workspace-based
entry point on two calls in a row, whether run alone or after every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
import w4a8_verify_gb300 as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    W.lib()


def _case(seed, M, K, N):
    q, s, x = synth.matmul_case(seed, M, K, N)
    wp2 = torch.from_numpy(W.w4a8_pack_weights(q).view(np.int32)).cuda()
    sp2 = torch.from_numpy(s.view(np.int16)).cuda()
    w_t, s_t = W.w4a8_repack_weights(wp2, sp2, N, K)
    a_q, a_s = W.w4a8_quantize_rows(torch.from_numpy(x).cuda(), 0)
    return a_q, a_s, w_t, s_t


@pytest.mark.parametrize("M,K,N", [(1, 4096, 6144), (16, 14336, 4096), (5, 704, 256), (8, 4096, 128256)])
def test_noalloc_matches_workspace_entry_point_twice(M, K, N):
    a_q, a_s, w_t, s_t = _case(9000 + M + K, M, K, N)
    ref = W.w4a8_matmul(a_q, a_s, w_t, s_t, N)
    for _ in range(2):                                   # the second call reuses the dirty array
        y = torch.full((M, N), float("nan"), device="cuda")
        W.w4a8_matmul_noalloc(a_q, a_s, w_t, s_t, N, y)
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
        assert W.w4a8_matmul_noalloc_check() == 0        # no bounded wait expired


def test_noalloc_alternating_shapes():
    # a split-K shape after a different shape: slice counters must start at zero again
    cases = [_case(9100, 4, 4096, 6144), _case(9101, 16, 896, 4864)]
    refs = [W.w4a8_matmul(*c, N) for c, N in zip(cases, (6144, 4864))]
    for _ in range(2):
        for c, N, ref in zip(cases, (6144, 4864), refs):
            y = torch.empty((c[0].shape[0], N), device="cuda")
            W.w4a8_matmul_noalloc(*c, N, y)
            torch.cuda.synchronize()
            assert torch.equal(y, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = W.lib()
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    # K = 2^20 needs more than the 32 MiB of fragments and corrections: refused before any launch
    st = lib.w4a8_matmul_noalloc(p, p, 1, 1 << 20, p, p, 16, p, None)
    assert st == 4
