"""Timeout paths, exercised without any GPU fault or hang.

* A device wait that runs out: ``w4a8_matmul_inject_timeout`` runs the matmul kernel in a
  test-only variant whose copy warp issues nothing, so each consumer's bounded wait (1 ms)
  expires; the kernel must report the timeout in the workspace status word, leave the output
  unwritten and return, and the next calls on the device must work.
* A host wait that runs out: ``spec_poll`` with a zero deadline on a window queued behind a
  bounded spin kernel must return W4A8_ERR_TIMEOUT and leave the window in flight; a second
  poll then returns its results.
"""
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


@pytest.mark.parametrize("M,K,N", [(1, 4096, 6144), (12, 4864, 896), (3, 704, 256)])
def test_expired_device_wait_is_reported_and_the_device_stays_usable(M, K, N):
    a_q, a_s, w_t, s_t = _case(300 + M, M, K, N)
    need = W.w4a8_matmul_workspace_bytes(M, K, N)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y = torch.full((M, N), 7.0, device="cuda")
    W.w4a8_matmul_inject_timeout(a_q, a_s, w_t, s_t, N, y, ws)
    torch.cuda.synchronize()
    assert W.w4a8_matmul_check(ws, M, K, N) == W.FLAG_ERR_TIMEOUT
    assert torch.all(y == 7.0)                          # the output was skipped
    # the device and the library keep working: a normal call on a fresh workspace
    ws2 = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y2 = W.w4a8_matmul(a_q, a_s, w_t, s_t, N, workspace=ws2)
    y3 = W.w4a8_matmul(a_q, a_s, w_t, s_t, N)
    torch.cuda.synchronize()
    assert W.w4a8_matmul_check(ws2, M, K, N) == 0
    assert torch.equal(y2, y3) and torch.isfinite(y2).all()


def test_spec_poll_deadline_expires_then_the_window_completes():
    from test_gpu_decoder import gpu_model
    m = gpu_model()
    prompt = synth.motif_prompt(1001, 64, 4, 16, 0.1, synth.TINY.vocab)
    s = W.Session(m, 256, 512, 8)
    ref, _ = s.decode(list(prompt), 8, window=8, fixed_width=4, in_flight=1)
    s.prefill(torch.as_tensor(prompt).cuda(), max_new=8)
    torch.cuda._sleep(100_000_000)                      # a bounded spin kernel ahead of the window (~50 ms)
    s.spec_window(4, 8)
    with pytest.raises(W.W4A8Error) as e:
        s.spec_poll(8, timeout_us=0)
    assert e.value.status == 6                           # W4A8_ERR_TIMEOUT: the window stays in flight
    c, st, toks = s.spec_poll(8)
    assert toks == ref and c.flags & W.FLAG_TERMINATED
    with pytest.raises(W.W4A8Error):
        s.spec_poll(1)                                   # nothing left in flight
