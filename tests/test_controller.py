"""Host-side width controller (no GPU): decision rule on injected costs and acceptance.

"GPU-Resident Speculative Decoding ...", Design > Feedback Control of Speculation Width.
Parity unpinned (heuristic); these tests pin its decision rule: the width maximising
expected tokens per microsecond, the probing of a wider tree after plain decoding, and the
moving-average cost update."""
import pytest

import w4a8_verify_gb300 as W
from w4a8_verify_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    W.lib()


def st(d, ell, emitted=None):
    return W.StepStats(d, ell, 16, d + 1 if emitted is None else emitted, 0)


def test_cheap_wide_steps_open_wide_and_expensive_open_plain():
    cheap = W.Controller([1, 4, 8], [100.0, 105.0, 110.0])
    assert cheap.choose() > 1
    costly = W.Controller([1, 4, 8], [100.0, 400.0, 800.0])
    assert costly.choose() == 1


def test_choice_is_argmax_of_expected_tokens_per_cost():
    c = W.Controller([1, 2, 4, 8], [100.0, 104.0, 120.0, 150.0])
    # observed: at match length 3, width 4 yields 3.5 tokens, width 8 yields 3.6
    for _ in range(200):
        c.observe(4, [st(2, 3, 3)] * 1 + [st(3, 3, 4)] * 1)
        c.observe(8, [st(3, 3, 4), st(2, 3, 3)] + [st(3, 3, 4)] * 0)
    e = {w: c.expected_tokens(w) for w in (1, 2, 4, 8)}
    best = max((e[w] / c.cost(w), -w) for w in (1, 2, 4, 8))
    assert c.choose() == -best[1]
    assert e[1] == 1.0


def test_zero_acceptance_falls_back_to_plain_then_probes():
    c = W.Controller([1, 8], [100.0, 130.0])
    for _ in range(50):
        c.observe(8, [st(0, 0, 1)] * 4)
    picks = [c.choose() for _ in range(20)]
    assert picks.count(1) > picks.count(8) >= 1            # mostly plain, with periodic probes
    first_probe = picks.index(8)
    assert picks[first_probe + 1:first_probe + 1 + 3] == [1, 1, 1]


def test_probe_spacing_follows_costs():
    def spacing(ratio):
        c = W.Controller([1, 8], [100.0, 100.0 * ratio])
        for _ in range(20):
            c.observe(8, [st(0, 0, 1)] * 4)
        picks = [c.choose() for _ in range(200)]
        return picks.index(8) + 1
    assert spacing(1.2) < spacing(4.0)


def test_failed_probes_back_off_and_an_accepting_probe_resets():
    c = W.Controller([1, 4], [100.0, 110.0])             # base spacing ceil(4 * 1.1) = 5
    for _ in range(20):
        c.observe(4, [st(0, 0, 1)] * 4)                  # wide windows accept nothing: plain is best
    gaps, last = [], 0
    for k in range(1, 400):
        w = c.choose()
        if w == 4:
            gaps.append(k - last)
            last = k
            c.observe(4, [st(0, 0, 1)])                  # the probe accepts no draft
        else:
            c.observe(1, [st(0, 0, 1)])
    assert gaps[:5] == [5, 10, 20, 40, 64] and all(g == 64 for g in gaps[5:])
    # a probe that accepts a draft returns the spacing to the cost-based one
    while c.choose() != 4:
        c.observe(1, [st(0, 0, 1)])
    c.observe(4, [st(1, 1, 2)])
    n = 1
    while c.choose() != 4:
        n += 1
    assert n == 5


def test_backoff_with_two_windows_in_flight():
    """Windows complete in the order they were chosen; with two in flight the choice of window
    k + 1 comes before the observation of window k, and a probe's own window still decides."""
    c = W.Controller([1, 4], [100.0, 110.0])
    for _ in range(20):
        c.observe(4, [st(0, 0, 1)] * 4)
    inflight = [c.choose(), c.choose()]
    gaps, last = [], 0
    for k in range(3, 400):
        w = inflight.pop(0)
        c.observe(w, [st(0, 0, 1)])                      # nothing is ever accepted
        inflight.append(c.choose())
        if inflight[-1] == 4:
            gaps.append(k - last)
            last = k
    assert gaps[1:5] == [10, 20, 40, 64]


def test_cost_moving_average():
    c = W.Controller([1, 4], [100.0, 200.0])
    c.observe(4, [st(1, 1)] * 4, interval_us=4 * 120.0)
    assert abs(c.cost(4) - (0.75 * 200.0 + 0.25 * 120.0)) < 1e-9
    c.observe(4, [st(1, 1)] * 2, interval_us=0.0)           # unknown interval: no update
    assert abs(c.cost(4) - 180.0) < 1e-9


def test_invalid_arguments():
    with pytest.raises(W.W4A8Error):
        W.Controller([4, 1], [1.0, 1.0])
    with pytest.raises(W.W4A8Error):
        W.Controller([1, 4], [1.0, 0.0])
    with pytest.raises(W.W4A8Error):
        W.Controller([1, 32], [1.0, 2.0])
