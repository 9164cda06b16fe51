"""Pins of the oracle's quantised decoder (CPU)."""
import numpy as np
import pytest
import scipy.special

import synth
from oracle import model as OM
from oracle import quant as Q
from oracle import spec as OS

SMALL = synth.ModelShape("pin-1L-64h", 1, 64, 4, 2, 16, 64, 64, 64, False)


@pytest.fixture(scope="module")
def tiny_weights():
    return OM.build_weights(synth.TINY, 1000)


def test_rmsnorm_closed_form():
    x = np.full(32, -3.0)
    eps = 1e-6
    assert np.allclose(OM.rmsnorm(x, eps), -3.0 / np.sqrt(9.0 + eps), rtol=1e-15)
    x = np.array([3.0, 4.0])
    assert np.allclose(OM.rmsnorm(x, 0.0), x / np.sqrt(12.5), rtol=1e-15)


def test_silu_matches_scipy():
    z = np.linspace(-20, 20, 101)
    assert np.allclose(OM.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)


def test_rope_rotation_and_relative_property():
    v = np.array([1.0, 0.0])                       # d=2: theta_0 = 1
    assert np.allclose(OM.rope(v, 3, 10000.0), [np.cos(3.0), np.sin(3.0)], rtol=1e-15)
    rng = np.random.default_rng(0)
    q, k = rng.normal(size=64), rng.normal(size=64)
    assert np.allclose(OM.rope(q, 0, 10000.0), q)
    assert np.isclose(np.linalg.norm(OM.rope(q, 17, 10000.0)), np.linalg.norm(q))
    a = OM.rope(q, 9, 10000.0) @ OM.rope(k, 4, 10000.0)
    b = OM.rope(q, 105, 10000.0) @ OM.rope(k, 100, 10000.0)
    assert np.isclose(a, b, rtol=1e-12)
    # rotate-half pairs dim i with dim i + d/2 (not adjacent dims)
    e = np.zeros(8); e[1] = 1.0
    r = OM.rope(e, 1, 10000.0)
    th = 10000.0 ** (-2.0 / 8)
    assert np.isclose(r[1], np.cos(th)) and np.isclose(r[5], np.sin(th)) and abs(r[0]) + abs(r[2]) == 0


def test_attend_special_cases():
    rng = np.random.default_rng(1)
    q = rng.normal(size=16)
    K1, V1 = rng.normal(size=(1, 16)), rng.normal(size=(1, 16))
    assert np.allclose(OM.attend(q, K1, V1), V1[0])
    K, V = rng.normal(size=(7, 16)), rng.normal(size=(7, 16))
    assert np.allclose(OM.attend(np.zeros(16), K, V), V.mean(axis=0))
    ref = scipy.special.softmax(K @ q / 4.0) @ V
    assert np.allclose(OM.attend(q, K, V), ref, rtol=1e-13)


def test_gqa_head_mapping():
    assert [OM.kv_head_of(h, 4, 2) for h in range(4)] == [0, 0, 1, 1]
    assert [OM.kv_head_of(h, 14, 2) for h in range(14)] == [0] * 7 + [1] * 7


def _crafted(zero_kinds=(), seed=3):
    w = OM.build_weights(SMALL, seed)
    for kind in zero_kinds:
        q, s = w.layers[0][kind]
        w.layers[0][kind] = (np.zeros_like(q), np.zeros_like(s))
    return w


def test_residual_structure_with_zero_blocks():
    # O and down projections zero: every layer is the identity, logits = lm_head(quant(rmsnorm(embedding)))
    w = _crafted(zero_kinds=(synth.T_WO, synth.T_WD))
    m = OM.Model(w, 8)
    toks = [5, 9, 2]
    lg = m.prefill(toks)
    lq, ls = w.lm_head
    for i, t in enumerate(toks):
        e = Q.dequantize_weights(w.embed[0][t:t + 1], w.embed[1][t:t + 1])[0]
        n = e / np.sqrt(np.mean(e * e) + SMALL.rms_eps)
        a_q, a_s = Q.quantize_act_per_token(n.astype(np.float32)[None, :])
        ref = (a_q[0].astype(np.float64) * float(a_s[0])) @ Q.dequantize_weights(lq, ls).T
        assert np.allclose(lg[i], ref, rtol=1e-13, atol=1e-13)


def test_gqa_group_reads_its_kv_head():
    # V rows of KV head 1 zeroed: query heads 2,3 attend to zero values, heads 0,1 do not
    w = _crafted()
    q, s = w.layers[0][synth.T_WV]
    q = q.copy(); s = s.copy()
    q[16:32] = 0; s[16:32] = 0
    w.layers[0][synth.T_WV] = (q, s)
    m = OM.Model(w, 8)
    tr = {}
    m.forward([3, 4], [0, 1], [0, 1], [[0], [0, 1]], trace=tr)
    att = tr["att"][1]                                  # token 1, [Hq][d]
    assert np.all(att[2:] == 0) and np.all(np.abs(att[:2]).sum(axis=1) > 0)


def test_swiglu_uses_silu_of_gate():
    w = _crafted()
    m = OM.Model(w, 4)
    n2 = np.random.default_rng(2).normal(size=64)
    out = m.mlp(0, w.layers[0], n2)
    gq, gs = w.layers[0][synth.T_WG]
    uq, us = w.layers[0][synth.T_WU]
    dq, ds = w.layers[0][synth.T_WD]
    def lin(qs, x):
        a_q, a_s = Q.quantize_act_per_token(np.asarray(x, np.float32)[None, :])
        return (a_q[0].astype(np.float64) * float(a_s[0])) @ Q.dequantize_weights(*qs).T
    g, u = lin((gq, gs), n2), lin((uq, us), n2)
    assert np.allclose(out, lin((dq, ds), scipy.special.expit(g) * g * u), rtol=1e-12, atol=1e-14)
    assert not np.allclose(out, lin((dq, ds), scipy.special.expit(u) * u * g), rtol=1e-6)


def test_causality_of_prefill(tiny_weights):
    toks = synth.motif_prompt(7, 12, 2, 6, 0.0, synth.TINY.vocab).tolist()
    a = OM.Model(tiny_weights, 16).prefill(toks)
    toks2 = toks[:8] + [1, 2, 3, 4]
    b = OM.Model(tiny_weights, 16).prefill(toks2)
    assert np.array_equal(a[:8], b[:8])
    assert not np.allclose(a[8:], b[8:])


def test_prefill_equals_sequential_steps(tiny_weights):
    toks = synth.motif_prompt(8, 10, 2, 5, 0.2, synth.TINY.vocab).tolist()
    a = OM.Model(tiny_weights, 16).prefill(toks)
    m = OM.Model(tiny_weights, 16)
    b = np.stack([m.step(t, i) for i, t in enumerate(toks)])
    assert np.array_equal(a, b)


def test_padded_ffn_is_exact(tiny_weights):
    # the zero-padded FFN rows (688 -> 704) carry code 0 and scale 0 after quantisation
    q, s = tiny_weights.layers[0][synth.T_WG]
    assert np.all(q[688:] == 0) and np.all(s[688:] == 0)
    qd, sd = tiny_weights.layers[0][synth.T_WD]
    assert np.all(qd[:, 688:] == 0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_verify_equals_sequential_root_paths(tiny_weights, seed):
    rng = np.random.default_rng(seed)
    ctx = synth.motif_prompt(100 + seed, 20, 3, 5, 0.1, synth.TINY.vocab).tolist()
    N = [16, 7, 3][seed]
    tok, parent = synth.random_tree(rng, N, synth.TINY.vocab)
    L_c = len(ctx)
    m = OM.Model(tiny_weights, L_c + N + 1)
    m.prefill(ctx)
    lg = OS.tree_verify(m, L_c, tok, parent)
    for i in range(N):
        path = OS.ancestors_or_self(parent, i)
        ref = OM.Model(tiny_weights, L_c + 20).prefill(ctx + [int(tok[j]) for j in path])[-1]
        assert np.array_equal(lg[i], ref), i


def test_decision_margins_closed_form():
    # amax 127 -> scale exactly 1.0, so the quotient of every input is the input itself
    x = np.array([127.0, 10.3, -5.51, 2.5, 0.0, -126.2], dtype=np.float32)
    m = OM.decision_margins(x)
    f = x.astype(np.float64)
    assert m[0] == 0.5                                   # at the clamp: distance to 126.5
    assert np.isclose(m[1], abs(10.3 - 10.5), atol=1e-6) and abs(m[1] - 0.2) < 1e-6
    assert m[2] == abs(abs(f[2]) - 5.5) and 0.0099 < m[2] < 0.0101   # sign does not matter
    assert m[3] == 0.0                                   # exactly on a rounding boundary
    assert m[4] == 0.5                                   # zero: midway between -1/2 and 1/2
    assert np.isclose(m[5], 0.3, atol=1e-5)
    assert OM.decision_margin(x) == 0.0
    assert OM.decision_margin(x[[0, 1, 2]]) == m[2]
    # scale 2: quotient = x / 2
    y = np.array([254.0, 5.0, 7.2], dtype=np.float32)
    my = OM.decision_margins(y)
    assert my[1] == 0.0 and np.isclose(my[2], 0.1, atol=1e-6)
    assert np.all(np.isinf(OM.decision_margins(np.zeros(8, np.float32))))


def test_decision_margin_predicts_code_changes():
    # a perturbation smaller than an input's margin (in code units) keeps its code; one
    # larger than the margin, towards the boundary, changes it
    rng = np.random.default_rng(11)
    x = rng.normal(size=256).astype(np.float32)
    q0, s = OM.quant_row(x)
    m = OM.decision_margins(x)
    k = int(np.argmin(m[np.abs(x) < np.abs(x).max()]))
    k = int(np.flatnonzero(np.abs(x) < np.abs(x).max())[k])
    r = abs(float(x[k])) / float(s)
    towards = np.sign(r - np.floor(r) - 0.5) * -np.sign(x[k])   # direction of the boundary
    y = x.astype(np.float64).copy()
    y[k] += towards * (m[k] + 1e-4) * float(s)
    q1, s1 = OM.quant_row(y)
    assert s1 == s and abs(int(q1[k]) - int(q0[k])) == 1
    z = x.astype(np.float64).copy()
    z[k] += towards * 0.5 * m[k] * float(s)
    q2, _ = OM.quant_row(z)
    assert np.array_equal(q2, q0)
