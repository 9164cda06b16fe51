"""Oracle parity of tree verification at the benchmarked model dimensions.

Two-layer decoders with the full per-layer dimensions of the benchmarked workloads:
* Llama-3-8B-shaped: hidden 4096, 32 query / 8 KV heads of 128, FFN 14336, untied vocab
  128256 (the headline workload);
* Qwen2.5-0.5B-shaped: hidden 896, 14 query / 2 KV heads of 64 (7 query heads per KV
  head), FFN 4864, tied vocab 151936.
A third two-layer model has awkward dimensions for the quantisers and the matmul: hidden
1120 (the last 64-input chunk of every hidden-wide input is half padding; the O, down and LM
projections end in a partial row group), FFN 16416 (33 statistics slices per token; a
half-padded last chunk), 10 query / 2 KV heads of 64 (5 query heads per KV head).
Weights are seeded int4 codes U{-8..7} with fp16 group scales U(0.001, 0.008) (about the
spread of N(0, 0.02) weights after quantisation), loaded into the library in the packed
layout and given to the oracle as the same codes; the cache below the tree is the same
seeded fp32 K/V on both sides (``w4a8_session_load_kv``), so that a context of thousands of
tokens costs the oracle no prefill.  Trees of 1, 8 and 16 nodes exercise the one- and
two-tile matmul paths, their split-K partial folds in the consumer kernels, the grouped
attention of both head sizes and the LM head of each shape.  Rows are compared at the code
level (``tests/parity.py``).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth
import w4a8_verify_gb300 as W
from oracle import model as OM

import parity as P

pytestmark = pytest.mark.gpu

LLAMA_2L = synth.ModelShape("llama3-8b-2layer", 2, 4096, 32, 8, 128, 14336, 14336, 128256, False)
QWEN_2L = synth.ModelShape("qwen2.5-0.5b-2layer", 2, 896, 14, 2, 64, 4864, 4864, 151936, True)
EDGE_2L = synth.ModelShape("edge-2layer", 2, 1120, 10, 2, 64, 16416, 16416, 4096, False)
TALLY = P.Tally()
CACHE_BYTES = 16 << 30        # the oracle keeps these models' dequantised weights (~8 GB)


def _codes(seed, stream, rows, cols):
    q = synth.uniform_codes(seed, stream, 0, rows * cols).reshape(rows, cols)
    s = synth.uniform_scales(seed, stream + 1, 0, rows * (cols // 32), 0.001, 0.008).reshape(rows, cols // 32)
    return q, s


def build_pair(shape, seed):
    """The same seeded int4 weights as a library model and as oracle Weights."""
    m = W.Model(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                shape.vocab, shape.tied, shape.rms_eps, shape.rope_base)
    kinds = {synth.T_WQ: W.T_Q, synth.T_WK: W.T_K, synth.T_WV: W.T_V, synth.T_WO: W.T_O, synth.T_WG: W.T_GATE,
             synth.T_WU: W.T_UP, synth.T_WD: W.T_DOWN}

    def load(kind, layer, q, s):
        wp2 = torch.from_numpy(W.w4a8_pack_weights(q).view(np.int32)).cuda()
        sp2 = torch.from_numpy(s.view(np.int16)).cuda()
        m.load_tensor(kind, layer, wp2, sp2)
        torch.cuda.synchronize()

    layers = []
    for l in range(shape.n_layers):
        d = {}
        for kind in range(7):
            rows, cols, _, _ = synth.tensor_shape(shape, kind)
            d[kind] = _codes(seed, 64 * l + 2 * kind, rows, cols)
            load(kinds[kind], l, *d[kind])
        layers.append(d)
    emb = _codes(seed, 1000, shape.vocab, shape.hidden)
    load(W.T_EMBED, 0, *emb)
    lm = emb
    if not shape.tied:
        lm = _codes(seed, 1002, shape.vocab, shape.hidden)
        load(W.T_LM_HEAD, 0, *lm)
    return m, OM.Weights(shape, layers, emb, lm)


@pytest.fixture(scope="module")
def models():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    W.lib()
    out = {}
    for shape in (LLAMA_2L, QWEN_2L, EDGE_2L):
        out[shape.name] = (shape,) + build_pair(shape, 1100 + len(out))
    yield out
    print("\n[benchmarked-shape parity] " + TALLY.summary())


@pytest.mark.parametrize("name", [LLAMA_2L.name, QWEN_2L.name])
@pytest.mark.parametrize("N,L,seed", [(1, 300, 0), (8, 300, 1), (16, 257, 2), (16, 1000, 3)])
def test_tree_verify_at_benchmarked_dims(models, name, N, L, seed, monkeypatch):
    shape, m, ow = models[name]
    monkeypatch.setattr(OM, "DEQ_CACHE_BYTES", CACHE_BYTES)
    rng = np.random.default_rng(seed)
    tok, parent = synth.random_tree(rng, N, shape.vocab, max_depth=8)
    s = W.Session(m, L + 64, L + 64, 4)
    s.prefill(torch.as_tensor(synth.motif_prompt(500 + seed, L + 1, 4, 16, 0.1, shape.vocab)).cuda(), max_new=8)
    P.verify_on_given_cache(s, ow, shape, L, tok, parent, 600 + seed, TALLY)
    s.close()


@pytest.mark.parametrize("N,L,seed", [(1, 130, 10), (5, 300, 11), (8, 257, 12), (16, 300, 13)])
def test_tree_verify_at_awkward_dims(models, N, L, seed, monkeypatch):
    shape, m, ow = models[EDGE_2L.name]
    monkeypatch.setattr(OM, "DEQ_CACHE_BYTES", CACHE_BYTES)
    tok, parent = synth.random_tree(np.random.default_rng(seed), N, shape.vocab, max_depth=8)
    s = W.Session(m, L + 64, L + 64, 4)
    s.prefill(torch.as_tensor(synth.motif_prompt(500 + seed, L + 1, 4, 16, 0.1, shape.vocab)).cuda(), max_new=8)
    P.verify_on_given_cache(s, ow, shape, L, tok, parent, 600 + seed, TALLY)
    s.close()


@pytest.mark.parametrize("name", [LLAMA_2L.name, QWEN_2L.name, EDGE_2L.name])
@pytest.mark.parametrize("n", [146, 176])
def test_prefill_buckets_equal_sequential_kv_at_benchmarked_dims(models, name, n):
    """n - 1 prompt tokens prefill as two 64-token buckets (the attention as four 16-node chains,
    with 4, 7 and 5 query heads per KV head), then 145: chains of 16 and 1; 175: one pass over
    two chains (32 tokens) and a chain of 15.  The cache must hold the bits that n - 1
    single-token steps write."""
    shape, m, _ = models[name]
    prompt = synth.motif_prompt(77, n, 4, 16, 0.1, shape.vocab)
    s = W.Session(m, n + 64, n + 64, 4)
    s.prefill(torch.as_tensor(prompt).cuda(), max_new=8)
    q = W.Session(m, n + 64, n + 64, 4)
    q.prefill(torch.as_tensor(prompt[:1]).cuda(), max_new=n + 4)
    for tok in prompt[:n - 1]:               # teacher-forced single-token steps
        q.set_tree([int(tok)], [-1])
        q.tree_verify_step(1)
        q.accept_greedy(1)
    L = n - 1
    for layer in range(shape.n_layers):
        k1, v1, k2, v2 = (torch.empty((shape.n_kv_heads, L, shape.head_dim), dtype=torch.float32, device="cuda")
                          for _ in range(4))
        s.copy_kv(layer, 0, L, k1, v1)
        q.copy_kv(layer, 0, L, k2, v2)
        torch.cuda.synchronize()
        assert torch.equal(k1, k2) and torch.equal(v1, v2), (name, layer)
    assert s.ctl().committed_len == L and q.ctl().committed_len == L
    s.close()
    q.close()


def test_tree_verify_at_full_context_8b(models, monkeypatch):
    """One node after a 4095-slot cache at the 8B dimensions (the headline context)."""
    shape, m, ow = models[LLAMA_2L.name]
    monkeypatch.setattr(OM, "DEQ_CACHE_BYTES", CACHE_BYTES)
    L = 4095
    s = W.Session(m, L + 32, L + 32, 4)
    s.prefill(torch.as_tensor(synth.motif_prompt(700, L + 1, 4, 16, 0.1, shape.vocab)).cuda(), max_new=8)
    P.verify_on_given_cache(s, ow, shape, L, np.array([17], np.int32), np.array([-1], np.int32), 701, TALLY)
    tok, parent = synth.random_tree(np.random.default_rng(9), 4, shape.vocab)
    P.verify_on_given_cache(s, ow, shape, L, tok, parent, 702, TALLY)
    s.close()


def test_most_rows_at_the_north_star_bound(models):
    if TALLY.strict + TALLY.loose == 0:
        pytest.skip("no parity rows ran in this session (test selection)")
    assert TALLY.strict > TALLY.loose, TALLY.summary()
